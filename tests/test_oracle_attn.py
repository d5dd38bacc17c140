"""Pins of the oracle's width-k attention verify against what the pages and
the mathematics fix, none of them re-typing the oracle's loops.

Pages: "QWEN38FLASH.md - Plan for supporting Qwen/Qwen3.8-Flash-Next" 2.2
(grouped-query attention, partial RoPE, sigmoid output gate, F16 cache) and
"Red Lite dev45 - speculative decoding with the Qwen3-Next MTP block",
"What it is" (attention runs per row: row r sees the earlier rows' K/V).
"""
import math

import numpy as np
import pytest

from oracle import oracle as O
from speculative_decode_verification_gb300 import synth as S


def bfv(bits):
    return S.bf16_to_f32(np.asarray(bits, np.uint16)).astype(np.float64)


def f16v(bits):
    return np.asarray(bits, np.uint16).view(np.float16).astype(np.float64)


def bf16(v):
    return S.f32_to_bf16(np.asarray(v, np.float32))


def sig(x):
    return 1.0 / (1.0 + np.exp(-x))


def test_f16_rounding_is_numpy_cast():
    """The binary16 rounding is the IEEE one: numpy's float16 cast, across
    normal, subnormal, overflow and halfway values."""
    rng = np.random.default_rng(0)
    v = np.concatenate([rng.standard_normal(20000) * 10.0 ** rng.integers(-9, 6, 20000),
                        np.arange(-2048, 2049) * 2.0 ** -25,           # subnormal halfway points
                        (1024 + np.arange(0, 1024) + 0.5) * 2.0 ** -9,  # halfway between normals
                        [65504.0, 65519.99, 65520.0, -65520.0, 1e9, -0.0, 0.0]])
    with np.errstate(over="ignore"):
        want = v.astype(np.float16).view(np.uint16)
    got = np.array([O.round_f16(x) for x in v], np.uint16)
    assert np.array_equal(got, want)


def _run(Hq, Hkv, D, P, inp, K, V, rope_dim=64, theta=1e7):
    return O.attn_verify(Hq, Hkv, D, P, inp["q"], inp["k"], inp["v"], inp["gate"], K, V, rope_dim, theta)


def test_single_key_closed_form():
    """An empty cache and one row: the softmax has one entry, so
    o = value * sigmoid(gate) with the value as the cache holds it."""
    Hq, Hkv, D = 4, 2, 128
    inp = S.attn_inputs(1, "one", 1, Hq, Hkv, D)
    K, V = S.attn_cache(1, "one", Hkv, 4, D, 0)
    o, _, v_app = _run(Hq, Hkv, D, 0, inp, K, V)
    G = Hq // Hkv
    for h in range(Hq):
        want = f16v(v_app[0, h // G]) * sig(bfv(inp["gate"][0, h]))
        assert np.allclose(o[0, h], want, rtol=1e-12, atol=0)
    assert np.array_equal(f16v(v_app), bfv(inp["v"]).astype(np.float16).astype(np.float64))


@pytest.mark.parametrize("P", [0, 1, 37, 300])
def test_zero_query_averages_the_window(P):
    """q = 0 gives equal scores, so row r's output is the mean of the values
    at positions 0 .. P + r (its window: the cache and rows 0..r), gated."""
    Hq, Hkv, D, k = 4, 2, 64, 5
    inp = S.attn_inputs(2, f"avg{P}", k, Hq, Hkv, D)
    inp["q"] = np.zeros_like(inp["q"])
    K, V = S.attn_cache(2, f"avg{P}", Hkv, P + k, D, P)
    o, _, v_app = _run(Hq, Hkv, D, P, inp, K, V)
    G = Hq // Hkv
    for r in range(k):
        for h in range(Hq):
            vals = np.concatenate([f16v(V[h // G, :P]), f16v(v_app[: r + 1, h // G])])
            want = vals.mean(axis=0) * sig(bfv(inp["gate"][r, h]))
            assert np.allclose(o[r, h], want, rtol=1e-12, atol=1e-15), (r, h)


@pytest.mark.parametrize("i", [0, 5, 31])
def test_rope_of_a_one_hot_key(i):
    """A key e_i (i below rope_dim/2) at position pos becomes
    cos(pos w_i) e_i + sin(pos w_i) e_{i+32}, w_i = theta^(-2i/64); entries
    from rope_dim on pass through unchanged."""
    Hq, Hkv, D, k, P = 2, 1, 256, 3, 1000
    inp = S.attn_inputs(3, "rope", k, Hq, Hkv, D)
    key = np.zeros((k, Hkv, D), np.float32)
    key[:, :, i] = 1.0
    key[:, :, 200] = 0.75  # beyond the rotated dims
    inp["k"] = bf16(key)
    K, V = S.attn_cache(3, "rope", Hkv, P + k, D, 0)
    _, k_app, _ = _run(Hq, Hkv, D, P, inp, K, V)
    for r in range(k):
        ang = (P + r) * 1e7 ** (-2 * i / 64)
        want = np.zeros(D)
        want[i], want[i + 32], want[200] = math.cos(ang), math.sin(ang), 0.75
        got = f16v(k_app[r, 0])
        assert np.array_equal(got, f16v(np.array([O.round_f16(x) for x in want], np.uint16)))  # -0 == +0


def test_scores_depend_on_relative_position_only():
    """Rotating query and keys by their positions leaves q.k depending on the
    distance alone: two keys with one-hot values give o0/o1 = exp(s0 - s1),
    and prepending 100 cached positions with zero keys and values (which only
    rescale the softmax) leaves that ratio unchanged."""
    Hq, Hkv, D, k = 1, 1, 128, 2
    inp = S.attn_inputs(4, "rel", k, Hq, Hkv, D)
    v = np.zeros((k, Hkv, D), np.float32)
    v[0, 0, 0], v[1, 0, 1] = 1.0, 1.0
    inp["v"] = bf16(v)
    inp["gate"] = bf16(np.full((k, Hq, D), 30.0))
    ratios = []
    for P in (0, 100):
        K, V = S.attn_cache(4, "rel", Hkv, P + k, D, 0)  # zero keys and values
        o, _, _ = _run(Hq, Hkv, D, P, inp, K, V, rope_dim=128, theta=1e4)
        ratios.append(o[1, 0, 0] / o[1, 0, 1])
    assert ratios[0] > 0 and abs(ratios[0] / ratios[1] - 1) < 1e-3  # keys are rounded to f16 at other angles
    # and a rotation in the wrong sense would move it: check the score gap is position-sensitive at all
    assert abs(math.log(ratios[0])) > 1e-3


def test_k_rows_equal_k_single_row_steps():
    """Row r of a width-k call is a width-1 call at position P + r whose cache
    holds rows 0..r-1 of the block: the window is causal and row r sees the
    earlier rows' keys and values."""
    Hq, Hkv, D, k, P = 6, 2, 64, 4, 50
    inp = S.attn_inputs(5, "seq", k, Hq, Hkv, D)
    K, V = S.attn_cache(5, "seq", Hkv, P + k, D, P)
    o, k_app, v_app = _run(Hq, Hkv, D, P, inp, K, V)
    K1, V1 = K.copy(), V.copy()
    for r in range(k):
        one = {key: val[r:r + 1] for key, val in inp.items()}
        o1, ka1, va1 = _run(Hq, Hkv, D, P + r, one, K1, V1)
        assert np.array_equal(o1[0], o[r])
        assert np.array_equal(ka1[0], k_app[r]) and np.array_equal(va1[0], v_app[r])
        K1[:, P + r], V1[:, P + r] = ka1[0], va1[0]


def test_query_heads_read_their_kv_group():
    """Query heads h read KV head h // (Hq / Hkv): with every value of KV head
    j equal to e_j, head h's output is e_{h // G} * sigmoid(gate)."""
    Hq, Hkv, D, k, P = 6, 3, 64, 2, 10
    inp = S.attn_inputs(6, "gqa", k, Hq, Hkv, D)
    v = np.zeros((k, Hkv, D), np.float32)
    for j in range(Hkv):
        v[:, j, j] = 1.0
    inp["v"] = bf16(v)
    K, V = S.attn_cache(6, "gqa", Hkv, P + k, D, P)
    V[:] = 0
    for j in range(Hkv):
        V[j, :P, j] = O.round_f16(1.0)
    o, _, _ = _run(Hq, Hkv, D, P, inp, K, V)
    G = Hq // Hkv
    for r in range(k):
        for h in range(Hq):
            want = np.zeros(D)
            want[h // G] = 1.0
            assert np.allclose(o[r, h], want * sig(bfv(inp["gate"][r, h])), rtol=1e-12, atol=1e-15)


def test_two_key_score_gap_is_the_scaled_dot_product():
    """Without rotation (rope_dim 0), two keys with one-hot values give
    log(o0 / o1) = (k0 - k1).q / sqrt(D): the softmax of scores q.k / sqrt(D)."""
    Hq, Hkv, D, k = 1, 1, 256, 2
    inp = S.attn_inputs(7, "gap", k, Hq, Hkv, D)
    v = np.zeros((k, Hkv, D), np.float32)
    v[0, 0, 0], v[1, 0, 1] = 1.0, 1.0
    inp["v"] = bf16(v)
    inp["gate"] = bf16(np.full((k, Hq, D), 30.0))
    K, V = S.attn_cache(7, "gap", Hkv, k, D, 0)
    o, k_app, _ = _run(Hq, Hkv, D, 0, inp, K, V, rope_dim=0)
    q1 = bfv(inp["q"][1, 0])
    k0, k1 = f16v(k_app[0, 0]), f16v(k_app[1, 0])
    assert abs(math.log(o[1, 0, 0] / o[1, 0, 1]) - float(np.dot(k0 - k1, q1)) / 16.0) < 1e-9
