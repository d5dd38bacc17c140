"""Pins of the CPU oracle against what the pages and the mathematics fix.

None of these compares the oracle with itself or retypes its loops: each
check is a closed form of a special case, a brute force computed another way,
or an invariant the pages state.  Pages (by title):
  [T] "Flash-Next optimization transfer to Ornith and Qwen 27B"
  [R] "Red Lite dev45 - speculative decoding with the Qwen3-Next MTP block"
  [F] "QWEN38FLASH.md - Plan for supporting Qwen/Qwen3.8-Flash-Next"
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest

from oracle import oracle as O
from speculative_decode_verification_gb300 import synth as S

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def bf16(v):
    return S.f32_to_bf16(np.asarray(v, np.float32))


def bfv(bits):
    return S.bf16_to_f32(bits).astype(np.float64)


# ------------------------------------------------------------------ Q4 / QMV

def _empty_q4(n, K):
    return (np.zeros((n, K // 8), np.uint32), np.zeros((n, K // 64), np.uint16),
            np.zeros((n, K // 64), np.uint16))


@pytest.mark.parametrize("col", [0, 1, 3, 7, 8, 9, 15, 63, 64, 65, 127, 191])
def test_q4_one_hot_column_picks_documented_nibble(col):
    """[T] table "Shared architecture": affine Q4, group 64.  With x one-hot at
    column c, y[n] = w[n][c] = s*q + b, where q sits in bits 4*(c%8) of word
    c/8 and s, b are group c/64's.  Distinct values per group make a wrong
    nibble order, word or group index, or a swapped scale/bias visible."""
    n, K = 3, 192
    packed, scales, biases = _empty_q4(n, K)
    for g in range(K // 64):
        scales[:, g] = bf16([0.25 * (g + 1)] * n)
        biases[:, g] = bf16([-0.125 * (g + 2)] * n)
    q_of_row = [5, 11, 15]
    for r in range(n):
        packed[r, col // 8] |= np.uint32(q_of_row[r] << (4 * (col % 8)))
    for probe in sorted({col, (col + 1) % K, (col + 8) % K}):
        x = np.zeros((1, K), np.uint16)
        x[0, probe] = bf16(1.0)
        y = O.q4_qmv(packed, scales, biases, x)[0]
        g = probe // 64
        for r in range(n):
            q = q_of_row[r] if probe == col else 0
            assert y[r] == 0.25 * (g + 1) * q - 0.125 * (g + 2)


def test_q4_exact_integer_case_bruteforce():
    """Exactly representable case: integer x in -2..2, s = 2^-3, b in
    {-1,0,1}*2^-4.  Every partial sum is a multiple of 2^-4 far below 2^50, so
    the float64 oracle must equal exact rational arithmetic bit for bit."""
    rng = np.random.default_rng(7)
    n, K, k = 24, 1024, 3
    packed = rng.integers(0, 2 ** 32, size=(n, K // 8), dtype=np.uint64).astype(np.uint32)
    scales = np.full((n, K // 64), bf16(0.125), np.uint16)
    bsel = rng.integers(-1, 2, size=(n, K // 64))
    biases = bf16(bsel * 0.0625).reshape(n, K // 64)
    xi = rng.integers(-2, 3, size=(k, K))
    x = bf16(xi.astype(np.float32)).reshape(k, K)
    y = O.q4_qmv(packed, scales, biases, x)
    for r in range(k):
        for row in range(n):
            tot = Fraction(0)
            for c in range(K):
                q = (int(packed[row, c // 8]) >> (4 * (c % 8))) & 15
                tot += (Fraction(1, 8) * q + Fraction(int(bsel[row, c // 64]), 16)) * int(xi[r, c])
            assert Fraction(y[r, row]) == tot


def test_q4_matches_bytewise_dequant_bruteforce():
    """Brute force through another decode path: view the words as little-endian
    bytes, split low/high nibbles, dequantise, float64 matmul."""
    m = S.q4_matrix(3, "pin.q4", 40, 256)
    x = S.bf16_normal(3, "pin.x", (4, 256))
    by = m.packed.view(np.uint8).reshape(40, 128)
    q = np.empty((40, 256), np.float64)
    q[:, 0::2] = by & 15
    q[:, 1::2] = by >> 4
    s = np.repeat(bfv(m.scales), 64, axis=1)
    b = np.repeat(bfv(m.biases), 64, axis=1)
    ref = (s * q + b) @ bfv(x).T
    y = O.q4_qmv(m.packed, m.scales, m.biases, x)
    np.testing.assert_allclose(y, ref.T, rtol=1e-12, atol=1e-12)


def test_q4_width_k_equals_k_width_1():
    """[T] "Exact verification kernels": width-k output equals serial QMV."""
    m = S.q4_matrix(5, "pin.q4w", 64, 512)
    x = S.bf16_normal(5, "pin.xw", (9, 512))
    y = O.q4_qmv(m.packed, m.scales, m.biases, x)
    for r in range(9):
        assert np.array_equal(y[r], O.q4_qmv(m.packed, m.scales, m.biases, x[r:r + 1])[0])


# ------------------------------------------------------------------ routing

def test_route_order_and_ties_match_sorted_bruteforce():
    """Top-T = the first T of the experts sorted by (-logit, index): ties keep
    the lower index (the reading for the pages' silence on ties)."""
    rng = np.random.default_rng(11)
    k, E, T = 6, 40, 8
    logits = rng.integers(-6, 7, size=(k, E)).astype(np.float32) * 0.5  # many exact ties
    idx, _ = O.route_topk(logits, T)
    for r in range(k):
        want = sorted(range(E), key=lambda e: (-float(logits[r, e]), e))[:T]
        assert list(idx[r]) == want


def test_route_weights_softmax_identities():
    """w sums to 1, w_i/w_j = exp(l_i - l_j); with T = E it is the full
    softmax; with two experts w_0 = 1/(1 + exp(l_1 - l_0))."""
    rng = np.random.default_rng(12)
    logits = rng.standard_normal((5, 16)).astype(np.float32)
    idx, w = O.route_topk(logits, 16)
    for r in range(5):
        assert abs(w[r].sum() - 1.0) < 1e-14
        l = logits[r, idx[r]].astype(np.float64)
        assert np.allclose(w[r] / w[r, 0], np.exp(l - l[0]), rtol=1e-13)
    two = np.array([[0.75, -0.5]], np.float32)
    i2, w2 = O.route_topk(two, 2)
    assert list(i2[0]) == [0, 1]
    assert abs(w2[0, 0] - 1.0 / (1.0 + math.exp(-0.5 - 0.75))) < 1e-15
    eq = np.zeros((1, 10), np.float32)
    ie, we = O.route_topk(eq, 4)
    assert list(ie[0]) == [0, 1, 2, 3] and np.all(we == 0.25)


# ----------------------------------------------------------- routed experts

def _silu(t):
    return t / (1.0 + np.exp(-t))


def _moe_case(seed, E=6, H=128, I=64):
    gu = S.q4_matrix(seed, "pin.gu", 2 * I, H, n_experts=E)
    dn = S.q4_matrix(seed, "pin.dn", H, I, n_experts=E)
    return gu, dn


def _expert_direct(gu, dn, e, xrow):
    """One expert assembled from pinned pieces: two dense products, SwiGLU,
    bf16, dense down product."""
    I = gu.n_out // 2
    gate = O.q4_qmv(gu.packed[e, :I], gu.scales[e, :I], gu.biases[e, :I], xrow)[0]
    up = O.q4_qmv(gu.packed[e, I:], gu.scales[e, I:], gu.biases[e, I:], xrow)[0]
    h = O.to_bf16(_silu(gate) * up)[None, :]
    return O.q4_qmv(dn.packed[e], dn.scales[e], dn.biases[e], h)[0], h[0]


def test_gather_single_expert_reduces_to_dense_products():
    """T = 1 with every row routed to one expert: the gathered path is two
    dense products, SwiGLU (gate half first, [F] 2.3), bf16, a dense down
    product, weight 1."""
    gu, dn = _moe_case(21)
    k, E = 3, 6
    x = S.bf16_normal(21, "pin.moe.x", (k, 128))
    logits = np.full((k, E), -1.0, np.float32)
    logits[:, 4] = 2.0
    idx, w, y, h = O.gather_experts((gu.packed, gu.scales, gu.biases), (dn.packed, dn.scales, dn.biases),
                                    logits, 1, x)
    assert np.all(idx == 4) and np.all(w == 1.0)
    for r in range(k):
        p, hr = _expert_direct(gu, dn, 4, x[r:r + 1])
        assert np.array_equal(h[r, 0], hr)
        np.testing.assert_allclose(y[r], p, rtol=0, atol=1e-12)


def test_gather_combines_experts_with_route_weights_in_rank_order():
    gu, dn = _moe_case(22)
    k, E, T = 2, 6, 3
    x = S.bf16_normal(22, "pin.moe.x2", (k, 128))
    logits = np.array([[0.1, 1.5, -0.3, 0.9, 0.2, -2.0], [2.0, -1.0, 0.5, 0.4, 1.1, 0.0]], np.float32)
    idx, w, y, _ = O.gather_experts((gu.packed, gu.scales, gu.biases), (dn.packed, dn.scales, dn.biases),
                                    logits, T, x)
    assert list(idx[0]) == [1, 3, 4] and list(idx[1]) == [0, 4, 2]
    for r in range(k):
        l = logits[r, idx[r]].astype(np.float64)
        np.testing.assert_allclose(w[r], np.exp(l) / np.exp(l).sum(), rtol=1e-14)
        ref = sum(w[r, j] * _expert_direct(gu, dn, idx[r, j], x[r:r + 1])[0] for j in range(T))
        np.testing.assert_allclose(y[r], ref, rtol=0, atol=1e-12)


def test_gather_expert_permutation_invariance():
    """Relabelling the experts (stack and logit columns together) changes
    the indices only."""
    gu, dn = _moe_case(23)
    k, E, T = 3, 6, 2
    x = S.bf16_normal(23, "pin.moe.x3", (k, 128))
    logits = S.f32_normal(23, "pin.moe.l3", (k, E))
    perm = np.array([3, 0, 5, 1, 4, 2])
    base = O.gather_experts((gu.packed, gu.scales, gu.biases), (dn.packed, dn.scales, dn.biases), logits, T, x)
    pm = O.gather_experts((gu.packed[perm], gu.scales[perm], gu.biases[perm]),
                          (dn.packed[perm], dn.scales[perm], dn.biases[perm]), logits[:, perm], T, x)
    assert np.array_equal(perm[pm[0]], base[0])
    assert np.array_equal(pm[2], base[2])


def test_gather_shared_expert_adds_sigmoid_gated_dense_expert():
    """[F] 2.3: 10 routed + 1 shared expert; the shared one is sigmoid-gated."""
    gu, dn = _moe_case(24)
    k, E, T = 2, 6, 2
    x = S.bf16_normal(24, "pin.moe.x4", (k, 128))
    logits = S.f32_normal(24, "pin.moe.l4", (k, E))
    sgl = np.array([0.3, -1.2], np.float32)
    args = ((gu.packed, gu.scales, gu.biases), (dn.packed, dn.scales, dn.biases), logits, T, x)
    shared = ((gu.packed[5], gu.scales[5], gu.biases[5]), (dn.packed[5], dn.scales[5], dn.biases[5]))
    _, _, y0, _ = O.gather_experts(*args)
    _, _, y1, h1 = O.gather_experts(*args, shared=shared, shared_logit=sgl)
    for r in range(k):
        p, hr = _expert_direct(gu, dn, 5, x[r:r + 1])
        assert np.array_equal(h1[r, T], hr)
        np.testing.assert_allclose(y1[r] - y0[r], p / (1.0 + math.exp(-float(sgl[r]))), atol=1e-12)


# ------------------------------------------------------------ Gated DeltaNet

def _gdn_setup(seed, Hk=2, Hv=2, d=32, k=1, s_std=0.0, tail_std=0.0):
    p = S.gdn_params(seed, "pin.gdn", Hk, Hv, d)
    inp = S.gdn_inputs(seed, "pin.gdn", k, Hk, Hv, d)
    S0, tail = S.gdn_initial_state(seed, "pin.gdn", Hk, Hv, d, s_std=s_std, tail_std=tail_std)
    return p, inp, S0.astype(np.float64), tail


def _current_tap_only(p):
    p["conv_w"][:] = 0.0
    p["conv_w"][:, 3] = 1.0


def test_gdn_zero_state_unit_decay_closed_form():
    """S0 = 0, g = 1, conv = current tap only, one row:  y = beta (k.q) v with
    q = l2(silu(x_q)) * q_scale, k = l2(silu(x_k)), v = silu(x_v)
    ([F] 2.1 steps 1-5 collapse to this when the state starts at zero)."""
    Hk = Hv = 2
    d = 32
    p, inp, S0, tail = _gdn_setup(31, Hk, Hv, d)
    _current_tap_only(p)
    p["A_log"][:] = -40.0
    o, Ss, _, info = O.gdn_verify(Hk, Hv, d, p, S0, tail, inp, 1, debug=True)
    x = bfv(inp["qkv"][0])
    c = _silu(x)
    qs = 1.0 / math.sqrt(d)
    for h in range(Hv):
        qr, kr = c[h * d:(h + 1) * d], c[Hk * d + h * d:Hk * d + (h + 1) * d]
        qn = qr / math.sqrt(qr @ qr + 1e-6) * qs
        kn = kr / math.sqrt(kr @ kr + 1e-6)
        v = c[2 * Hk * d + h * d:2 * Hk * d + (h + 1) * d]
        beta = 1.0 / (1.0 + math.exp(-float(bfv(inp["b"][0, h]))))
        y = beta * (kn @ qn) * v
        np.testing.assert_allclose(info["y"][0, h], y, rtol=1e-12, atol=1e-15)
        # the state after the row is the rank-1 update beta * v k^T
        np.testing.assert_allclose(Ss[0, h], beta * np.outer(v, kn), rtol=1e-12, atol=1e-15)
        z = bfv(inp["z"][0, h * d:(h + 1) * d])
        on = y / math.sqrt(np.mean(y * y) + 1e-6) * p["norm_w"] / (1.0 + np.exp(-z))
        np.testing.assert_allclose(o[0, h * d:(h + 1) * d], on, rtol=1e-12, atol=1e-15)


def test_gdn_delta_rule_writes_v_along_k():
    """beta = 1, g = 1, |k| = 1 (up to l2_eps): after the update S k = v, for any
    prior state ([F] 2.1 steps 2-4: delta = v - S k).  A transposed update
    (S[j][i] += delta_i k_j) fails this."""
    p, inp, S0, tail = _gdn_setup(32, s_std=0.3)
    p["A_log"][:] = -40.0
    inp["b"][:] = bf16(40.0)
    o, Ss, _, info = O.gdn_verify(2, 2, 32, p, S0, tail, inp, 1, l2_eps=0.0, debug=True)
    for h in range(2):
        kn = info["k"][0, h]
        np.testing.assert_allclose(Ss[0, h] @ kn, info["v"][0, h], rtol=1e-12, atol=1e-13)


def _golden_decay_cases():
    rows = []
    with open(os.path.join(GOLDEN, "gdn_decay.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                rows.append([float(t) for t in line.split()])
    return rows


@pytest.mark.parametrize("case", _golden_decay_cases())
def test_gdn_decay_closed_form_with_beta_zero(case):
    """beta -> 0 leaves only the decay S <- g S; g = exp(-exp(A_log) *
    softplus(a + dt_bias)) takes the closed-form values in golden/gdn_decay.txt
    (0.5 when everything is 0, since softplus(0) = ln 2)."""
    A_log, a, dt_bias, g_expected = case
    p, inp, S0, tail = _gdn_setup(33, s_std=0.5)
    p["A_log"][:] = A_log
    p["dt_bias"][:] = dt_bias
    inp["a"][:] = bf16(a)
    inp["b"][:] = bf16(-60.0)
    _, Ss, _, info = O.gdn_verify(2, 2, 32, p, S0, tail, inp, 1, debug=True)
    np.testing.assert_allclose(info["g"][0], g_expected, rtol=1e-12)
    np.testing.assert_allclose(Ss[0], g_expected * S0, rtol=1e-12, atol=1e-20)
    for h in range(2):
        np.testing.assert_allclose(info["y"][0, h], Ss[0, h] @ info["q"][0, h], rtol=1e-12, atol=1e-15)


@pytest.mark.parametrize("tap", [0, 1, 2, 3])
def test_gdn_conv_taps_and_window_slide(tap):
    """One-hot conv weights pick one window entry: window of row r = the 3 tail
    rows followed by rows 0..r, last 4 ([F] 3.1: 3-tap history + current)."""
    k = 3
    p, inp, S0, tail = _gdn_setup(34, k=k, tail_std=1.0)
    p["conv_w"][:] = 0.0
    p["conv_w"][:, tap] = 1.0
    _, _, tails, info = O.gdn_verify(2, 2, 32, p, S0, tail, inp, k, debug=True)
    hist = np.concatenate([tail, inp["qkv"]], axis=0)  # rows: tail0, tail1, tail2, x0, x1, x2
    C = hist.shape[1]
    for r in range(k):
        want = _silu(bfv(hist[r + tap]))
        np.testing.assert_allclose(info["v"][r].ravel(), want[2 * 2 * 32:], rtol=1e-15)
        assert np.array_equal(tails[r], hist[r + 1:r + 4])
    assert tails.shape[2] == C


def test_gdn_v_heads_share_qk_heads_contiguously():
    """Hk = 2, Hv = 4: V heads 0,1 read QK head 0 and V heads 2,3 QK head 1
    ([F] 3.1: each k head shared by several v heads).  QK head 0 gets q
    orthogonal to k, so with S0 = 0 its V heads output exactly 0."""
    Hk, Hv, d = 2, 4, 32
    p, inp, S0, tail = _gdn_setup(35, Hk, Hv, d)
    _current_tap_only(p)
    p["A_log"][:] = -40.0
    x = np.zeros(2 * Hk * d + Hv * d, np.float32)
    x[0:d // 2] = 1.0            # q of QK head 0: first half
    x[Hk * d + d // 2:Hk * d + d] = 1.0  # k of QK head 0: second half -> q.k = 0
    x[d:2 * d] = 0.5             # q of QK head 1
    x[Hk * d + d:Hk * d + 2 * d] = 0.5   # k of QK head 1 == q
    x[2 * Hk * d:] = np.linspace(-1, 1, Hv * d)
    inp["qkv"][0] = bf16(x)
    _, _, _, info = O.gdn_verify(Hk, Hv, d, p, S0, tail, inp, 1, debug=True)
    assert np.all(info["y"][0, 0] == 0) and np.all(info["y"][0, 1] == 0)
    assert np.all(np.abs(info["y"][0, 2]) > 0) and np.all(np.abs(info["y"][0, 3]) > 0)


def test_gdn_norm_scales_and_gates():
    """L2 norms: |q| = q_scale |.|/sqrt(|.|^2+eps), |k| likewise without the
    scale.  Gated RMSNorm with z -> +inf (sigmoid 1): mean((o/w)^2) =
    ms/(ms+eps); with gate_act = silu and z = 0 the output is exactly 0."""
    p, inp, S0, tail = _gdn_setup(36, s_std=0.2)
    inp["z"][:] = bf16(60.0)
    o, _, _, info = O.gdn_verify(2, 2, 32, p, S0, tail, inp, 1, debug=True)
    qs = 1 / math.sqrt(32)
    for h in range(2):
        assert abs(np.linalg.norm(info["q"][0, h]) - qs) < 1e-6 * qs
        assert abs(np.linalg.norm(info["k"][0, h]) - 1.0) < 1e-6
        y = info["y"][0, h]
        ms = np.mean(y * y)
        on = o[0, h * 32:(h + 1) * 32] / p["norm_w"]
        assert abs(np.mean(on * on) - ms / (ms + 1e-6)) < 1e-12
    inp["z"][:] = 0
    o2, _, _, _ = O.gdn_verify(2, 2, 32, p, S0, tail, inp, 1, gate_act=1, debug=True)
    assert np.all(o2 == 0)


def test_gdn_k_rows_equal_k_single_row_steps_and_rollback_prefix():
    """[R] "What it is": row r runs from row r-1's state, snapshots after each
    row; rolling back to snapshot a (pointer swap) leaves exactly the state a
    fresh a-row verify reaches."""
    Hk, Hv, d, k = 2, 4, 32, 5
    p, inp, S0, tail = _gdn_setup(37, Hk, Hv, d, k=k, s_std=0.1, tail_std=1.0)
    o, Ss, ts = O.gdn_verify(Hk, Hv, d, p, S0, tail, inp, k)
    st, tl = S0, tail
    for r in range(k):
        one = {key: val[r:r + 1] for key, val in inp.items()}
        o1, S1, t1 = O.gdn_verify(Hk, Hv, d, p, st, tl, one, 1)
        assert np.array_equal(o1[0], o[r]) and np.array_equal(S1[0], Ss[r]) and np.array_equal(t1[0], ts[r])
        st, tl = S1[0], t1[0]
    for a in range(1, k + 1):
        pre = {key: val[:a] for key, val in inp.items()}
        _, Sa, ta = O.gdn_verify(Hk, Hv, d, p, S0, tail, pre, a)
        assert np.array_equal(Sa[a - 1], Ss[a - 1]) and np.array_equal(ta[a - 1], ts[a - 1])


# ------------------------------------------------------------------ glue

def test_rmsnorm_forms():
    """[F] 2.4: zero-centred y*(1+w) (w = 0 -> unit RMS) vs conventional y*w."""
    x = S.f32_normal(41, "pin.rms", (3, 64)).astype(np.float64) * 3.0
    w = np.zeros(64, np.float32)
    out = O.rmsnorm(x, w, eps=0.0, zero_centered=True)
    np.testing.assert_allclose(np.sqrt(np.mean(out * out, axis=1)), 1.0, rtol=1e-14)
    w2 = S.f32_uniform(41, "pin.rmsw", (64,), -0.5, 0.5)
    a = O.rmsnorm(x, w2, eps=1e-6, zero_centered=True)
    b = O.rmsnorm(x, (1.0 + w2.astype(np.float64)).astype(np.float32), eps=1e-6, zero_centered=False)
    np.testing.assert_allclose(a, b, rtol=1e-7)


def test_bf16_rounding_is_nearest_even():
    """The oracle's float64 -> bf16 rounding against exact midpoints."""
    one = 1.0
    ulp = 2.0 ** -7
    assert O.round_bf16(one + ulp / 2) == 0x3F80          # tie -> even (1.0)
    assert O.round_bf16(one + 1.5 * ulp) == 0x3F82        # tie -> even (1 + 2ulp)
    assert O.round_bf16(one + ulp / 2 + 2 ** -30) == 0x3F81
    assert O.round_bf16(-(one + ulp / 2)) == 0xBF80
    vals = S.f32_normal(42, "pin.bf16", (1000,))
    assert np.array_equal(O.to_bf16(vals.astype(np.float64)), S.f32_to_bf16(vals))
