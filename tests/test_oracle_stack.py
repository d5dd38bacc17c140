"""Pins of the oracle's layer composition (``oracle.stack_layer``) against
special cases that reduce the layer to something simpler.

The layer, as "QWEN38FLASH.md - Plan for supporting Qwen/Qwen3.8-Flash-Next"
section 2 defines it: a Gated DeltaNet mixer with a residual add (2.1, 2.4),
then a MoE of routed experts plus one sigmoid-gated shared expert with a
residual add (2.3), each half behind a zero-centred RMSNorm (2.4).  Each test
zeroes or replaces some of the layer's Q4 matrices so that the expected
output follows from a brute-force dense product computed here (nibbles
unpacked with numpy, float64 matmul), not from the oracle's own routines.
A plausible composition mistake (a dropped residual, routing from the
mixer's norm instead of the MoE's, an ungated or sign-flipped shared expert,
a wrong split of the in-projection, the out-projection fed the unrounded GDN
output) fails one of them.
"""
import numpy as np
import pytest

from oracle import oracle as O
from speculative_decode_verification_gb300 import synth as S
from speculative_decode_verification_gb300.stack import shapes

CFG = dict(layers=1, H=256, E=16, T=4, I=256, n_qk_heads=2, n_v_heads=4, d=64, conv_kernel=4)
EPS = 1e-6


def _zero_q4(n, K):
    return (np.zeros((n, K // 8), np.uint32), np.zeros((n, K // 64), np.uint16),
            np.zeros((n, K // 64), np.uint16))


def _identity_q4(n):
    """w = I exactly: code 1 on the diagonal, scale 1.0, bias 0."""
    packed, scales, biases = _zero_q4(n, n)
    for i in range(n):
        packed[i, i // 8] |= np.uint32(1 << (4 * (i % 8)))
    scales[:] = 0x3F80  # bf16 1.0
    return packed, scales, biases


def _bf(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def dequant(m):
    """Brute force: float64 [N, K] weights w = s*q + b from the row layout."""
    packed, scales, biases = (np.asarray(a) for a in m)
    n = packed.shape[0]
    q = (packed[:, :, None].astype(np.uint64) >> (4 * np.arange(8, dtype=np.uint64))) & 15
    q = q.reshape(n, -1).astype(np.float64)
    s = np.repeat(_bf(scales), 64, axis=1)
    b = np.repeat(_bf(biases), 64, axis=1)
    return s * q + b


def norm_zc(h, w):
    h = np.asarray(h, np.float64)
    return h / np.sqrt(np.mean(h * h, axis=1, keepdims=True) + EPS) * (1.0 + np.asarray(w, np.float64))


def swiglu_expert(gu, dn, x_bits):
    """Dense SwiGLU expert on bf16 rows: h = bf16(silu(g) * u), then down . h."""
    W = dequant(gu)
    I = W.shape[0] // 2
    gu_out = _bf(x_bits) @ W.T
    g, u = gu_out[:, :I], gu_out[:, I:]
    hmid = O.to_bf16(g / (1.0 + np.exp(-g)) * u)
    return _bf(hmid) @ dequant(dn).T


class Layer:
    """The synthetic stack's layer 0 with some matrices replaced."""

    def __init__(self, seed=0, zero_out_proj=False, identity_out_proj=False, zero_routed=False,
                 zero_shared=False):
        sh = shapes(CFG)
        self.sh = sh
        base = S.HostLayerWeights(seed, 0, sh["H"], sh["NP"], sh["Z"], sh["E"], sh["I"], CFG["n_qk_heads"],
                                  CFG["n_v_heads"], CFG["d"])
        self.base = base
        self.in_proj, self.router, self.gdn = base.in_proj, base.router, base.gdn
        self.norm1, self.norm2 = base.norm1, base.norm2
        H, Z, I = sh["H"], sh["Z"], sh["I"]
        self.out_proj = base.out_proj
        if zero_out_proj:
            self.out_proj = _zero_q4(H, Z)
        if identity_out_proj:
            assert Z == H
            self.out_proj = _identity_q4(H)
        self.shared_gate_up, self.shared_down = base.shared_gate_up, base.shared_down
        if zero_shared:
            self.shared_gate_up, self.shared_down = _zero_q4(2 * I, H), _zero_q4(H, I)
        self.zero_routed = zero_routed

    def expert(self, e):
        if self.zero_routed:
            H, I = self.sh["H"], self.sh["I"]
            return _zero_q4(2 * I, H), _zero_q4(H, I)
        return self.base.expert(e)


def _inputs(seed, k):
    sh = shapes(CFG)
    h = S.f32_normal(seed, "pin.stack.h", (k, sh["H"])).astype(np.float64)
    S0, t0 = S.gdn_initial_state(seed, "pin.stack.gdn", CFG["n_qk_heads"], CFG["n_v_heads"], CFG["d"],
                                 s_std=0.02, tail_std=1.0)
    return h, S0.astype(np.float64), t0


def _run(w, h, S0, t0, k, T=None):
    return O.stack_layer(w, h, S0, t0, k, CFG["n_qk_heads"], CFG["n_v_heads"], CFG["d"],
                         CFG["T"] if T is None else T)


def _router_logits(w, x_bits):
    return (_bf(x_bits) @ dequant(w.router).T).astype(np.float32)


@pytest.mark.parametrize("k", [1, 3])
def test_zero_products_keep_the_residual_exactly(k):
    """Out-projection and every expert (routed and shared) zero: both residual
    adds add exact zeros, so the layer returns its input bit for bit."""
    w = Layer(zero_out_proj=True, zero_routed=True, zero_shared=True)
    h, S0, t0 = _inputs(1, k)
    h_out, _, _, _, _ = _run(w, h, S0, t0, k)
    assert np.array_equal(h_out, h)


@pytest.mark.parametrize("k", [1, 4])
def test_shared_expert_only_adds_its_sigmoid_gated_output(k):
    """Zero out-projection (h unchanged by the mixer) and zero routed experts:
    the layer adds exactly sigmoid(l_E) * shared(bf16(norm2(h))), with l_E
    the router's last row applied to the same normalised rows."""
    w = Layer(zero_out_proj=True, zero_routed=True)
    h, S0, t0 = _inputs(2, k)
    h_out, _, _, _, lg = _run(w, h, S0, t0, k)
    x2 = O.to_bf16(norm_zc(h, w.norm2))
    l_ref = _router_logits(w, x2)
    np.testing.assert_allclose(lg, l_ref, rtol=1e-6, atol=1e-6)
    E = w.sh["E"]
    gate = 1.0 / (1.0 + np.exp(-lg[:, E].astype(np.float64)))
    want = gate[:, None] * swiglu_expert(w.shared_gate_up, w.shared_down, x2)
    np.testing.assert_allclose(h_out - h, want, rtol=1e-9, atol=1e-9 * np.abs(want).max())
    assert np.abs(want).max() > 1e-3  # the check is not vacuous


@pytest.mark.parametrize("k", [4, 9])
def test_router_reads_the_moe_norm_not_the_mixer_norm(k):
    """The routing input is the second (pre-MoE) norm of the residual after the
    mixer.  With a zero out-projection both norms see the same h and differ
    only by their weights; the layer's logits and routes must be those of the
    second; the first norm's logits differ well beyond the tolerance used."""
    w = Layer(zero_out_proj=True)
    h, S0, t0 = _inputs(3, k)
    _, _, _, idx, lg = _run(w, h, S0, t0, k)
    E, T = w.sh["E"], w.sh["T"]
    l2 = _router_logits(w, O.to_bf16(norm_zc(h, w.norm2)))
    l1 = _router_logits(w, O.to_bf16(norm_zc(h, w.norm1)))
    np.testing.assert_allclose(lg, l2, rtol=1e-6, atol=1e-6)

    def top(l):  # descending logit, ties to the lower index
        return np.stack([sorted(range(E), key=lambda e: (-float(l[r, e]), e))[:T] for r in range(k)])

    assert np.array_equal(idx, top(l2))
    assert np.abs(l1 - l2).max() > 1e3 * 1e-6 * np.abs(l2).max()


@pytest.mark.parametrize("k", [1, 5])
def test_top1_routing_adds_the_chosen_dense_expert(k):
    """Top-1 routing with a zero shared expert and zero out-projection: the
    routing weight is exactly 1, so the layer adds the dense SwiGLU expert of
    each row's largest logit, applied to bf16(norm2(h))."""
    w = Layer(zero_out_proj=True, zero_shared=True)
    h, S0, t0 = _inputs(4, k)
    h_out, _, _, idx, lg = _run(w, h, S0, t0, k, T=1)
    x2 = O.to_bf16(norm_zc(h, w.norm2))
    E = w.sh["E"]
    for r in range(k):
        e = int(np.argmax(lg[r, :E]))
        assert idx[r, 0] == e
        gu, dn = w.expert(e)
        want = swiglu_expert(gu, dn, x2[r:r + 1])[0]
        np.testing.assert_allclose(h_out[r] - h[r], want, rtol=1e-9, atol=1e-9 * np.abs(want).max())


@pytest.mark.parametrize("k", [1, 3])
def test_mixer_output_reaches_the_residual_through_out_proj(k):
    """Identity out-projection (w = I exactly) and zero experts: the layer adds
    exactly the bf16-rounded GDN output, where the GDN step takes the
    in-projection of bf16(norm1(h)) split as conv channels q|k|v, then z,
    then a, then b; its state snapshots are the layer's."""
    w = Layer(identity_out_proj=True, zero_routed=True, zero_shared=True)
    sh = w.sh
    h, S0, t0 = _inputs(5, k)
    h_out, S_snap, tail_snap, _, _ = _run(w, h, S0, t0, k)
    xn = O.to_bf16(norm_zc(h, w.norm1))
    p = O.to_bf16(_bf(xn) @ dequant(w.in_proj).T)
    C, Z, Hv = sh["C"], sh["Z"], CFG["n_v_heads"]
    inp = dict(qkv=p[:, :C], z=p[:, C:C + Z], a=p[:, C + Z:C + Z + Hv], b=p[:, C + Z + Hv:C + Z + 2 * Hv])
    o, S_ref, t_ref = O.gdn_verify(CFG["n_qk_heads"], Hv, CFG["d"], w.gdn, S0, t0, inp, k)
    want = _bf(O.to_bf16(o))
    np.testing.assert_allclose(h_out - h, want, rtol=1e-12, atol=1e-12 * np.abs(want).max())
    np.testing.assert_allclose(S_snap, S_ref, rtol=1e-12, atol=1e-15)
    assert np.array_equal(tail_snap, t_ref)
    # the split order matters: a swapped z / qkv split gives another output
    swapped = dict(inp, z=p[:, :Z], qkv=np.concatenate([p[:, Z:C], p[:, C:C + Z]], axis=1))
    o_bad, _, _ = O.gdn_verify(CFG["n_qk_heads"], Hv, CFG["d"], w.gdn, S0, t0, swapped, k)
    assert not np.allclose(_bf(O.to_bf16(o_bad)), want)


def test_threaded_oracle_build_is_bit_identical():
    """The OpenMP build (timing only) spreads output rows over the cores but
    sums every output in the same order: a whole layer gives the same bits."""
    k = 3
    w = Layer()
    h, S0, t0 = _inputs(6, k)
    O.use_threads(False)
    want = _run(w, h, S0, t0, k)
    try:
        if O.build_threaded() is None:
            pytest.skip("no OpenMP build of the oracle on this host")
        n = O.use_threads(True)
        got = _run(w, h, S0, t0, k)
    finally:
        O.use_threads(False)
    assert n >= 1
    for g, r in zip(got, want):
        assert np.array_equal(np.asarray(g), np.asarray(r))
