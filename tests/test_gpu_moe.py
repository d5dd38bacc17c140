"""GPU parity of the routed experts (q4_gather_experts_k) against the CPU oracle.

Pages: "Flash-Next optimization transfer to Ornith and Qwen 27B", section
"Exact verification kernels" (gathered affine-Q4 experts, top-8 of 256,
2048/512, fused gate/up, widths 2..9); "Red Lite dev45 - speculative decoding
with the Qwen3-Next MTP block", "What it is" (all (expert,row) pairs in one
dispatch, one tail); "QWEN38FLASH.md - Plan for supporting
Qwen/Qwen3.8-Flash-Next", 2.3 (512 experts, 10 routed + 1 shared, 640).
"""
import numpy as np
import pytest

from oracle import oracle as O
from speculative_decode_verification_gb300 import binding as B
from speculative_decode_verification_gb300 import synth as S
from tests.gpu_util import DevQ4, assert_close, dev, host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def vf():
    import torch

    assert torch.cuda.is_available()
    v = B.Verify(0)
    yield v
    st, code = v.device_status()
    assert st == B.OK, f"device error word {code}"
    v.close()


def gather(vf, gu, dn, logits, T, x, k, H, shared=None, dtype=B.F32):
    import torch

    idx = torch.zeros((k, T), dtype=torch.int32, device="cuda")
    w = torch.zeros((k, T), dtype=torch.float32, device="cuda")
    y = torch.zeros((k, H), dtype=torch.float32 if dtype != B.BF16 else torch.int16, device="cuda")
    E = logits.shape[1]
    if shared is None:
        vf.q4_gather_experts_k(gu.struct, dn.struct, logits, E, T, x, k, idx, w, y, dtype)
    else:
        sgu, sdn, sl = shared
        vf.q4_gather_experts_k(gu.struct, dn.struct, logits, E, T, x, k, idx, w, y, dtype,
                               sgu.struct, sdn.struct, sl)
    torch.cuda.synchronize()
    return host(idx), host(w), host(y)


def moe_case(seed, E, H, I):
    gu = S.q4_matrix(seed, "moe.gu", 2 * I, H, n_experts=E)
    dn = S.q4_matrix(seed, "moe.dn", H, I, n_experts=E)
    return gu, dn


@pytest.mark.parametrize("k", [1, 2, 5, 9, 16, 25, 32])
def test_small_moe_matches_oracle(vf, k):
    E, H, I, T = 16, 256, 256, 4
    gu, dn = moe_case(10, E, H, I)
    x = S.bf16_normal(10, f"moe.x{k}", (k, H))
    logits = S.f32_normal(10, f"moe.l{k}", (k, E))
    oi, ow, oy, _ = O.gather_experts((gu.packed, gu.scales, gu.biases), (dn.packed, dn.scales, dn.biases),
                                     logits, T, x)
    gud, dnd = DevQ4(vf, gu, True), DevQ4(vf, dn, down=True)
    before = vf.launch_count()
    gi, gw, gy = gather(vf, gud, dnd, dev(logits), T, dev(x), k, H)
    # the routing kernel, the routed experts kernel, then the combine, per pass of up to 16 rows
    assert vf.launch_count() - before == 3 * ((k + 15) // 16)
    assert np.array_equal(gi, oi)
    np.testing.assert_allclose(gw, ow, rtol=1e-5, atol=1e-6)
    assert_close(gy, oy, what=f"k={k}")


def test_routing_ties_and_crowded_lanes(vf):
    """Top-16 of 512 with many equal logits (ties -> lower expert index) and a
    row whose largest logits all sit at experts 3, 35, 67, ... (one lane of
    the warp holds every winner): indices equal the oracle's bit for bit."""
    E, H, I, T, k = 512, 256, 128, 16, 6
    gu, dn = moe_case(14, E, H, I)
    x = S.bf16_normal(14, "moe.t.x", (k, H))
    lg = np.round(S.f32_normal(14, "moe.t.l", (k, E)) * 2.0) / 2.0  # coarse grid: many ties
    lg[1, :] = 0.0
    lg[2, 3::32] = 5.0 + np.arange(16, dtype=np.float32) / 64.0  # 16 winners in one lane
    lg[3, 3::32] = 7.0  # 16 equal winners in one lane
    lg[4, :] = -0.0
    lg = lg.astype(np.float32)
    oi, ow, oy, _ = O.gather_experts((gu.packed, gu.scales, gu.biases), (dn.packed, dn.scales, dn.biases),
                                     lg, T, x)
    gi, gw, gy = gather(vf, DevQ4(vf, gu, True), DevQ4(vf, dn, down=True), dev(lg), T, dev(x), k, H)
    assert np.array_equal(gi, oi)
    np.testing.assert_allclose(gw, ow, rtol=1e-5, atol=1e-6)
    assert_close(gy, oy, what="ties")


@pytest.mark.parametrize("k", [3, 9])
def test_moe_with_k_not_a_multiple_of_128(vf, k):
    """H = 320 and I = 192: partial 256-column chunks on both products and a
    ragged last 128-row tile of the down product."""
    E, H, I, T = 12, 320, 192, 3
    gu, dn = moe_case(12, E, H, I)
    x = S.bf16_normal(12, f"moe.r.x{k}", (k, H))
    logits = S.f32_normal(12, f"moe.r.l{k}", (k, E))
    oi, ow, oy, _ = O.gather_experts((gu.packed, gu.scales, gu.biases), (dn.packed, dn.scales, dn.biases),
                                     logits, T, x)
    gi, gw, gy = gather(vf, DevQ4(vf, gu, True), DevQ4(vf, dn, down=True), dev(logits), T, dev(x), k, H)
    assert np.array_equal(gi, oi)
    assert_close(gy, oy, what=f"H=320 I=192 k={k}")


def test_shared_expert_and_ragged_down(vf):
    """640-wide intermediate (ragged last 256-column chunk), 10 routed + 1 shared."""
    E, H, I, T, k = 24, 384, 640, 10, 9
    gu, dn = moe_case(11, E, H, I)
    sgu = S.q4_matrix(11, "moe.sgu", 2 * I, H)
    sdn = S.q4_matrix(11, "moe.sdn", H, I)
    x = S.bf16_normal(11, "moe.xs", (k, H))
    logits = S.f32_normal(11, "moe.ls", (k, E))
    sl = S.f32_normal(11, "moe.sl", (k,))
    oi, ow, oy, _ = O.gather_experts((gu.packed, gu.scales, gu.biases), (dn.packed, dn.scales, dn.biases),
                                     logits, T, x, shared=((sgu.packed, sgu.scales, sgu.biases),
                                                           (sdn.packed, sdn.scales, sdn.biases)),
                                     shared_logit=sl)
    # the shared gate logit is read at row stride logits_ld = E: store it in a [k, E] array
    slm = np.zeros((k, E), np.float32)
    slm[:, 0] = sl
    gi, gw, gy = gather(vf, DevQ4(vf, gu, True), DevQ4(vf, dn, down=True), dev(logits), T, dev(x), k, H,
                        shared=(DevQ4(vf, sgu, True), DevQ4(vf, sdn, down=True), dev(slm)))
    assert np.array_equal(gi, oi)
    assert_close(gy, oy, what="shared")


def test_width_k_rows_bit_identical_to_width_1(vf):
    E, H, I, T = 32, 512, 256, 8
    gu, dn = moe_case(12, E, H, I)
    G, D = DevQ4(vf, gu, True), DevQ4(vf, dn, down=True)
    x = S.bf16_normal(12, "moe.xb", (9, H))
    logits = S.f32_normal(12, "moe.lb", (9, E))
    _, _, y9 = gather(vf, G, D, dev(logits), T, dev(x), 9, H)
    for r in range(9):
        _, _, y1 = gather(vf, G, D, dev(logits[r:r + 1]), T, dev(x[r:r + 1]), 1, H)
        assert np.array_equal(y9[r].view(np.uint32), y1[0].view(np.uint32)), f"row {r}"


def test_single_expert_reduces_to_dense_products(vf):
    """T = 1, every row routed to one expert: the routed path equals the dense
    gate/up product, SwiGLU in bf16 and the dense down product."""
    import torch

    E, H, I, k = 8, 256, 256, 4
    gu, dn = moe_case(13, E, H, I)
    logits = np.full((k, E), -2.0, np.float32)
    logits[:, 5] = 3.0
    x = S.bf16_normal(13, "moe.x1", (k, H))
    gi, gw, gy = gather(vf, DevQ4(vf, gu, True), DevQ4(vf, dn, down=True), dev(logits), 1, dev(x), k, H)
    assert np.all(gi == 5) and np.all(gw == 1.0)
    Wg = DevQ4(vf, S.Q4Matrix(gu.packed[5], gu.scales[5], gu.biases[5], 2 * I, H))
    Wd = DevQ4(vf, S.Q4Matrix(dn.packed[5], dn.scales[5], dn.biases[5], H, I))
    g = torch.zeros((k, 2 * I), device="cuda")
    vf.q4_qmv_k(Wg.struct, dev(x), k, g)
    torch.cuda.synchronize()
    gh = host(g).astype(np.float32)
    gate, up = gh[:, :I], gh[:, I:]
    h = S.f32_to_bf16((gate / (1.0 + np.exp(-gate))) * up)
    yd = torch.zeros((k, H), device="cuda")
    vf.q4_qmv_k(Wd.struct, dev(h), k, yd)
    torch.cuda.synchronize()
    assert_close(gy, host(yd), tol=1e-5, what="single expert")


def test_ornith_shape_matches_oracle(vf):
    """256 experts, H 2048, I 512, top-8, at every width k = 2..9 (routes
    differ per row); then every row of the 9-row call against a 1-row call
    on that row, bit for bit."""
    import torch

    c = S.ORNITH_MOE
    E, T, H, I = c["E"], c["T"], c["H"], c["I"]
    seeds_gu, seeds_dn = S.q4_seeds(0, "ornith.gu"), S.q4_seeds(0, "ornith.dn")
    gu_p = torch.empty((E, 2 * I, H // 8), dtype=torch.int32, device="cuda")
    gu_s = torch.empty((E, 2 * I, H // 64), dtype=torch.int16, device="cuda")
    gu_b = torch.empty_like(gu_s)
    dn_p = torch.empty((E, H, I // 8), dtype=torch.int32, device="cuda")
    dn_s = torch.empty((E, H, I // 64), dtype=torch.int16, device="cuda")
    dn_b = torch.empty_like(dn_s)
    vf.synth_q4(gu_p, gu_s, gu_b, seeds_gu, S.SCALE_RANGE, S.BIAS_RANGE)
    vf.synth_q4(dn_p, dn_s, dn_b, seeds_dn, S.SCALE_RANGE, S.BIAS_RANGE)

    G = vf.tile(B.q4_experts(gu_p, gu_s, gu_b), gate_up=True)
    D = vf.tile(B.q4_experts(dn_p, dn_s, dn_b), down=True)
    experts = {}

    def expert(e):
        if e not in experts:
            experts[e] = (S.q4_expert(0, "ornith.gu", 2 * I, H, e), S.q4_expert(0, "ornith.dn", H, I, e))
        return experts[e]

    for k in range(2, 10):
        x = S.bf16_normal(0, f"ornith.x{k}", (k, H))
        logits = S.f32_normal(0, f"ornith.l{k}", (k, E))
        gi, gw, gy = gather(vf, G, D, dev(logits), T, dev(x), k, H)
        oi, ow = O.route_topk(logits, T)
        assert np.array_equal(gi, oi)
        np.testing.assert_allclose(gw, ow, rtol=1e-5, atol=1e-6)
        ref = np.zeros((k, H))
        for r in range(k):
            for j in range(T):
                mg, md = expert(int(oi[r, j]))
                gate_up = O.q4_qmv(mg.packed, mg.scales, mg.biases, x[r:r + 1])[0]
                h = O.to_bf16(gate_up[:I] / (1.0 + np.exp(-gate_up[:I])) * gate_up[I:])
                ref[r] += ow[r, j] * O.q4_qmv(md.packed, md.scales, md.biases, h[None, :])[0]
        assert_close(gy, ref, what=f"ornith k={k}")
        if k == 9:
            for r in range(k):
                i1, w1, y1 = gather(vf, G, D, dev(logits[r:r + 1]), T, dev(x[r:r + 1]), 1, H)
                assert np.array_equal(i1[0], gi[r])
                assert np.array_equal(w1[0].view(np.uint32), gw[r].view(np.uint32)), f"ornith weights row {r}"
                assert np.array_equal(y1[0].view(np.uint32), gy[r].view(np.uint32)), f"ornith row {r}"


def test_width_32_rows_equal_single_rows(vf):
    """A 32-row call runs as two 16-row passes: every row's indices, weights
    and output equal a 1-row call on that row, bit for bit."""
    E, H, I, T, k = 64, 256, 256, 8, 32
    gu, dn = moe_case(15, E, H, I)
    x = S.bf16_normal(15, "moe.w32.x", (k, H))
    logits = S.f32_normal(15, "moe.w32.l", (k, E))
    gud, dnd = DevQ4(vf, gu, True), DevQ4(vf, dn, down=True)
    gi, gw, gy = gather(vf, gud, dnd, dev(logits), T, dev(x), k, H)
    for r in (0, 7, 15, 16, 24, 31):
        i1, w1, y1 = gather(vf, gud, dnd, dev(logits[r:r + 1]), T, dev(x[r:r + 1]), 1, H)
        assert np.array_equal(i1[0], gi[r]) and np.array_equal(w1[0].view(np.uint32), gw[r].view(np.uint32))
        assert np.array_equal(y1[0].view(np.uint32), gy[r].view(np.uint32)), f"row {r}"


@pytest.mark.parametrize("k", [1, 9])
def test_progress_beside_a_concurrent_kernel(vf, k):
    """The expert kernel's down items wait for their unit's gate/up items.  With
    another stream's long matmuls holding SMs, not every expert CTA is
    resident at once; the call must still finish without a wait running out
    (the device error word stays clear) and give a solo run's result bit for
    bit.  k = 1 has fewer gate/up items than CTAs."""
    import torch

    E, H, I, T = 64, 1024, 512, 8
    gu, dn = moe_case(16, E, H, I)
    G, D = DevQ4(vf, gu, True), DevQ4(vf, dn, down=True)
    x = dev(S.bf16_normal(16, f"moe.cc.x{k}", (k, H)))
    logits = dev(S.f32_normal(16, f"moe.cc.l{k}", (k, E)))
    ref = gather(vf, G, D, logits, T, x, k, H)
    a = torch.randn((8192, 8192), device="cuda", dtype=torch.bfloat16)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    for _ in range(3):
        with torch.cuda.stream(side):
            for _ in range(8):
                a = torch.matmul(a, a) * 1e-4
        got = gather(vf, G, D, logits, T, x, k, H)
        for g, r in zip(got, ref):
            assert np.array_equal(g.view(np.uint32), r.view(np.uint32))
    torch.cuda.synchronize()
    st, code = vf.device_status()
    assert st == B.OK, f"device error word {code}"
