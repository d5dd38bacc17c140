"""GPU parity of the dense width-k Q4 product (q4_qmv_k) against the CPU oracle.

Pages: "Flash-Next optimization transfer to Ornith and Qwen 27B", section
"Exact verification kernels" (widths 4/8/9 agree exactly with serial QMV) and
"Red Lite dev45 - speculative decoding with the Qwen3-Next MTP block", "What it
is" (each row in exactly the 1-row kernel's order).
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


def run_qmv(vf, W, x_dev, k, N, dtype=B.F32, y=None):
    import torch

    if y is None:
        y = torch.zeros((k, N), dtype=torch.float32 if dtype != B.BF16 else torch.int16, device="cuda")
    vf.q4_qmv_k(W.struct, x_dev, k, y, dtype)
    torch.cuda.synchronize()
    return y


def test_tiny_projection_matches_oracle_widths_1_to_4(vf):
    """512 x 512, k = 1..4, seed 0 (the tiny workload)."""
    m = S.q4_matrix(0, "tiny.q4", 512, 512)
    W = DevQ4(vf, m)
    for k in range(1, 5):
        x = S.bf16_normal(0, f"tiny.x{k}", (k, 512))
        ref = O.q4_qmv(m.packed, m.scales, m.biases, x)
        y = host(run_qmv(vf, W, dev(x), k, 512))
        assert_close(y, ref, what=f"k={k}")


@pytest.mark.parametrize("N,K", [(1, 256), (96, 2560), (100, 640), (129, 1152), (300, 512), (1000, 2048),
                                 (200, 576), (130, 192), (5, 64)])
@pytest.mark.parametrize("k", [1, 5, 9, 16, 32])
def test_ragged_shapes_match_oracle(vf, N, K, k):
    m = S.q4_matrix(1, f"rag.{N}.{K}", N, K)
    W = DevQ4(vf, m)
    x = S.bf16_normal(1, f"rag.x.{N}.{K}.{k}", (k, K))
    ref = O.q4_qmv(m.packed, m.scales, m.biases, x)
    y = host(run_qmv(vf, W, dev(x), k, N))
    assert_close(y, ref, what=f"N={N} K={K} k={k}")


@pytest.mark.parametrize("N,K", [(512, 512), (100, 640), (1000, 2048), (5120, 5120)])
def test_width_k_rows_bit_identical_to_width_1(vf, N, K):
    m = S.q4_matrix(2, f"bit.{N}.{K}", N, K)
    W = DevQ4(vf, m)
    x = S.bf16_normal(2, f"bit.x.{N}.{K}", (32, K))
    xd = dev(x)
    singles = [host(run_qmv(vf, W, dev(x[r:r + 1]), 1, N))[0] for r in range(32)]
    for k in (2, 4, 8, 9, 16, 17, 32):
        y = host(run_qmv(vf, W, xd, k, N))
        for r in range(k):
            assert np.array_equal(y[r].view(np.uint32), singles[r].view(np.uint32)), f"k={k} row {r}"


def test_exact_integer_case_is_bitwise(vf):
    """Integer activations in -2..2, scale 2^-3, bias in {-1,0,1} 2^-4: every
    partial sum is exact in fp32, so the GPU must equal the oracle bit for bit."""
    rng = np.random.default_rng(5)
    N, K, k = 300, 2048, 9
    packed = rng.integers(0, 2 ** 32, size=(N, K // 8), dtype=np.uint64).astype(np.uint32)
    scales = np.full((N, K // 64), S.f32_to_bf16(np.float32(0.125)), np.uint16)
    biases = S.f32_to_bf16((rng.integers(-1, 2, size=(N, K // 64)) * 0.0625).astype(np.float32))
    x = S.f32_to_bf16(rng.integers(-2, 3, size=(k, K)).astype(np.float32))
    ref = O.q4_qmv(packed, scales, biases, x)
    W = DevQ4(vf, S.Q4Matrix(packed, scales, biases, N, K))
    y = host(run_qmv(vf, W, dev(x), k, N))
    assert np.array_equal(y.astype(np.float64), ref)


def test_bf16_and_accumulate_outputs(vf):
    import torch

    m = S.q4_matrix(3, "dt.q4", 640, 1024)
    W = DevQ4(vf, m)
    x = dev(S.bf16_normal(3, "dt.x", (7, 1024)))
    y32 = host(run_qmv(vf, W, x, 7, 640))
    y16 = host(run_qmv(vf, W, x, 7, 640, dtype=B.BF16), np.uint16)
    assert np.array_equal(y16, S.f32_to_bf16(y32))
    base = torch.from_numpy(S.f32_normal(3, "dt.base", (7, 640))).cuda()
    want = host(base) + y32
    yadd = host(run_qmv(vf, W, x, 7, 640, dtype=B.F32_ADD, y=base.clone()))
    assert np.array_equal(yadd, want.astype(np.float32))


@pytest.mark.parametrize("N,K", S.DENSE_SHAPES + [S.LM_HEAD])
def test_dense_full_size_sampled_rows(vf, N, K):
    """The Qwen-27B-shaped projections and the Flash-Next-shaped LM head
    (248,320 x 2560, the full vocabulary) at full size, weights drawn on the
    device; the oracle recomputes 48 sampled output rows drawn on the host."""
    import torch

    name = f"dense.{N}x{K}"
    sp, ss, sb = S.q4_seeds(0, name)
    packed = torch.empty((N, K // 8), dtype=torch.int32, device="cuda")
    scales = torch.empty((N, K // 64), dtype=torch.int16, device="cuda")
    biases = torch.empty((N, K // 64), dtype=torch.int16, device="cuda")
    vf.synth_q4(packed, scales, biases, (sp, ss, sb), S.SCALE_RANGE, S.BIAS_RANGE)
    Wt = vf.tile(B.q4_weight(packed, scales, biases))
    W = Wt.struct
    x = S.bf16_normal(0, name + ".x", (32, K))
    rows = np.unique(np.concatenate([[0, N - 1], np.random.default_rng(N + K).integers(0, N, 46)]))
    sub = S.q4_rows(0, name, N, K, rows)
    # the device generator reproduces the host draw bit for bit
    assert np.array_equal(host(packed[rows.tolist()]).view(np.uint32), sub.packed)
    assert np.array_equal(host(scales[rows.tolist()]).view(np.uint16), sub.scales)
    ref = O.q4_qmv(sub.packed, sub.scales, sub.biases, x)
    for k in S.DENSE_WIDTHS + [16, 32]:
        y = torch.zeros((k, N), dtype=torch.float32, device="cuda")
        vf.q4_qmv_k(W, dev(x[:k]), k, y, B.F32)
        torch.cuda.synchronize()
        assert_close(host(y)[:, rows], ref[:k], what=f"{name} k={k}")
        if k in (9, 32):  # a row of the second column block, and one of the second pass
            r = k - 1
            y1 = torch.zeros((1, N), dtype=torch.float32, device="cuda")
            vf.q4_qmv_k(W, dev(x[r:r + 1]), 1, y1, B.F32)
            torch.cuda.synchronize()
            assert torch.equal(y[r], y1[0])


def test_argument_errors_are_reported_before_launch(vf):
    import torch

    m = S.q4_matrix(4, "err.q4", 128, 512)
    W = DevQ4(vf, m)
    x = dev(S.bf16_normal(4, "err.x", (2, 512)))
    y = torch.zeros((2, 128), device="cuda")
    before = vf.launch_count()
    with pytest.raises(B.VerifyError) as e:
        vf.q4_qmv_k(W.struct, x, 0, y)
    assert e.value.status == B.EUNSUPPORTED
    with pytest.raises(B.VerifyError) as e:
        vf.q4_qmv_k(W.struct, x, 33, y)  # wider than VERIFY_MAX_K
    assert e.value.status == B.EUNSUPPORTED
    hx = torch.zeros((2, 512), dtype=torch.int16)  # host memory
    with pytest.raises(B.VerifyError) as e:
        vf.q4_qmv_k(W.struct, hx, 2, y)
    assert e.value.status == B.EINVAL
    bad = B.Q4Weight(W.struct.packed, None, None, 128, 520, 64, 4, B.TILED)  # k_in % 64 != 0
    with pytest.raises(B.VerifyError) as e:
        vf.q4_qmv_k(bad, x, 2, y)
    assert e.value.status == B.EUNSUPPORTED
    bad = B.Q4Weight(W.struct.packed, None, None, 128, 512, 32, 4, B.TILED)  # group 32
    with pytest.raises(B.VerifyError) as e:
        vf.q4_qmv_k(bad, x, 2, y)
    assert e.value.status == B.EUNSUPPORTED
    with pytest.raises(B.VerifyError) as e:  # the row layout is only an input of q4_tile
        vf.q4_qmv_k(W.rows, x, 2, y)
    assert e.value.status == B.EINVAL
    assert vf.launch_count() == before
