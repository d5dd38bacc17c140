"""GPU parity of the layer norm glue (verify_rmsnorm_k) against the CPU oracle.

Page: "QWEN38FLASH.md - Plan for supporting Qwen/Qwen3.8-Flash-Next", 2.4
(non-gated norms are zero-centred, y*(1+w))."""
import numpy as np
import pytest

from oracle import oracle as O
from speculative_decode_verification_gb300 import binding as B
from speculative_decode_verification_gb300 import synth as S
from tests.gpu_util import assert_close, dev, host

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("zc", [True, False])
@pytest.mark.parametrize("n,k", [(2560, 9), (5120, 1), (64, 3)])
def test_rmsnorm_matches_oracle(zc, n, k):
    import torch

    vf = B.Verify(0)
    x = S.f32_normal(20, f"rms.x{n}", (k, n)) * 2.0
    w = S.f32_uniform(20, f"rms.w{n}", (n,), -0.1, 0.1)
    out = torch.zeros((k, n), dtype=torch.float32, device="cuda")
    vf.verify_rmsnorm_k(dev(x), dev(w), 1e-6, zc, n, k, out, B.F32)
    out16 = torch.zeros((k, n), dtype=torch.int16, device="cuda")
    vf.verify_rmsnorm_k(dev(x), dev(w), 1e-6, zc, n, k, out16, B.BF16)
    torch.cuda.synchronize()
    ref = O.rmsnorm(x.astype(np.float64), w, 1e-6, zc)
    assert_close(host(out), ref)
    assert np.array_equal(host(out16, np.uint16), S.f32_to_bf16(host(out)))
    vf.close()
