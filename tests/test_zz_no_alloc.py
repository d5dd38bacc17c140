"""The routed-expert entry point that allocates nothing
(q4_gather_experts_k_noalloc), called through the C ABI, against the
regular entry point (q4_gather_experts_k).

It serves callers that may not allocate device memory (memory owned by a
host framework's arena; loops where cudaMalloc would synchronise the device):
its scratch is a fixed array inside the library.  The file name makes pytest
collect it last, so a run that stops at the first failure has run everything
else first; it also passes on its own in a fresh process.
"""
import ctypes as C

import numpy as np
import pytest

from speculative_decode_verification_gb300 import binding as B
from speculative_decode_verification_gb300 import synth as S
from tests.gpu_util import DevQ4, assert_close, dev, host

pytestmark = pytest.mark.gpu


def _noalloc(lib, gu, dn, logits, E, T, x, k, idx, w, y, shared=None, err=None, dtype=B.F32):
    import torch

    sgu, sdn, sl = shared if shared is not None else (None, None, None)
    st = lib.q4_gather_experts_k_noalloc(
        C.byref(gu), C.byref(dn), C.c_void_p(logits.data_ptr()), E, T, C.c_void_p(x.data_ptr()), k,
        C.c_void_p(idx.data_ptr()), C.c_void_p(w.data_ptr()), C.c_void_p(y.data_ptr()), dtype,
        C.byref(sgu) if sgu is not None else None, C.byref(sdn) if sdn is not None else None,
        C.c_void_p(sl.data_ptr()) if sl is not None else None,
        C.c_void_p(err.data_ptr()) if err is not None else None,
        C.c_void_p(torch.cuda.current_stream().cuda_stream))
    return st


# (k, output dtype, with the shared expert): two calls in a row per case
CASES = [(9, B.F32, True), (4, B.F32, True), (16, B.BF16, True), (3, B.F32_ADD, True), (7, B.F32, False),
         (1, B.F32_ADD, False)]


def test_noalloc_matches_regular_entry_point_on_two_calls():
    """Both entry points run the same kernels with the same fixed-order
    combine, so routes, weights and outputs agree bit for bit, call after
    call, with and without the shared expert and for every output type.  The
    caller's error word stays zero after every no-allocation call."""
    import torch

    assert torch.cuda.is_available()
    lib = B.load()
    vf = B.Verify(0)
    E, H, I, T = 24, 384, 640, 10
    gu = S.q4_matrix(50, "na.gu", 2 * I, H, n_experts=E)
    dn = S.q4_matrix(50, "na.dn", H, I, n_experts=E)
    sgu = S.q4_matrix(50, "na.sgu", 2 * I, H)
    sdn = S.q4_matrix(50, "na.sdn", H, I)
    GU, DN, SGU, SDN = (DevQ4(vf, gu, True), DevQ4(vf, dn, down=True), DevQ4(vf, sgu, True),
                        DevQ4(vf, sdn, down=True))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    for call, (k, dtype, with_shared) in enumerate(CASES):
        x = dev(S.bf16_normal(50, f"na.x{call}", (k, H)))
        logits = dev(S.f32_normal(50, f"na.l{call}", (k, E)))
        sl = dev(np.ascontiguousarray(np.pad(S.f32_normal(50, f"na.s{call}", (k, 1)), ((0, 0), (0, E - 1)))))
        y_init = S.f32_normal(50, f"na.y{call}", (k, H))  # the residual F32_ADD adds to
        outs = []
        for use_noalloc in (False, True):
            idx = torch.full((k, T), -1, dtype=torch.int32, device="cuda")
            w = torch.zeros((k, T), device="cuda")
            if dtype == B.BF16:
                y = torch.zeros((k, H), dtype=torch.int16, device="cuda")
            else:
                y = torch.from_numpy(y_init.copy()).cuda() if dtype == B.F32_ADD else torch.zeros((k, H), device="cuda")
            shared = (SGU.struct, SDN.struct, sl) if with_shared else None
            if use_noalloc:
                st = _noalloc(lib, GU.struct, DN.struct, logits, E, T, x, k, idx, w, y, shared=shared, err=err,
                              dtype=dtype)
                assert st == B.OK, f"case {call}: status {st}"
                torch.cuda.synchronize()
                assert int(err.item()) == 0, f"case {call}: device error reported"
            else:
                vf.q4_gather_experts_k(GU.struct, DN.struct, logits, E, T, x, k, idx, w, y, dtype,
                                       *(shared if with_shared else (None, None, None)))
                torch.cuda.synchronize()
            outs.append((host(idx), host(w), host(y)))
        (i0, w0, y0), (i1, w1, y1) = outs
        assert np.array_equal(i0, i1), f"case {call}: routing differs"
        assert np.array_equal(w0.view(np.uint32), w1.view(np.uint32)), f"case {call}: routing weights differ"
        assert np.array_equal(y0.view(np.uint32 if y0.dtype == np.float32 else np.uint16),
                              y1.view(np.uint32 if y1.dtype == np.float32 else np.uint16)), f"case {call}: y differs"
        if dtype == B.F32_ADD:
            assert not np.array_equal(y1, y_init)
    # the regular entry point's own error word (the no-allocation call never writes it)
    st, code = vf.device_status()
    assert st == B.OK, f"regular entry point: device error word {code}"
    vf.close()


def test_noalloc_rejects_sizes_beyond_its_scratch():
    import torch

    lib = B.load()
    E, H, I, T, k = 16, 8192, 256, 16, 16  # k*T*H*4 = 8 MiB of partials alone: too large
    # tiled operands of the right shapes (the call stops at the size check)
    gu = torch.zeros(int(lib.q4_tiled_bytes(2 * I, H, E, B.TILE_GATE_UP)), dtype=torch.uint8, device="cuda")
    dn = torch.zeros(int(lib.q4_tiled_bytes(H, I, E, B.TILE_DOWN)), dtype=torch.uint8, device="cuda")
    GU = B.Q4Experts(B.Q4Weight(gu.data_ptr(), None, None, 2 * I, H, 64, 4, B.TILED_GATE_UP), E)
    DN = B.Q4Experts(B.Q4Weight(dn.data_ptr(), None, None, H, I, 64, 4, B.TILED_DOWN), E)
    x = torch.zeros((k, H), dtype=torch.int16, device="cuda")
    logits = torch.zeros((k, E), device="cuda")
    idx = torch.zeros((k, E), dtype=torch.int32, device="cuda")
    w = torch.zeros((k, E), device="cuda")
    y = torch.zeros((k, H), device="cuda")
    st = _noalloc(lib, GU, DN, logits, E, T, x, k, idx, w, y)
    assert st == B.EUNSUPPORTED
    torch.cuda.synchronize()


@pytest.mark.parametrize("H, I, k", [(16384, 64, 1), (256, 96, 1), (256, 8192, 1), (256, 64, 17)])
def test_noalloc_applies_the_regular_shape_rules(H, I, k):
    """Shapes the regular entry point refuses (hidden above 8192, I not a
    multiple of 64, I above 4096, k above one pass) are refused with
    VERIFY_EUNSUPPORTED before anything runs, as the regular call does."""
    import torch

    lib = B.load()
    vf = B.Verify(0)
    E, T = 2, 1
    gu = torch.zeros(1 << 16, dtype=torch.uint8, device="cuda")
    dn = torch.zeros(1 << 16, dtype=torch.uint8, device="cuda")
    GU = B.Q4Experts(B.Q4Weight(gu.data_ptr(), None, None, 2 * I, H, 64, 4, B.TILED_GATE_UP), E)
    DN = B.Q4Experts(B.Q4Weight(dn.data_ptr(), None, None, H, I, 64, 4, B.TILED_DOWN), E)
    x = torch.zeros((k, H), dtype=torch.int16, device="cuda")
    logits = torch.zeros((k, E), device="cuda")
    idx = torch.zeros((k, T), dtype=torch.int32, device="cuda")
    w = torch.zeros((k, T), device="cuda")
    y = torch.zeros((k, H), device="cuda")
    assert _noalloc(lib, GU, DN, logits, E, T, x, k, idx, w, y) == B.EUNSUPPORTED
    if k <= B.PASS_K:  # (the regular call takes 17 rows as two passes)
        with pytest.raises(B.VerifyError) as ex:
            vf.q4_gather_experts_k(GU, DN, logits, E, T, x, k, idx, w, y, B.F32)
        assert ex.value.status == B.EUNSUPPORTED
    vf.close()
