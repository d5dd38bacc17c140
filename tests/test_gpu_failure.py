"""Failure detection without a GPU fault: every wait in the verify kernels is
bounded.  A probe kernel runs the same two waits - a pipeline barrier that
nothing arrives on, a counter that nothing increments - until they give up;
the host then reads the timeout from the device error word, and the context
goes on computing correctly."""
import time

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
    v.close()


def test_stuck_waits_time_out_and_the_context_stays_usable(vf):
    import torch

    assert vf.device_status() == (B.OK, 0)
    before = vf.launch_count()
    t0 = time.perf_counter()
    vf.selftest_stuck_wait()
    st, code = vf.device_status()  # synchronises: the probe has given up and returned
    elapsed = time.perf_counter() - t0
    assert vf.launch_count() - before == 1
    assert st == B.EDEVICE and code == 1, (st, code)  # 1: a pipeline wait timed out
    assert elapsed < 30.0
    assert vf.device_status() == (B.OK, 0)  # read once, then cleared
    # the same context computes as before
    m = S.q4_matrix(11, "fail.q4", 256, 512)
    W = DevQ4(vf, m)
    x = S.bf16_normal(11, "fail.x", (3, 512))
    y = torch.zeros((3, 256), dtype=torch.float32, device="cuda")
    vf.q4_qmv_k(W.struct, dev(x), 3, y, B.F32)
    torch.cuda.synchronize()
    assert_close(host(y), O.q4_qmv(m.packed, m.scales, m.biases, x), what="after the probe")
    assert vf.device_status() == (B.OK, 0)
