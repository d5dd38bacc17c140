"""GPU parity of the width-k attention verify (attn_verify_k) and the cache
rollback (attn_commit) against the CPU oracle.

Pages: "QWEN38FLASH.md - Plan for supporting Qwen/Qwen3.8-Flash-Next" 2.2
(24 query / 2 KV heads of dim 256, partial RoPE, sigmoid output gate, F16
cache); "Red Lite dev45 - speculative decoding with the Qwen3-Next MTP block",
"What it is" (attention runs per row; rejected rows are overwritten later);
"Flash-Next optimization transfer to Ornith and Qwen 27B", "Exact
verification kernels" (each row's serial KV window, caches through 65,536
tokens).
"""
import numpy as np
import pytest

from oracle import oracle as O
from speculative_decode_verification_gb300 import binding as B
from speculative_decode_verification_gb300 import synth as S
from tests.gpu_util import assert_close, dev, host

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


class Cache:
    """A KV cache on the device, its workspace, and the host copy it started from."""

    def __init__(self, seed, name, Hq, Hkv, D, cap, P, split=256, max_k=16, rope_dim=64, theta=1e7):
        import torch

        self.Hq, self.Hkv, self.D, self.rope_dim, self.theta = Hq, Hkv, D, rope_dim, theta
        self.K0, self.V0 = S.attn_cache(seed, name, Hkv, cap, D, P)
        self.K = dev(self.K0)
        self.V = dev(self.V0)
        self.params = B.attn_params(Hq, Hkv, D, rope_dim, theta)
        nb = B.attn_workspace_bytes(self.params, cap, split, max_k)
        assert nb > 0
        self.work = torch.empty(nb, dtype=torch.uint8, device="cuda")
        self.c = B.kv_cache(self.K, self.V, self.work, P, split)

    def verify(self, vf, inp, k, dtype=B.F32):
        import torch

        d = {key: dev(v.reshape(v.shape[0], -1)) for key, v in inp.items()}
        o = torch.zeros((k, self.Hq * self.D), dtype=torch.float32 if dtype == B.F32 else torch.int16,
                        device="cuda")
        vf.attn_verify_k(self.params, self.c, B.attn_inputs(d["q"], d["gate"], d["k"], d["v"]), k, o, dtype)
        torch.cuda.synchronize()
        return host(o)

    def oracle(self, inp, P, K=None, V=None):
        return O.attn_verify(self.Hq, self.Hkv, self.D, P, inp["q"], inp["k"], inp["v"], inp["gate"],
                             self.K0 if K is None else K, self.V0 if V is None else V, self.rope_dim, self.theta)


def _f16(bits):
    return np.asarray(bits, np.uint16).view(np.float16).astype(np.float64)


def _check_appended(cache, P, k, k_app, v_app):
    Kd = host(cache.K, np.uint16)
    Vd = host(cache.V, np.uint16)
    for r in range(k):
        assert np.array_equal(Vd[:, P + r], v_app[r]), f"V row {r}"
        # keys: rotation angles in float64 on both sides, so at most one
        # binary16 ulp apart where libm and CUDA differ in the last bit
        a, b = _f16(Kd[:, P + r]), _f16(k_app[r])
        ulp = np.spacing(np.abs(b).astype(np.float16)).astype(np.float64)
        assert np.all(np.abs(a - b) <= ulp), f"K row {r}"


CASES = [
    # Hq, Hkv, D, P, k, split
    (4, 2, 128, 0, 1, 32),
    (4, 2, 128, 5, 4, 32),
    (8, 2, 128, 300, 9, 64),
    (24, 2, 256, 0, 16, 256),
    (24, 2, 256, 37, 9, 256),
    (24, 2, 256, 1000, 4, 256),
    (24, 2, 256, 2047, 16, 512),
    (6, 1, 256, 700, 9, 32),
    (24, 2, 256, 500, 32, 256),
]


@pytest.mark.parametrize("case", CASES, ids=[f"H{c[0]}_{c[1]}_D{c[2]}_P{c[3]}_k{c[4]}_s{c[5]}" for c in CASES])
def test_attn_matches_oracle(vf, case):
    Hq, Hkv, D, P, k, split = case
    cache = Cache(20, f"attn.{Hq}.{D}.{P}", Hq, Hkv, D, P + k + 3, P, split, max_k=max(16, k))
    inp = S.attn_inputs(20, f"attn.in.{Hq}.{P}.{k}", k, Hq, Hkv, D)
    o = cache.verify(vf, inp, k)
    oo, k_app, v_app = cache.oracle(inp, P)
    assert_close(o, oo.reshape(k, -1), what="o")
    _check_appended(cache, P, k, k_app, v_app)
    assert cache.c.pending_k == k and cache.c.len == P


# The split kernel's pipeline edges: the ten-slot ring of head dim 128
# wrapping many times, splits that are not a multiple of its 64-position
# sub-tile, a cache filled exactly to capacity (the tile loads' zero fill
# starts at P + k) and one KV head holding 16 rows x 12 query heads (two
# 128-pair tiles).
PIPE_CASES = [
    # Hq, Hkv, D, P, k, split, capacity - (P + k)
    (8, 2, 128, 4000, 9, 2048, 0),
    (8, 2, 128, 1000, 9, 96, 0),
    (24, 2, 256, 3000, 4, 1024, 0),
    (12, 1, 256, 777, 16, 160, 5),
]


@pytest.mark.parametrize("case", PIPE_CASES, ids=[f"H{c[0]}_{c[1]}_D{c[2]}_P{c[3]}_k{c[4]}_s{c[5]}_x{c[6]}" for c in PIPE_CASES])
def test_pipeline_shapes(vf, case):
    Hq, Hkv, D, P, k, split, extra = case
    cache = Cache(27, f"pipe.{D}.{P}.{split}", Hq, Hkv, D, P + k + extra, P, split, max_k=max(16, k))
    inp = S.attn_inputs(27, f"pipe.in.{D}.{P}.{k}", k, Hq, Hkv, D)
    o = cache.verify(vf, inp, k)
    oo, k_app, v_app = cache.oracle(inp, P)
    assert_close(o, oo.reshape(k, -1), what="o")
    _check_appended(cache, P, k, k_app, v_app)


def test_growing_scores_raise_the_running_max(vf):
    """Keys scaled up with their position (x (1 + pos/16)), so that nearly
    every 64-position sub-tile raises each row's running maximum by far more
    than 2^8: the rescale of the output tile and the sum, against the
    oracle."""
    Hq, Hkv, D, P, k = 24, 2, 256, 2000, 9
    cache = Cache(28, "grow", Hq, Hkv, D, P + k, P, 512)
    K1 = cache.K0.view(np.float16).astype(np.float32)
    K1[:, :P] *= (1.0 + np.arange(P, dtype=np.float32) / 16.0)[None, :, None]
    cache.K0 = K1.astype(np.float16).view(np.uint16)
    cache.K.copy_(dev(cache.K0))
    inp = S.attn_inputs(28, "grow.in", k, Hq, Hkv, D)
    o = cache.verify(vf, inp, k)
    oo, _, _ = cache.oracle(inp, P)
    assert_close(o, oo.reshape(k, -1), what="o")


def test_stale_workspace_does_not_leak(vf):
    """The query rows past k * Hq / Hkv of the workspace are never cleared:
    a workspace filled with NaN bits, then a width-16 call, then a width-3
    call over the same cache, each against the oracle."""
    import torch

    Hq, Hkv, D, P = 24, 2, 256, 600
    cache = Cache(29, "stale", Hq, Hkv, D, P + 16, P, 256)
    cache.work.fill_(0xFF)
    for k in (16, 3):
        inp = S.attn_inputs(29, f"stale.in.{k}", k, Hq, Hkv, D)
        o = cache.verify(vf, inp, k)
        oo, _, _ = cache.oracle(inp, P)
        assert np.all(np.isfinite(o)), f"k={k}"
        assert_close(o, oo.reshape(k, -1), what=f"o k={k}")
    torch.cuda.synchronize()


def test_bf16_output_is_rne_of_f32(vf):
    Hq, Hkv, D, P, k = 24, 2, 256, 100, 5
    cache = Cache(21, "attn.bf", Hq, Hkv, D, P + k, P)
    inp = S.attn_inputs(21, "attn.bf.in", k, Hq, Hkv, D)
    o32 = cache.verify(vf, inp, k)
    o16 = cache.verify(vf, inp, k, B.BF16).view(np.uint16)
    assert np.array_equal(o16, S.f32_to_bf16(o32))


@pytest.mark.parametrize("P,split", [(0, 32), (61, 32), (1000, 256), (4090, 256)])
def test_rows_bit_identical_to_single_row_calls(vf, P, split):
    """Row r of a width-9 call equals a width-1 call at P + r after the first
    r rows were committed one by one: outputs and cached rows, bit for bit."""
    Hq, Hkv, D, k = 24, 2, 256, 9
    a = Cache(22, f"seq.{P}", Hq, Hkv, D, P + k + 1, P, split)
    b = Cache(22, f"seq.{P}", Hq, Hkv, D, P + k + 1, P, split)
    inp = S.attn_inputs(22, f"seq.in.{P}", k, Hq, Hkv, D)
    o = a.verify(vf, inp, k)
    for r in range(k):
        o1 = b.verify(vf, {key: v[r:r + 1] for key, v in inp.items()}, 1)
        assert np.array_equal(o1[0].view(np.uint32), o[r].view(np.uint32)), f"row {r}"
        vf.attn_commit(b.c, 1)
    Ka, Kb = host(a.K, np.uint16), host(b.K, np.uint16)
    Va, Vb = host(a.V, np.uint16), host(b.V, np.uint16)
    assert np.array_equal(Ka[:, : P + k], Kb[:, : P + k]) and np.array_equal(Va[:, : P + k], Vb[:, : P + k])


def test_commit_then_continue(vf):
    """verify(k), commit(a): the next verify starts at P + a, overwriting the
    rejected rows, and matches the oracle on the cache holding only the a
    accepted rows."""
    Hq, Hkv, D, P, k, a = 24, 2, 256, 500, 8, 3
    cache = Cache(23, "cont", Hq, Hkv, D, P + 2 * k, P)
    inp = S.attn_inputs(23, "cont.in1", k, Hq, Hkv, D)
    cache.verify(vf, inp, k)
    _, k_app, v_app = cache.oracle(inp, P)
    vf.attn_commit(cache.c, a)
    assert cache.c.len == P + a and cache.c.pending_k == 0
    with pytest.raises(B.VerifyError):
        vf.attn_commit(cache.c, 1)
    K1, V1 = cache.K0.copy(), cache.V0.copy()
    K1[:, P:P + a] = np.transpose(k_app[:a], (1, 0, 2))
    V1[:, P:P + a] = np.transpose(v_app[:a], (1, 0, 2))
    inp2 = S.attn_inputs(23, "cont.in2", 5, Hq, Hkv, D)
    o2 = cache.verify(vf, inp2, 5)
    oo2, _, _ = cache.oracle(inp2, P + a, K1, V1)
    assert_close(o2, oo2.reshape(5, -1), what="continued verify")


@pytest.mark.parametrize("k,P", [(4, 65536), (9, 16384)])
def test_flash_next_shape_long_cache(vf, k, P):
    """The Flash-Next attention shape over long caches (65,536 positions is the
    longest window the pages' fixtures exercise), every output against the
    oracle."""
    c = S.FLASH_ATTN
    cache = Cache(24, "long", c["n_q_heads"], c["n_kv_heads"], c["d"], P + k, P, split=256,
                  rope_dim=c["rope_dim"], theta=c["theta"])
    inp = S.attn_inputs(24, f"long.in{k}", k, c["n_q_heads"], c["n_kv_heads"], c["d"])
    o = cache.verify(vf, inp, k)
    oo, k_app, v_app = cache.oracle(inp, P)
    assert_close(o, oo.reshape(k, -1), what="o")
    _check_appended(cache, P, k, k_app, v_app)


def test_argument_errors(vf):
    import torch

    cache = Cache(25, "err", 24, 2, 256, 40, 30)
    inp = S.attn_inputs(25, "err.in", 16, 24, 2, 256)
    with pytest.raises(B.VerifyError) as e:
        cache.verify(vf, inp, 16)  # 30 + 16 > 40
    assert e.value.status == B.EINVAL
    small = B.attn_params(24, 2, 256)
    c2 = B.kv_cache(cache.K, cache.V, torch.empty(64, dtype=torch.uint8, device="cuda"), 0, 256)
    d = {key: dev(v[:1].reshape(1, -1)) for key, v in inp.items()}
    o = torch.zeros((1, 24 * 256), device="cuda")
    with pytest.raises(B.VerifyError):
        vf.attn_verify_k(small, c2, B.attn_inputs(d["q"], d["gate"], d["k"], d["v"]), 1, o)  # workspace too small


@pytest.mark.parametrize("rope_dim,theta", [(0, 1e7), (128, 1e4), (32, 5e5)])
def test_rope_dim_variants(vf, rope_dim, theta):
    """No rotation, full rotation (rope_dim = head_dim) and a narrow band,
    at another base: outputs and appended keys against the oracle."""
    Hq, Hkv, D, P, k = 8, 2, 128, 300, 9
    cache = Cache(26, f"rd.{rope_dim}", Hq, Hkv, D, P + k, P, 64, rope_dim=rope_dim, theta=theta)
    inp = S.attn_inputs(26, f"rd.in.{rope_dim}", k, Hq, Hkv, D)
    o = cache.verify(vf, inp, k)
    oo, k_app, v_app = cache.oracle(inp, P)
    assert_close(o, oo.reshape(k, -1), what=f"rope_dim={rope_dim}")
    _check_appended(cache, P, k, k_app, v_app)
