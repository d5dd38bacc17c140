"""GPU parity of the k-row Gated DeltaNet step (gdn_verify_k) and the
accepted-prefix rollback (gdn_commit) against the CPU oracle.

Pages: "QWEN38FLASH.md - Plan for supporting Qwen/Qwen3.8-Flash-Next" 2.1
(per-token pipeline, delta rule, gated RMSNorm) and 3.1; "Red Lite dev45 -
speculative decoding with the Qwen3-Next MTP block", "What it is" (row r runs
from row r-1's state, in-kernel snapshots, rollback by pointer swap);
"Flash-Next optimization transfer to Ornith and Qwen 27B", section "Checkpoint
correctness" (every accepted-prefix GDN rollback at widths 4, 8, 9).
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


class Layer:
    """A GDN layer on the device: parameters, a ring of k_max+1 state slots."""

    def __init__(self, seed, Hk, Hv, d, n_slots=10, s_std=0.0, tail_std=0.0, gate_act=0):
        import torch

        self.Hk, self.Hv, self.d = Hk, Hv, d
        self.C = 2 * Hk * d + Hv * d
        self.p = S.gdn_params(seed, "gdn", Hk, Hv, d)
        self.S0, self.tail0 = S.gdn_initial_state(seed, "gdn", Hk, Hv, d, s_std=s_std, tail_std=tail_std)
        self.dp = {key: dev(v) for key, v in self.p.items()}
        self.params = B.gdn_params(Hk, Hv, d, self.dp["conv_w"], self.dp["A_log"], self.dp["dt_bias"],
                                   self.dp["norm_w"], gate_act=gate_act)
        self.gate_act = gate_act
        self.S_slots = [torch.zeros((Hv, d, d), dtype=torch.float32, device="cuda") for _ in range(n_slots)]
        self.conv_slots = [torch.zeros((3, self.C), dtype=torch.int16, device="cuda") for _ in range(n_slots)]
        self.reset()

    def reset(self, S=None, tail=None, cur=0):
        import torch

        S = self.S0 if S is None else S
        tail = self.tail0 if tail is None else tail
        self.S_slots[cur].copy_(torch.from_numpy(np.ascontiguousarray(S, np.float32)))
        self.conv_slots[cur].copy_(torch.from_numpy(np.ascontiguousarray(tail).view(np.int16)))
        self.state = B.gdn_state(self.S_slots, self.conv_slots, cur=cur)

    def verify(self, vf, inp, k, dtype=B.F32):
        import torch

        d_in = {key: dev(v) for key, v in inp.items()}
        o = torch.zeros((k, self.Hv * self.d), dtype=torch.float32 if dtype == B.F32 else torch.int16,
                        device="cuda")
        vf.gdn_verify_k(self.params, self.state,
                        B.gdn_inputs(d_in["qkv"], d_in["z"], d_in["a"], d_in["b"]), k, o, dtype)
        torch.cuda.synchronize()
        return host(o)

    def slot(self, s):
        return host(self.S_slots[s]), host(self.conv_slots[s], np.uint16)

    def oracle(self, inp, k, S0=None, tail0=None):
        return O.gdn_verify(self.Hk, self.Hv, self.d, self.p, self.S0 if S0 is None else S0,
                            self.tail0 if tail0 is None else tail0, inp, k, gate_act=self.gate_act)


@pytest.mark.parametrize("gate_act", [0, 1])
def test_tiny_step_matches_oracle(vf, gate_act):
    """2 QK heads, 2 V heads, d = 32, zero initial state, k = 2 (tiny workload)."""
    L = Layer(0, 2, 2, 32, gate_act=gate_act)
    inp = S.gdn_inputs(0, "tiny.gdn", 2, 2, 2, 32)
    o = L.verify(vf, inp, 2)
    oo, oS, ot = L.oracle(inp, 2)
    assert_close(o, oo, what="o")
    for r in range(2):
        S_r, t_r = L.slot(L.state.pending[r + 1])
        assert_close(S_r, oS[r], what=f"S after row {r}")
        assert np.array_equal(t_r, ot[r])


@pytest.mark.parametrize("k", [1, 4, 9, 16, 17, 32])
def test_flash_shape_matches_oracle(vf, k):
    """16/48 heads, d = 128, S0 ~ N(0, 0.02^2), conv tail ~ N(0,1).  k > 16
    runs as two launches, the second continuing from row 15's snapshot."""
    c = S.FLASH_GDN
    L = Layer(3, c["n_qk_heads"], c["n_v_heads"], c["d"], n_slots=33, s_std=0.02, tail_std=1.0)
    inp = S.gdn_inputs(3, f"flash.gdn.{k}", k, c["n_qk_heads"], c["n_v_heads"], c["d"])
    o = L.verify(vf, inp, k)
    oo, oS, ot = L.oracle(inp, k)
    assert_close(o, oo, what="o")
    for r in range(k):
        S_r, t_r = L.slot(L.state.pending[r + 1])
        assert_close(S_r, oS[r], what=f"S after row {r}")
        assert np.array_equal(t_r, ot[r])


@pytest.mark.parametrize("k", range(1, 10))
def test_flash_shape_every_width_with_random_rollback(vf, k):
    """Flash-Next shape at every width k = 1..9: output and every row's
    snapshot against the oracle, then a commit of a seeded random accepted
    prefix a in 0..k, whose state must be the oracle's state after a rows
    and, bit for bit, the state a fresh verify(a) leaves."""
    c = S.FLASH_GDN
    L = Layer(8, c["n_qk_heads"], c["n_v_heads"], c["d"], n_slots=10, s_std=0.02, tail_std=1.0)
    inp = S.gdn_inputs(8, f"wr.gdn.{k}", k, c["n_qk_heads"], c["n_v_heads"], c["d"])
    o = L.verify(vf, inp, k)
    oo, oS, ot = L.oracle(inp, k)
    assert_close(o, oo, what=f"o, k={k}")
    for r in range(k):
        S_r, t_r = L.slot(L.state.pending[r + 1])
        assert_close(S_r, oS[r], what=f"S after row {r}, k={k}")
        assert np.array_equal(t_r, ot[r])
    a = int(S.draws(S.tensor_seed(8, f"wr.accept.{k}"), 0, 1)[0] % np.uint64(k + 1))
    vf.gdn_commit(L.state, a)
    got = L.slot(L.state.cur)
    if a == 0:
        assert L.state.cur == 0
        assert np.array_equal(got[0], L.S0) and np.array_equal(got[1], L.tail0)
        return
    assert_close(got[0], oS[a - 1], what=f"committed state, k={k}, a={a}")
    assert np.array_equal(got[1], ot[a - 1])
    L.reset()
    L.verify(vf, {key: v[:a] for key, v in inp.items()}, a)
    want = L.slot(L.state.pending[a])
    assert np.array_equal(got[0].view(np.uint32), want[0].view(np.uint32)), f"k={k}, a={a}"
    assert np.array_equal(got[1], want[1])


@pytest.mark.parametrize("k", [9, 32])
def test_k_rows_bit_identical_to_sequential_single_rows(vf, k):
    """Row r of a k-row call equals a 1-row call started from the snapshot
    after r rows: outputs and states, bit for bit."""
    c = S.FLASH_GDN
    L = Layer(4, c["n_qk_heads"], c["n_v_heads"], c["d"], n_slots=k + 1, s_std=0.02, tail_std=1.0)
    inp = S.gdn_inputs(4, "seq.gdn", k, c["n_qk_heads"], c["n_v_heads"], c["d"])
    o = L.verify(vf, inp, k)
    snaps = [L.slot(L.state.pending[r + 1]) for r in range(k)]
    S_prev, t_prev = L.S0, L.tail0
    for r in range(k):
        L.reset(S_prev, t_prev)
        one = {key: v[r:r + 1] for key, v in inp.items()}
        o1 = L.verify(vf, one, 1)
        assert np.array_equal(o1[0].view(np.uint32), o[r].view(np.uint32)), f"o row {r}"
        S1, t1 = L.slot(L.state.pending[1])
        assert np.array_equal(S1.view(np.uint32), snaps[r][0].view(np.uint32)), f"S row {r}"
        assert np.array_equal(t1, snaps[r][1])
        S_prev, t_prev = S1, t1


@pytest.mark.parametrize("k", [4, 8, 9, 20])
def test_rollback_to_every_accepted_prefix(vf, k):
    """verify(k) + commit(a) leaves exactly the state of a fresh verify(a), for
    every a in 0..k; a = 0 keeps the pre-verify state."""
    c = S.FLASH_GDN
    L = Layer(5, c["n_qk_heads"], c["n_v_heads"], c["d"], n_slots=max(10, k + 1), s_std=0.02, tail_std=1.0)
    inp = S.gdn_inputs(5, f"rb.gdn.{k}", k, c["n_qk_heads"], c["n_v_heads"], c["d"])
    for a in range(k + 1):
        L.reset()
        L.verify(vf, inp, k)
        vf.gdn_commit(L.state, a)
        got = L.slot(L.state.cur)
        if a == 0:
            assert L.state.cur == 0
            assert np.array_equal(got[0], L.S0) and np.array_equal(got[1], L.tail0)
            continue
        L.reset()
        L.verify(vf, {key: v[:a] for key, v in inp.items()}, a)
        want = L.slot(L.state.pending[a])
        assert np.array_equal(got[0].view(np.uint32), want[0].view(np.uint32)), f"a={a}"
        assert np.array_equal(got[1], want[1])
    # the committed state continues: a second verify runs from it
    L.reset()
    L.verify(vf, inp, k)
    vf.gdn_commit(L.state, 2)
    with pytest.raises(B.VerifyError):
        vf.gdn_commit(L.state, 1)  # nothing pending any more
    inp2 = S.gdn_inputs(5, "rb.gdn.next", 3, c["n_qk_heads"], c["n_v_heads"], c["d"])
    o2 = L.verify(vf, inp2, 3)
    _, oS, ot = L.oracle(inp, 2)
    oo2, _, _ = L.oracle(inp2, 3, S0=oS[1], tail0=ot[1])
    assert_close(o2, oo2, what="continued verify")


def test_bf16_output_is_rne_of_f32(vf):
    L = Layer(6, 2, 4, 64, s_std=0.05)
    inp = S.gdn_inputs(6, "bf.gdn", 3, 2, 4, 64)
    o32 = L.verify(vf, inp, 3)
    L.reset()
    o16 = L.verify(vf, inp, 3, dtype=B.BF16).view(np.uint16)
    assert np.array_equal(o16, S.f32_to_bf16(o32))


def test_slot_errors(vf):
    L = Layer(7, 2, 2, 32, n_slots=3)
    inp = S.gdn_inputs(7, "err.gdn", 3, 2, 2, 32)
    with pytest.raises(B.VerifyError) as e:
        L.verify(vf, inp, 3)  # needs 4 slots
    assert e.value.status == B.EINVAL
    L.verify(vf, {key: v[:2] for key, v in inp.items()}, 2)
    with pytest.raises(B.VerifyError):
        vf.gdn_commit(L.state, 3)
    vf.gdn_commit(L.state, 2)
    assert L.state.cur == L.state.pending[2]
