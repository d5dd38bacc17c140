"""GPU parity of a full hybrid verify layer stack (verify_layer_k: GDN mixer
then routed + shared MoE, 8 kernels per layer) against the oracle's
composition of its pinned pieces.

Pages: "QWEN38FLASH.md - Plan for supporting Qwen/Qwen3.8-Flash-Next" section 2
(layer = Gated DeltaNet -> MoE, 512 experts, 10 routed + 1 shared, hidden 2560)
and "Red Lite dev45 - speculative decoding with the Qwen3-Next MTP block",
"Acceptance" (the verified rows equal what ordinary one-row steps give).
"""
import numpy as np
import pytest

from oracle import oracle as O
from speculative_decode_verification_gb300 import binding as B
from speculative_decode_verification_gb300 import synth as S
from speculative_decode_verification_gb300.stack import DeviceStack, shapes
from tests.gpu_util import assert_close, host

pytestmark = pytest.mark.gpu

SMALL = dict(layers=2, H=256, E=16, T=4, I=256, n_qk_heads=2, n_v_heads=4, d=64, conv_kernel=4)


@pytest.fixture(scope="module")
def vf():
    import torch

    assert torch.cuda.is_available()
    v = B.Verify(0)
    yield v
    st, code = v.device_status()
    assert st == B.OK, f"device error word {code}"
    v.close()


def oracle_stack(cfg, seed, h0, k, layers):
    sh = shapes(cfg)
    h = h0.astype(np.float64)
    snaps = []
    for l in range(layers):
        w = S.HostLayerWeights(seed, l, sh["H"], sh["NP"], sh["Z"], sh["E"], sh["I"], cfg["n_qk_heads"],
                               cfg["n_v_heads"], cfg["d"])
        S0, t0 = S.gdn_initial_state(seed, f"stack.L{l}.gdn", cfg["n_qk_heads"], cfg["n_v_heads"], cfg["d"],
                                     s_std=0.02, tail_std=1.0)
        h, Ss, ts, idx, lg = O.stack_layer(w, h, S0.astype(np.float64), t0, k, cfg["n_qk_heads"],
                                           cfg["n_v_heads"], cfg["d"], sh["T"])
        snaps.append((Ss, ts, idx, lg))
    return h, snaps


@pytest.mark.parametrize("k", [1, 4, 9])
def test_small_stack_matches_oracle(vf, k):
    import torch

    ds = DeviceStack(vf, SMALL, seed=1)
    h0 = S.f32_normal(1, f"stack.h{k}", (k, SMALL["H"]))
    h = torch.from_numpy(h0.copy()).cuda()
    idx = [torch.zeros((k, SMALL["T"]), dtype=torch.int32, device="cuda") for _ in range(ds.n_layers)]
    ds.verify(h, k, idx)
    torch.cuda.synchronize()
    ref, snaps = oracle_stack(SMALL, 1, h0, k, ds.n_layers)
    for l in range(ds.n_layers):
        assert np.array_equal(host(idx[l]), snaps[l][2]), f"routing of layer {l}"
        st = ds.states[l]
        S_last = host(ds.state_tensors[l][0][st.pending[k]])
        assert_close(S_last, snaps[l][0][k - 1], what=f"GDN state layer {l}")
    assert_close(host(h), ref, what="residual stream")


def test_stack_rows_equal_single_row_steps(vf):
    """Row r of a k-row verify through the whole stack is bit-identical to a
    1-row verify started from the states after r rows (every layer)."""
    import torch

    k = 9
    ds = DeviceStack(vf, SMALL, seed=2)
    h0 = S.f32_normal(2, "stack.rows", (k, SMALL["H"]))
    h = torch.from_numpy(h0.copy()).cuda()
    ds.verify(h, k)
    torch.cuda.synchronize()
    hk = host(h)
    saved = []
    for l in range(ds.n_layers):
        st = ds.states[l]
        slots, tails = ds.state_tensors[l]
        saved.append([(slots[st.pending[r]].clone(), tails[st.pending[r]].clone()) for r in range(k)])
    for r in range(k):
        for l in range(ds.n_layers):
            slots, tails = ds.state_tensors[l]
            slots[0].copy_(saved[l][r][0])
            tails[0].copy_(saved[l][r][1])
            ds.states[l].cur = 0
            ds.states[l].pending_k = 0
        h1 = torch.from_numpy(h0[r:r + 1].copy()).cuda()
        ds.verify(h1, 1)
        torch.cuda.synchronize()
        assert np.array_equal(host(h1)[0].view(np.uint32), hk[r].view(np.uint32)), f"row {r}"


def test_flash_next_shape_two_layers_match_oracle(vf):
    """Hidden 2560, GDN 16/48/128, 512 experts top-10 + shared, I = 640, k = 9
    (two of the stack's twelve layers)."""
    import torch

    cfg = dict(S.STACK)
    k = 9
    ds = DeviceStack(vf, cfg, seed=0, layers=2)
    h0 = S.f32_normal(0, "stack.full.h", (k, cfg["H"]))
    h = torch.from_numpy(h0.copy()).cuda()
    idx = [torch.zeros((k, cfg["T"]), dtype=torch.int32, device="cuda") for _ in range(2)]
    ds.verify(h, k, idx)
    torch.cuda.synchronize()
    ref, snaps = oracle_stack(cfg, 0, h0, k, 2)
    for l in range(2):
        lg = snaps[l][3][:, :cfg["E"]].astype(np.float64)
        srt = -np.sort(-lg, axis=1)
        margin = np.min(srt[:, cfg["T"] - 1] - srt[:, cfg["T"]])
        assert margin > 1e-3 * np.std(lg), "top-k boundary too close for an fp32/fp64 comparison"
        assert np.array_equal(host(idx[l]), snaps[l][2]), f"routing of layer {l}"
    assert_close(host(h), ref, what="residual stream")
