"""One small width-k verify through every entry point on cuda:0, checked
against the CPU oracle (used by __graft_entry__.smoke)."""
import numpy as np

from oracle import oracle as O
from speculative_decode_verification_gb300 import binding as B
from speculative_decode_verification_gb300 import synth as S
from tests.gpu_util import DevQ4, assert_close, dev, host


def run():
    import torch

    assert torch.cuda.is_available(), "smoke needs cuda:0"
    torch.cuda.set_device(0)
    vf = B.Verify(0)
    k = 4
    # dense Q4 product (tiny workload)
    m = S.q4_matrix(0, "tiny.q4", 512, 512)
    x = S.bf16_normal(0, "smoke.x", (k, 512))
    y = torch.zeros((k, 512), device="cuda")
    W = DevQ4(vf, m)  # keeps the device tensors alive while the struct points at them
    xd = dev(x)
    vf.q4_qmv_k(W.struct, xd, k, y)
    torch.cuda.synchronize()
    assert_close(host(y), O.q4_qmv(m.packed, m.scales, m.biases, x), what="q4_qmv_k")
    # routed experts
    E, H, I, T = 16, 256, 256, 4
    gu = S.q4_matrix(0, "smoke.gu", 2 * I, H, n_experts=E)
    dn = S.q4_matrix(0, "smoke.dn", H, I, n_experts=E)
    xm = S.bf16_normal(0, "smoke.xm", (k, H))
    lg = S.f32_normal(0, "smoke.lg", (k, E))
    idx = torch.zeros((k, T), dtype=torch.int32, device="cuda")
    w = torch.zeros((k, T), device="cuda")
    ym = torch.zeros((k, H), device="cuda")
    GU, DN = DevQ4(vf, gu, True), DevQ4(vf, dn, down=True)
    lgd, xmd = dev(lg), dev(xm)
    vf.q4_gather_experts_k(GU.struct, DN.struct, lgd, E, T, xmd, k, idx, w, ym)
    torch.cuda.synchronize()
    oi, _, oy, _ = O.gather_experts((gu.packed, gu.scales, gu.biases), (dn.packed, dn.scales, dn.biases), lg, T, xm)
    assert np.array_equal(host(idx), oi)
    assert_close(host(ym), oy, what="q4_gather_experts_k")
    # Gated DeltaNet verify + commit (tiny workload)
    Hk = Hv = 2
    d = 32
    C = 2 * Hk * d + Hv * d
    p = S.gdn_params(0, "gdn", Hk, Hv, d)
    dp = {key: dev(v) for key, v in p.items()}
    S0, t0 = S.gdn_initial_state(0, "gdn", Hk, Hv, d)
    slots = [torch.zeros((Hv, d, d), device="cuda") for _ in range(k + 1)]
    tails = [torch.zeros((3, C), dtype=torch.int16, device="cuda") for _ in range(k + 1)]
    st = B.gdn_state(slots, tails)
    inp = S.gdn_inputs(0, "smoke.gdn", k, Hk, Hv, d)
    di = {key: dev(v) for key, v in inp.items()}  # kept alive until the synchronize below
    o = torch.zeros((k, Hv * d), device="cuda")
    vf.gdn_verify_k(B.gdn_params(Hk, Hv, d, dp["conv_w"], dp["A_log"], dp["dt_bias"], dp["norm_w"]), st,
                    B.gdn_inputs(di["qkv"], di["z"], di["a"], di["b"]), k, o)
    vf.gdn_commit(st, 2)
    torch.cuda.synchronize()
    oo, oS, ot = O.gdn_verify(Hk, Hv, d, p, S0.astype(np.float64), t0, inp, k)
    assert_close(host(o), oo, what="gdn_verify_k")
    assert_close(host(slots[st.cur]), oS[1], what="gdn_commit state")
    # greedy acceptance on the device, fused with a device-held commit
    arr = (B.GdnState * 1)()
    arr[0] = st
    words = torch.zeros((1, 2), dtype=torch.int32, device="cuda")
    vf.gdn_state_to_device(arr, words)
    vf.gdn_verify_k(B.gdn_params(Hk, Hv, d, dp["conv_w"], dp["A_log"], dp["dt_bias"], dp["norm_w"]), arr[0],
                    B.gdn_inputs(di["qkv"], di["z"], di["a"], di["b"]), k, o)
    V = 3000
    lx = S.vocab_logits(0, "smoke.logits", k, V, 4)
    _, _, t = O.accept_greedy(lx, np.zeros(k - 1, np.int32))
    draft = t[: k - 1].copy()
    draft[2] = (t[2] + 1) % V  # two drafts stand
    a, nxt, _ = O.accept_greedy(lx, draft)
    res = torch.zeros(2 + k, dtype=torch.int32, device="cuda")
    lxd, drd = dev(lx), dev(draft)
    vf.accept_greedy(lxd, k, drd, res, states=arr)
    torch.cuda.synchronize()
    assert host(res).tolist() == [a, nxt] + t.tolist(), "verify_accept_greedy"
    c = st.cur  # the slot the device verify started from
    assert a == 3 and host(words).tolist() == [[2 + (2 >= c), 0]], "device commit"
    _, oS2, _ = O.gdn_verify(Hk, Hv, d, p, oS[1], ot[1], inp, k)
    assert_close(host(slots[2 + (2 >= c)]), oS2[2], what="device-committed state")
    # width-k attention over a small binary16 cache
    Hq, Hkv, D, P = 4, 2, 128, 37
    Kc, Vc = S.attn_cache(0, "smoke.attn", Hkv, P + k, D, P)
    ai = S.attn_inputs(0, "smoke.attn.in", k, Hq, Hkv, D)
    Kd, Vd = dev(Kc), dev(Vc)
    ap = B.attn_params(Hq, Hkv, D)
    work = torch.empty(B.attn_workspace_bytes(ap, P + k, 32, k), dtype=torch.uint8, device="cuda")
    kc = B.kv_cache(Kd, Vd, work, P, 32)
    aid = {key: dev(v.reshape(k, -1)) for key, v in ai.items()}
    ao = torch.zeros((k, Hq * D), device="cuda")
    vf.attn_verify_k(ap, kc, B.attn_inputs(aid["q"], aid["gate"], aid["k"], aid["v"]), k, ao)
    torch.cuda.synchronize()
    oo_attn, _, _ = O.attn_verify(Hq, Hkv, D, P, ai["q"], ai["k"], ai["v"], ai["gate"], Kc, Vc)
    assert_close(host(ao), oo_attn.reshape(k, -1), what="attn_verify_k")
    status, code = vf.device_status()
    assert status == B.OK, f"device error word {code}"
    vf.close()
    print("smoke OK")
