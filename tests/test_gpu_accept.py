"""GPU parity of greedy acceptance on the device (verify_accept_greedy) and of
the device-held commit (gdn_commit_dev, the commit fused into acceptance).

Pages: "Red Lite dev45 - speculative decoding with the Qwen3-Next MTP block",
sections "What it is" (the pending token and the drafts are the rows of one
pass; a rejected draft is undone by swapping the DeltaNet state pointers with
the snapshots) and "Acceptance" (a draft stands when the token chosen from the
previous row's logits equals it).  The greedy choices, the accepted count and
the next token are integers: they must equal the oracle's exactly.
"""
import numpy as np
import pytest

from oracle import oracle as O
from speculative_decode_verification_gb300 import binding as B
from speculative_decode_verification_gb300 import synth as S
from tests.gpu_util import dev, host
from tests.test_gpu_gdn import Layer

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


def _drafts(t, m, V, rng):
    """Drafts d_1..d_{k-1}: the first m equal the greedy choices t_0..t_{m-1},
    d_{m+1} differs from t_m, the rest are arbitrary tokens."""
    k = len(t)
    d = rng.integers(0, V, max(k - 1, 0)).astype(np.int32)
    d[:m] = t[:m]
    if m < k - 1:
        d[m] = (t[m] + 1) % V if V > 1 else V  # V itself is outside the vocabulary
    return d


def _gpu_logits(x, ld_extra=0, offset=0):
    """x fp32 [k, V] on the device with row stride V + ld_extra, starting
    `offset` floats into its buffer (offset 1: rows not 16-byte aligned)."""
    import torch

    k, V = x.shape
    ld = V + ld_extra
    buf = torch.full((offset + k * ld,), float("nan"), dtype=torch.float32, device="cuda")
    view = buf[offset:].view(k, ld)
    view[:, :V].copy_(torch.from_numpy(np.ascontiguousarray(x)))
    return buf, view[:, :V]


def _accept(vf, x, draft, ld_extra=0, offset=0, states=None):
    import torch

    k = x.shape[0]
    _, lg = _gpu_logits(x, ld_extra, offset)
    d = dev(np.asarray(draft, np.int32)) if k > 1 else None
    res = torch.full((2 + k,), -7, dtype=torch.int32, device="cuda")
    vf.accept_greedy(lg, k, d, res, states=states)
    torch.cuda.synchronize()
    return host(res)


CASES = [
    # k, V, levels (ties), ld_extra, offset
    (1, 1, 0, 0, 0),
    (2, 3, 0, 0, 0),
    (9, 1000, 4, 0, 0),
    (3, 1023, 0, 5, 0),
    (4, 4099, 2, 1, 0),     # odd row stride: scalar loads
    (16, 5000, 8, 0, 1),    # rows not 16-byte aligned
    (1, S.FLASH_VOCAB, 0, 0, 0),
    (9, S.FLASH_VOCAB, 0, 0, 0),
    (16, S.FLASH_VOCAB, 16, 0, 0),
    (32, S.FLASH_VOCAB, 4, 0, 0),
    (32, 777, 0, 3, 1),
]


@pytest.mark.parametrize("case", CASES, ids=[f"k{c[0]}_V{c[1]}_lv{c[2]}_ld{c[3]}_off{c[4]}" for c in CASES])
def test_accept_matches_oracle(vf, case):
    k, V, levels, ld_extra, offset = case
    x = S.vocab_logits(11, f"accept.{k}.{V}.{levels}", k, V, levels)
    _, _, t = O.accept_greedy(x, np.zeros(k - 1, np.int32))
    rng = np.random.default_rng(k * 7919 + V)
    for m in sorted({0, k // 2, k - 1}):
        draft = _drafts(t, m, V, rng)
        a, nxt, t_o = O.accept_greedy(x, draft)
        assert a == m + 1
        got = _accept(vf, x, draft, ld_extra, offset)
        want = np.concatenate([[a, nxt], t_o]).astype(np.int32)
        assert np.array_equal(got, want), f"m={m}: gpu {got.tolist()} oracle {want.tolist()}"


def test_ties_signed_zeros_infinities_nans(vf):
    """Rows built around the tie readings: equal maxima (lowest index wins),
    -0 == +0, +inf, NaN above everything (the first NaN wins)."""
    V = 3001
    rows = []
    r = np.full(V, -5.0, np.float32); r[[17, 900, 2999]] = 2.5; rows.append(r)
    r = np.full(V, -1.0, np.float32); r[[5, 6]] = [-0.0, 0.0]; r[1000:] = -0.0; rows.append(r)
    r = np.zeros(V, np.float32); r[[40, 2000]] = np.inf; rows.append(r)
    r = np.zeros(V, np.float32); r[[2500, 1200]] = np.nan; r[3] = np.inf; rows.append(r)
    r = np.full(V, -np.inf, np.float32); rows.append(r)
    r = np.full(V, -np.inf, np.float32); r[V - 1] = -3e38; rows.append(r)
    x = np.stack(rows)
    k = x.shape[0]
    _, _, t = O.accept_greedy(x, np.zeros(k - 1, np.int32))
    assert t.tolist() == [int(np.argmax(row)) for row in x]
    for m in range(k):
        draft = _drafts(t, m, V, np.random.default_rng(m))
        a, nxt, t_o = O.accept_greedy(x, draft)
        got = _accept(vf, x, draft)
        assert np.array_equal(got, np.concatenate([[a, nxt], t_o]).astype(np.int32)), f"m={m}"


def test_repeated_calls_leave_no_state(vf):
    """The scratch is reset by every call: alternating inputs give the same
    results as fresh calls."""
    xs = [S.vocab_logits(12, f"rep.{i}", 5, 20000, 0) for i in range(3)]
    ts = [O.accept_greedy(x, np.zeros(4, np.int32))[2] for x in xs]
    for rep in range(2):
        for x, t in zip(xs, ts):
            got = _accept(vf, x, t[:4])
            assert got[0] == 5 and got[1] == t[4] and np.array_equal(got[2:], t)


def test_k_out_of_range_rejected(vf):
    import torch

    lg = torch.zeros((33, 8), dtype=torch.float32, device="cuda")
    res = torch.zeros(35, dtype=torch.int32, device="cuda")
    d = torch.zeros(32, dtype=torch.int32, device="cuda")
    with pytest.raises(B.VerifyError) as e:
        vf.accept_greedy(lg, 33, d, res)
    assert e.value.status == B.EUNSUPPORTED


# ------------------------------------------------------- device-held commit

def _device_layer(seed, Hk, Hv, d, n_slots=17):
    """A GDN layer whose committed slot lives on the device, and its dev words."""
    import torch

    L = Layer(seed, Hk, Hv, d, n_slots=n_slots, s_std=0.02, tail_std=1.0)
    arr = (B.GdnState * 1)()
    arr[0] = L.state
    L.state = arr[0]  # a view: the library's changes show through
    words = torch.full((1, 2), -1, dtype=torch.int32, device="cuda")
    return L, arr, words


def _dev_cur(words):
    return int(host(words)[0, 0])


@pytest.mark.parametrize("shape,k", [((2, 4, 64), 1), ((2, 4, 64), 4), ((2, 4, 64), 16), ((2, 4, 64), 32),
                                     ((16, 48, 128), 9)])
def test_device_commit_equals_host_commit(vf, shape, k):
    """The same verify + commit sequence, once with host-held and once with
    device-held commits: outputs, committed slots and their contents agree
    bit for bit after every step (accepted counts 0..k, including 0 and k)."""
    import torch

    Hk, Hv, d = shape
    A = Layer(21, Hk, Hv, d, n_slots=33, s_std=0.02, tail_std=1.0)
    Bl, arr, words = _device_layer(21, Hk, Hv, d, n_slots=33)
    vf.gdn_state_to_device(arr, words)
    assert _dev_cur(words) == 0
    rng = np.random.default_rng(k)
    acc_t = torch.zeros(1, dtype=torch.int32, device="cuda")
    for step in range(5):
        inp = S.gdn_inputs(21, f"devc.{k}.{step}", k, Hk, Hv, d)
        oa = A.verify(vf, inp, k)
        ob = Bl.verify(vf, inp, k)
        assert np.array_equal(oa.view(np.uint32), ob.view(np.uint32)), f"step {step} o"
        assert int(host(words)[0, 1]) == k  # rows pending on the device
        a = [0, k, int(rng.integers(0, k + 1)), 1, int(rng.integers(0, k + 1))][step]
        vf.gdn_commit(A.state, a)
        acc_t.fill_(a)
        vf.gdn_commit_dev(arr, acc_t)
        torch.cuda.synchronize()
        cur = _dev_cur(words)
        assert cur == A.state.cur, f"step {step}: device slot {cur}, host slot {A.state.cur}"
        assert int(host(words)[0, 1]) == 0
        Sa, ta = A.slot(A.state.cur)
        Sb, tb = Bl.slot(cur)
        assert np.array_equal(Sa.view(np.uint32), Sb.view(np.uint32)) and np.array_equal(ta, tb)
    vf.gdn_state_to_host(arr)
    assert arr[0].dev is None and arr[0].cur == A.state.cur


def test_accept_commits_every_state(vf):
    """verify_accept_greedy with states: the accepted count a = m + 1 is
    committed on every layer's state, as a host commit of a would."""
    import torch

    k, V, n = 6, 7000, 3
    layers = [Layer(30 + l, 2, 4, 32, n_slots=8, s_std=0.02, tail_std=1.0) for l in range(n)]
    host_layers = [Layer(30 + l, 2, 4, 32, n_slots=8, s_std=0.02, tail_std=1.0) for l in range(n)]
    arr = (B.GdnState * n)()
    for l, L in enumerate(layers):
        arr[l] = L.state
        L.state = arr[l]
    words = torch.full((n, 2), -1, dtype=torch.int32, device="cuda")
    vf.gdn_state_to_device(arr, words)
    for step, m in enumerate([2, 5, 0, 3]):
        for l in range(n):
            inp = S.gdn_inputs(30 + l, f"acc.{step}", k, 2, 4, 32)
            layers[l].verify(vf, inp, k)
            host_layers[l].verify(vf, inp, k)
        x = S.vocab_logits(13, f"acc.logits.{step}", k, V, 0)
        _, _, t = O.accept_greedy(x, np.zeros(k - 1, np.int32))
        draft = _drafts(t, m, V, np.random.default_rng(step))
        a, nxt, _ = O.accept_greedy(x, draft)
        got = _accept(vf, x, draft, states=arr)
        assert got[0] == a == m + 1 and got[1] == nxt
        w = host(words)
        for l in range(n):
            vf.gdn_commit(host_layers[l].state, a)
            assert w[l, 0] == host_layers[l].state.cur and w[l, 1] == 0
            Sa, ta = host_layers[l].slot(host_layers[l].state.cur)
            Sb, tb = layers[l].slot(int(w[l, 0]))
            assert np.array_equal(Sa.view(np.uint32), Sb.view(np.uint32)) and np.array_equal(ta, tb)
    vf.gdn_state_to_host(arr)


def test_device_commit_sequence_errors(vf):
    """A device commit with no verify pending, or beyond the pending rows,
    commits nothing and reports device error 3; a corrupted committed slot
    makes the verify write nothing and report device error 4.  No fault, no
    hang: the context stays usable."""
    import torch

    L, arr, words = _device_layer(40, 2, 2, 32, n_slots=6)
    vf.gdn_state_to_device(arr, words)
    acc_t = torch.ones(1, dtype=torch.int32, device="cuda")
    vf.gdn_commit_dev(arr, acc_t)  # nothing pending
    assert vf.device_status() == (B.EDEVICE, 3)
    assert host(words).tolist() == [[0, 0]]
    inp = S.gdn_inputs(40, "seq", 3, 2, 2, 32)
    L.verify(vf, inp, 3)
    acc_t.fill_(4)
    vf.gdn_commit_dev(arr, acc_t)  # more rows than verified
    assert vf.device_status() == (B.EDEVICE, 3)
    assert host(words).tolist() == [[0, 3]]
    # greedy acceptance requires the pending width to equal k
    x = S.vocab_logits(14, "seq.logits", 2, 100, 0)
    _accept(vf, x, [0], states=arr)
    assert vf.device_status() == (B.EDEVICE, 3)
    assert host(words).tolist() == [[0, 3]]
    acc_t.fill_(2)
    vf.gdn_commit_dev(arr, acc_t)
    assert vf.device_status() == (B.OK, 0)
    assert host(words).tolist() == [[2, 0]]  # state after 2 rows: slot 1 + (1 >= 0)
    # a committed slot outside the ring: the verify leaves every slot untouched
    before = [L.slot(s) for s in range(6)]
    words[0, 0] = 6
    L.verify(vf, inp, 3)
    assert vf.device_status() == (B.EDEVICE, 4)
    for s in range(6):
        after = L.slot(s)
        assert np.array_equal(after[0].view(np.uint32), before[s][0].view(np.uint32))
        assert np.array_equal(after[1], before[s][1])
    assert host(words).tolist() == [[6, 0]]
    words[0, 0] = 2
    # host commits refuse a device-held state; a second move to the device too
    with pytest.raises(B.VerifyError):
        vf.gdn_commit(L.state, 1)
    with pytest.raises(B.VerifyError):
        vf.gdn_state_to_device(arr, words)
    vf.gdn_state_to_host(arr)
    assert arr[0].cur == 2


# ------------------------------------------------- the stack, graph replays

@pytest.mark.parametrize("k", [4, 9])
def test_stack_device_loop_equals_host_loop(vf, k):
    """Several verify steps through a small 2-layer stack: once with host
    commits (verify, then the oracle's accepted count committed from the
    host), once as one graph replay per step of verify + device acceptance
    with its fused commit.  The residual outputs agree bit for bit, and so do
    the committed slots and their contents."""
    import torch

    from speculative_decode_verification_gb300.stack import DeviceStack

    cfg = dict(layers=2, H=256, E=16, T=4, I=256, n_qk_heads=2, n_v_heads=4, d=64, conv_kernel=4)
    V = 5000
    host_st = DeviceStack(vf, cfg, seed=5, n_slots=k + 1)
    dev_st = DeviceStack(vf, cfg, seed=5, n_slots=k + 1)
    dev_st.to_device()
    h_a = torch.zeros((k, cfg["H"]), dtype=torch.float32, device="cuda")
    h_b = torch.zeros_like(h_a)
    logits = torch.zeros((k, V), dtype=torch.float32, device="cuda")
    draft = torch.zeros(max(k - 1, 1), dtype=torch.int32, device="cuda")
    result = torch.zeros(2 + k, dtype=torch.int32, device="cuda")
    rng = np.random.default_rng(k)
    for step, m in enumerate([k - 1, 0, k // 2, 1, k - 1, 2]):
        h0 = torch.from_numpy(S.f32_normal(5, f"loop.h.{k}.{step}", (k, cfg["H"])))
        x = S.vocab_logits(5, f"loop.logits.{k}.{step}", k, V, 0)
        _, _, t = O.accept_greedy(x, np.zeros(k - 1, np.int32))
        d = _drafts(t, m, V, rng)
        a, nxt, _ = O.accept_greedy(x, d)
        h_a.copy_(h0)
        h_b.copy_(h0)
        logits.copy_(torch.from_numpy(x))
        draft[: k - 1].copy_(torch.from_numpy(d))
        host_st.verify(h_a, k)
        host_st.commit(a)
        dev_st.verify_accept(h_b, k, logits, draft, result)
        torch.cuda.synchronize()
        assert np.array_equal(host(h_a).view(np.uint32), host(h_b).view(np.uint32)), f"step {step}"
        res = host(result)
        assert res[0] == a == m + 1 and res[1] == nxt
        w = host(dev_st.dev_words)
        for l in range(cfg["layers"]):
            cur = int(host_st.states[l].cur)
            assert w[l, 0] == cur and w[l, 1] == 0
            Sa = host(host_st.state_tensors[l][0][cur])
            Sb = host(dev_st.state_tensors[l][0][cur])
            assert np.array_equal(Sa.view(np.uint32), Sb.view(np.uint32))
    assert len(dev_st._graphs) == 1  # one capture served every step
    dev_st.to_host()
    assert [int(s.cur) for s in dev_st.states] == [int(s.cur) for s in host_st.states]


# ------------------------------------------- token selection at the target

@pytest.mark.parametrize("k", [1, 4, 9])
def test_token_selection_over_a_q4_lm_head(vf, k):
    """GPU token selection over the full vocabulary: the Q4 LM head
    (q4_qmv_k at N = 248,320, hidden 256 here so that the oracle computes
    every logit) and then greedy acceptance on the device.  The argmax is
    decided on fp32 logits on both sides (the oracle's float64 sums rounded
    to fp32); a row whose two largest oracle logits lie within twice the
    product tolerance may resolve either way, and then the GPU's choice must
    be one of the near-maximal tokens."""
    import torch

    from tests.gpu_util import DevQ4, assert_close

    V, H = S.FLASH_VOCAB, 256
    m = S.q4_matrix(7, "select.lm_head", V, H, centered=True)
    W = DevQ4(vf, m)
    x = S.bf16_normal(7, f"select.x{k}", (k, H))
    y = torch.zeros((k, V), dtype=torch.float32, device="cuda")
    vf.q4_qmv_k(W.struct, dev(x), k, y, B.F32)
    ref = O.q4_qmv(m.packed, m.scales, m.biases, x)
    torch.cuda.synchronize()
    assert_close(host(y), ref, what="LM head logits")
    ref32 = ref.astype(np.float32)
    _, _, t_o = O.accept_greedy(ref32, np.zeros(k - 1, np.int32))
    tol = 2e-3 * float(np.sqrt(np.mean(ref * ref)))
    decisive = []
    for r in range(k):
        top2 = np.partition(ref[r], -2)[-2:]
        decisive.append(top2[1] - top2[0] > tol)
    assert sum(decisive) >= k - 1
    n_lead = next((r for r, dcs in enumerate(decisive) if not dcs), k)  # rows decided without doubt
    m_acc = max(0, min(n_lead - 1, k - 1))
    draft = _drafts(t_o, m_acc, V, np.random.default_rng(k))
    a, nxt, _ = O.accept_greedy(ref32, draft)
    res = torch.zeros(2 + k, dtype=torch.int32, device="cuda")
    vf.accept_greedy(y, k, dev(draft) if k > 1 else None, res)
    torch.cuda.synchronize()
    got = host(res)
    for r in range(k):
        if decisive[r]:
            assert got[2 + r] == t_o[r], f"row {r}"
        else:
            assert ref[r, got[2 + r]] >= ref[r].max() - tol, f"row {r}: not a near-maximal token"
    if all(decisive[: m_acc + 1]):
        assert got[0] == a and got[1] == nxt


def test_stack_select_accept_graph_equals_eager_composition(vf):
    """The whole target side of a decode step as one graph replay (verify,
    final norm, Q4 LM head over the full vocabulary, device acceptance and
    commit) gives bit for bit what the same calls give launched one by one
    with host commits, step after step."""
    import torch

    from speculative_decode_verification_gb300.stack import DeviceStack

    cfg = dict(layers=2, H=256, E=16, T=4, I=256, n_qk_heads=2, n_v_heads=4, d=64, conv_kernel=4)
    k, V = 5, S.FLASH_VOCAB
    a_st = DeviceStack(vf, cfg, seed=9, n_slots=k + 1, vocab=V, graphs=False)
    b_st = DeviceStack(vf, cfg, seed=9, n_slots=k + 1, vocab=V)
    b_st.to_device()
    h_a = torch.zeros((k, cfg["H"]), dtype=torch.float32, device="cuda")
    h_b = torch.zeros_like(h_a)
    draft = torch.zeros(k - 1, dtype=torch.int32, device="cuda")
    res_a = torch.zeros(2 + k, dtype=torch.int32, device="cuda")
    res_b = torch.zeros_like(res_a)
    for step in range(4):
        h0 = torch.from_numpy(S.f32_normal(9, f"select.h.{step}", (k, cfg["H"])))
        h_a.copy_(h0)
        h_b.copy_(h0)
        # drafts: the eager side's own choices up to row `step`, so that the
        # accepted count varies from step to step
        a_st.verify(h_a, k)
        lg = a_st.select(h_a, k)
        vf.accept_greedy(lg, k, None if k == 1 else draft, res_a)
        torch.cuda.synchronize()
        t = host(res_a)[2:]
        d = t[: k - 1].copy()
        if step < k - 1:
            d[step] = (t[step] + 1) % V
        draft.copy_(torch.from_numpy(d))
        vf.accept_greedy(lg, k, draft, res_a)
        torch.cuda.synchronize()
        a = int(host(res_a)[0])
        assert a == min(step, k - 1) + 1
        a_st.commit(a)
        b_st.verify_select_accept(h_b, k, draft, res_b)
        torch.cuda.synchronize()
        assert np.array_equal(host(h_a).view(np.uint32), host(h_b).view(np.uint32)), f"step {step}"
        assert np.array_equal(host(res_a), host(res_b)), f"step {step}"
        w = host(b_st.dev_words)
        assert [int(x) for x in w[:, 0]] == [int(s.cur) for s in a_st.states]
    assert len(b_st._graphs) == 1


@pytest.mark.parametrize("V,H,k", [(S.FLASH_VOCAB, 256, 1), (S.FLASH_VOCAB, 256, 9), (S.FLASH_VOCAB, 256, 32),
                                   (1000, 512, 16), (333, 1024, 5)])
def test_lm_head_accept_equals_product_then_accept(vf, V, H, k):
    """verify_lm_head_accept (the LM head with its argmax epilogue) gives bit
    for bit what q4_qmv_k followed by verify_accept_greedy gives, for
    several accepted prefixes."""
    import torch

    from tests.gpu_util import DevQ4

    m = S.q4_matrix(31, f"lmf.{V}.{H}", V, H, centered=True)
    W = DevQ4(vf, m)
    x = dev(S.bf16_normal(31, f"lmf.x.{k}", (k, H)))
    y = torch.zeros((k, V), dtype=torch.float32, device="cuda")
    vf.q4_qmv_k(W.struct, x, k, y, B.F32)
    res_a = torch.zeros(2 + k, dtype=torch.int32, device="cuda")
    res_b = torch.full((2 + k,), -5, dtype=torch.int32, device="cuda")
    draft = torch.zeros(max(k - 1, 1), dtype=torch.int32, device="cuda")
    vf.accept_greedy(y, k, None if k == 1 else draft, res_a)
    torch.cuda.synchronize()
    t = host(res_a)[2:]
    for mm in sorted({0, k // 2, k - 1}):
        d = _drafts(t, mm, V, np.random.default_rng(mm))
        if k > 1:
            draft[: k - 1].copy_(torch.from_numpy(d))
        vf.accept_greedy(y, k, None if k == 1 else draft, res_a)
        vf.lm_head_accept(W.struct, x, k, None if k == 1 else draft, res_b)
        torch.cuda.synchronize()
        assert np.array_equal(host(res_a), host(res_b)), f"m={mm}"
        assert host(res_b)[0] == mm + 1


def test_stack_fused_and_unfused_target_steps_agree(vf):
    """One graph per step of the whole target side, with the fused LM-head
    acceptance and with the logits written and read back: the same results,
    residuals and committed slots, step after step."""
    import torch

    from speculative_decode_verification_gb300.stack import DeviceStack

    cfg = dict(layers=2, H=256, E=16, T=4, I=256, n_qk_heads=2, n_v_heads=4, d=64, conv_kernel=4)
    k, V = 9, 50000
    a_st = DeviceStack(vf, cfg, seed=12, n_slots=k + 1, vocab=V)
    b_st = DeviceStack(vf, cfg, seed=12, n_slots=k + 1, vocab=V)
    a_st.to_device()
    b_st.to_device()
    h_a = torch.zeros((k, cfg["H"]), dtype=torch.float32, device="cuda")
    h_b = torch.zeros_like(h_a)
    draft = torch.zeros(k - 1, dtype=torch.int32, device="cuda")
    res_a = torch.zeros(2 + k, dtype=torch.int32, device="cuda")
    res_b = torch.zeros_like(res_a)
    for step in range(4):
        h0 = torch.from_numpy(S.f32_normal(12, f"fused.h.{step}", (k, cfg["H"])))
        h_a.copy_(h0)
        h_b.copy_(h0)
        draft.copy_(torch.from_numpy(S.f32_uniform(12, f"fused.d.{step}", (k - 1,), 0, V).astype(np.int32)))
        a_st.verify_select_accept(h_a, k, draft, res_a, fused=False)
        b_st.verify_select_accept(h_b, k, draft, res_b, fused=True)
        torch.cuda.synchronize()
        assert np.array_equal(host(res_a), host(res_b)), f"step {step}"
        assert np.array_equal(host(h_a).view(np.uint32), host(h_b).view(np.uint32))
        assert np.array_equal(host(a_st.dev_words), host(b_st.dev_words))
