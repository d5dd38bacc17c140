"""A synthetic hybrid verify stack on the device: L layers of (Gated DeltaNet
mixer -> MoE with 10 routed + 1 shared expert), random-init weights drawn by
the seeded generator (large Q4 tensors by its device twin), one ring of GDN
state slots per layer.  Running a verify pass is one ``verify_layer_k`` call
per layer; committing the accepted prefix is one ``gdn_commit`` per layer, or,
with the committed slots held on the device (``to_device``), one acceptance
kernel that also commits (``verify_accept``), with no host round trip.

Tensor names (the seeds of the generator) are shared with the host side, so
any weight can be re-drawn on the host bit for bit.
"""
from __future__ import annotations

import numpy as np

from . import binding as B
from . import synth as S


def layer_names(l: int):
    p = f"stack.L{l}"
    return dict(in_proj=p + ".in_proj", out_proj=p + ".out_proj", router=p + ".router", gate_up=p + ".gate_up",
                down=p + ".down", shared_gate_up=p + ".shared_gate_up", shared_down=p + ".shared_down",
                gdn=p + ".gdn", norm1=p + ".norm1", norm2=p + ".norm2")


def shapes(cfg):
    H, d, Hk, Hv = cfg["H"], cfg["d"], cfg["n_qk_heads"], cfg["n_v_heads"]
    C = 2 * Hk * d + Hv * d
    NP = C + Hv * d + 2 * Hv
    return dict(H=H, C=C, NP=NP, Z=Hv * d, E=cfg["E"], I=cfg["I"], T=cfg["T"])


class DeviceStack:
    """All layers' weights and GDN state slots on the current CUDA device."""

    def __init__(self, vf: B.Verify, cfg, seed: int = 0, n_slots: int = 10, s_std: float = 0.02,
                 tail_std: float = 1.0, layers: int | None = None, keep_rows: bool = False, graphs: bool = True,
                 vocab: int = 0):
        import torch

        self.vf, self.cfg, self.seed = vf, cfg, seed
        self.use_graphs = graphs
        self._graphs = {}
        self.dev_words = None  # int32 [layers, 2] once the committed slots live on the device
        self.n_layers = cfg["layers"] if layers is None else layers
        sh = shapes(cfg)
        self.sh = sh
        H, E, I = sh["H"], sh["E"], sh["I"]
        d, Hk, Hv = cfg["d"], cfg["n_qk_heads"], cfg["n_v_heads"]
        self.keep = []
        self.rows = []  # with keep_rows: the row-layout (packed, scales, biases) of every Q4 tensor, in draw order
        # ctypes arrays, passed whole to verify_stack_k / gdn_commit_all; indexing
        # gives views that write through (e.g. resetting one layer's cur)
        self.layers = (B.Layer * self.n_layers)()
        self.states = (B.GdnState * self.n_layers)()
        self.state_tensors = []

        def q4(name, n_out, k_in, n_experts=None, gate_up=False, down=False):
            # drawn in the row layout, kept only in the tiled layout
            e = 1 if n_experts is None else n_experts
            shp = (e, n_out, k_in // 8) if n_experts else (n_out, k_in // 8)
            gshp = (e, n_out, k_in // 64) if n_experts else (n_out, k_in // 64)
            p = torch.empty(shp, dtype=torch.int32, device="cuda")
            sc = torch.empty(gshp, dtype=torch.int16, device="cuda")
            bi = torch.empty(gshp, dtype=torch.int16, device="cuda")
            vf.synth_q4(p, sc, bi, S.q4_seeds(seed, name), S.SCALE_RANGE, S.CENTERED_RANGE, centered=True)
            rows = B.q4_experts(p, sc, bi) if n_experts else B.q4_weight(p, sc, bi)
            t = vf.tile(rows, gate_up=gate_up, down=down)
            torch.cuda.synchronize()
            if keep_rows:
                self.rows.append((p, sc, bi))
            del p, sc, bi
            self.keep.append(t.buf)
            return t.struct

        def dev(a):
            t = torch.from_numpy(np.ascontiguousarray(a)).cuda()
            self.keep.append(t)
            return t

        for l in range(self.n_layers):
            nm = layer_names(l)
            gp = {k: dev(v) for k, v in S.gdn_params(seed, nm["gdn"], Hk, Hv, d).items()}
            L = B.Layer()
            L.in_proj = q4(nm["in_proj"], sh["NP"], H)
            L.out_proj = q4(nm["out_proj"], H, sh["Z"])
            L.router = q4(nm["router"], E + 1, H)
            L.gate_up = q4(nm["gate_up"], 2 * I, H, E, gate_up=True)
            L.down = q4(nm["down"], H, I, E, down=True)
            L.shared_gate_up = q4(nm["shared_gate_up"], 2 * I, H, gate_up=True)
            L.shared_down = q4(nm["shared_down"], H, I, down=True)
            L.gdn = B.gdn_params(Hk, Hv, d, gp["conv_w"], gp["A_log"], gp["dt_bias"], gp["norm_w"])
            L.norm1_w = dev(S.f32_uniform(seed, nm["norm1"], (H,), -0.1, 0.1)).data_ptr()
            L.norm2_w = dev(S.f32_uniform(seed, nm["norm2"], (H,), -0.1, 0.1)).data_ptr()
            L.norm_eps = 1e-6
            L.top_k = sh["T"]
            self.layers[l] = L
            S0, t0 = S.gdn_initial_state(seed, nm["gdn"], Hk, Hv, d, s_std=s_std, tail_std=tail_std)
            slots = [torch.zeros((Hv, d, d), dtype=torch.float32, device="cuda") for _ in range(n_slots)]
            tails = [torch.zeros((3, sh["C"]), dtype=torch.int16, device="cuda") for _ in range(n_slots)]
            slots[0].copy_(torch.from_numpy(S0))
            tails[0].copy_(torch.from_numpy(t0.view(np.int16)))
            self.state_tensors.append((slots, tails))
            self.states[l] = B.gdn_state(slots, tails, cur=0)
        # target head (vocab > 0): final zero-centred norm and a Q4 LM head [vocab, H]
        self.vocab = vocab
        if vocab:
            self.final_norm_w = dev(S.f32_uniform(seed, "stack.final_norm", (H,), -0.1, 0.1))
            self.lm_head = q4("stack.lm_head", vocab, H)
            self.xn = torch.zeros((16, H), dtype=torch.int16, device="cuda")
            self.logits = torch.zeros((16, vocab), dtype=torch.float32, device="cuda")

    def verify(self, h, k: int, idx=None, stream=None):
        """One verify pass of k rows through every layer; h (fp32 [k, H]) is
        updated in place.  idx (optional): per-layer int32 [k, T] device
        tensors receiving the routed expert indices."""
        if idx is None:
            if self.use_graphs:
                self._verify_graphed(h, k, stream)
            else:  # one call for the whole pass
                self.vf.verify_stack_k(self.layers, self.states, h, k, None, stream)
            return
        for l, (L, st) in enumerate(zip(self.layers, self.states)):
            self.vf.verify_layer_k(L, st, h, k, idx[l], stream)

    def _verify_graphed(self, h, k: int, stream=None):
        """verify_stack_k through a CUDA graph: captured once per (k, h buffer,
        every layer's current slot and pending count) and replayed after.  Which
        slots a pass writes depends only on those, so a replay does what the
        call would.  The capture runs the host side of the call (checks, slot
        bookkeeping) without running kernels; its resulting states are restored
        before every replay."""
        import ctypes

        import torch

        if self.dev_words is not None:  # the kernels read the committed slots themselves
            key = (k, h.data_ptr(), "dev")
        else:
            key = (k, h.data_ptr(), tuple((int(st.cur), int(st.pending_k)) for st in self.states))
        ent = self._graphs.get(key)
        if ent is None:
            ent = self._capture(key, lambda st: self.vf.verify_stack_k(self.layers, self.states, h, k, None, st))
        g, post = ent
        ctypes.memmove(ctypes.addressof(self.states), post, len(post))
        run = torch.cuda.ExternalStream(stream) if stream else torch.cuda.current_stream()
        with torch.cuda.stream(run):
            g.replay()

    def _capture(self, key, enqueue):
        import torch

        g = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream()
        cap.wait_stream(torch.cuda.current_stream())
        with torch.cuda.graph(g, stream=cap, capture_error_mode="thread_local"):
            enqueue(cap.cuda_stream)
        ent = (g, bytes(self.states))
        self._graphs[key] = ent
        return ent

    def commit(self, accepted: int):
        self.vf.gdn_commit_all(self.states, accepted)

    # ------------------------------------------------ device-held commits

    def to_device(self):
        """Moves every layer's committed slot to the device: from here on the
        verify kernels read it there and only device commits change it."""
        import torch

        words = torch.zeros((self.n_layers, 2), dtype=torch.int32, device="cuda")
        self.vf.gdn_state_to_device(self.states, words)
        self.dev_words = words
        self._graphs.clear()

    def to_host(self):
        self.vf.gdn_state_to_host(self.states)
        self.dev_words = None
        self._graphs.clear()

    def commit_dev(self, accepted, stream=None):
        """Commits the device-held int32 count `accepted` on every layer."""
        self.vf.gdn_commit_dev(self.states, accepted, stream)

    def select(self, h, k: int, stream=None):
        """Target logits of the k rows of h: final norm (bf16 rows), then the Q4
        LM head; returns the fp32 [k, vocab] view of the logits buffer."""
        import torch

        st = stream if stream else torch.cuda.current_stream().cuda_stream
        H = self.sh["H"]
        self.vf.verify_rmsnorm_k(h, self.final_norm_w, 1e-6, True, H, k, self.xn, B.BF16, st)
        lg = self.logits[:k]
        self.vf.q4_qmv_k(self.lm_head, self.xn, k, lg, B.F32, st)
        return lg

    def verify_select_accept(self, h, k: int, draft, result, stream=None, fused: bool = True):
        """The whole target side of a decode step on the device: the verify
        pass, the final norm and LM head over the full vocabulary, greedy
        acceptance of `draft` (int32 [k-1]) and the commit of every layer.
        `result` (int32 [2 + k]) receives the accepted rows, the next token and
        the k greedy choices.  fused: the LM head's argmax epilogue does the
        acceptance (verify_lm_head_accept; the logits never reach memory), else
        the logits are written and verify_accept_greedy reads them.  Needs
        vocab > 0 and device-held commits; with graphs, one replay per call."""
        import torch

        if self.dev_words is None or not self.vocab:
            raise RuntimeError("verify_select_accept needs vocab > 0 and to_device()")

        def enqueue(st):
            self.vf.verify_stack_k(self.layers, self.states, h, k, None, st)
            if fused:
                H = self.sh["H"]
                self.vf.verify_rmsnorm_k(h, self.final_norm_w, 1e-6, True, H, k, self.xn, B.BF16, st)
                self.vf.lm_head_accept(self.lm_head, self.xn, k, draft, result, states=self.states, stream=st)
            else:
                lg = self.select(h, k, st)
                self.vf.accept_greedy(lg, k, draft, result, states=self.states, stream=st)

        if not self.use_graphs:
            enqueue(stream if stream else torch.cuda.current_stream().cuda_stream)
            return
        key = ("select", fused, k, h.data_ptr(), None if draft is None else draft.data_ptr(), result.data_ptr())
        g, _ = self._graphs.get(key) or self._capture(key, enqueue)
        run = torch.cuda.ExternalStream(stream) if stream else torch.cuda.current_stream()
        with torch.cuda.stream(run):
            g.replay()

    def verify_accept(self, h, k: int, logits, draft, result, stream=None):
        """A verify pass, then greedy acceptance of the block against `logits`
        (fp32 [k, V], the target's logits of the k rows) and `draft` (int32
        [k-1]) with the commit of every layer, all on the device: `result`
        (int32 [2 + k]) receives the accepted rows, the next token and the k
        greedy choices.  With graphs, one replay per call."""
        import torch

        if self.dev_words is None:
            raise RuntimeError("verify_accept needs device-held commits: call to_device() first")

        def enqueue(st):
            self.vf.verify_stack_k(self.layers, self.states, h, k, None, st)
            self.vf.accept_greedy(logits, k, draft, result, states=self.states, stream=st)

        if not self.use_graphs:
            enqueue(stream if stream else torch.cuda.current_stream().cuda_stream)
            return
        key = ("accept", k, h.data_ptr(), logits.data_ptr(), logits.stride(0), logits.shape[1],
               None if draft is None else draft.data_ptr(), result.data_ptr())
        g, _ = self._graphs.get(key) or self._capture(key, enqueue)
        run = torch.cuda.ExternalStream(stream) if stream else torch.cuda.current_stream()
        with torch.cuda.stream(run):
            g.replay()

    def weight_bytes(self):
        return sum(t.numel() * t.element_size() for t in self.keep)
