"""Thin ctypes binding of libverify.so (include/verify.h).

Argument marshalling only: every step of the verify pass runs in the CUDA
library.  Tensors are passed as device pointers (``tensor.data_ptr()``) and
the stream as ``torch.cuda.current_stream().cuda_stream``; PyTorch is used for
device memory and streams, nothing else.  There is no CPU fallback: if the
library is missing, loading fails with an error that says how to build it.
"""
from __future__ import annotations

import ctypes as C
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libverify.so")

OK, EINVAL, EUNSUPPORTED, ECUDA, EDEVICE = 0, 1, 2, 3, 4
F32, BF16, F32_ADD = 0, 1, 2
ROWS, TILED, TILED_GATE_UP, TILED_DOWN = 0, 1, 2, 3  # verify_q4_layout
TILE_DENSE, TILE_GATE_UP, TILE_DOWN = 0, 1, 2  # verify_tile_kind
MAX_K = 32
PASS_K = 16
GDN_MAX_SLOTS = 33

_lib = None


class VerifyError(RuntimeError):
    def __init__(self, status, msg):
        super().__init__(f"status {status}: {msg}")
        self.status = status


class Q4Weight(C.Structure):
    _fields_ = [("packed", C.c_void_p), ("scales", C.c_void_p), ("biases", C.c_void_p),
                ("n_out", C.c_int32), ("k_in", C.c_int32), ("group_size", C.c_int32), ("bits", C.c_int32),
                ("layout", C.c_int32)]


class Q4Experts(C.Structure):
    _fields_ = [("w", Q4Weight), ("n_experts", C.c_int32)]


class GdnParams(C.Structure):
    _fields_ = [("n_qk_heads", C.c_int32), ("n_v_heads", C.c_int32), ("head_dim_k", C.c_int32),
                ("head_dim_v", C.c_int32), ("conv_kernel", C.c_int32), ("q_scale", C.c_float),
                ("l2_eps", C.c_float), ("norm_eps", C.c_float), ("gate_act", C.c_int32),
                ("conv_w", C.c_void_p), ("A_log", C.c_void_p), ("dt_bias", C.c_void_p), ("norm_w", C.c_void_p)]


class GdnState(C.Structure):
    _fields_ = [("S_slots", C.c_void_p * GDN_MAX_SLOTS), ("conv_slots", C.c_void_p * GDN_MAX_SLOTS),
                ("n_slots", C.c_int32), ("cur", C.c_int32), ("pending_k", C.c_int32),
                ("pending", C.c_int32 * GDN_MAX_SLOTS), ("dev", C.c_void_p)]


class GdnInputs(C.Structure):
    _fields_ = [("qkv", C.c_void_p), ("ld_qkv", C.c_int64), ("z", C.c_void_p), ("ld_z", C.c_int64),
                ("a", C.c_void_p), ("ld_a", C.c_int64), ("b", C.c_void_p), ("ld_b", C.c_int64)]


class AttnParams(C.Structure):
    _fields_ = [("n_q_heads", C.c_int32), ("n_kv_heads", C.c_int32), ("head_dim", C.c_int32),
                ("rope_dim", C.c_int32), ("rope_theta", C.c_float)]


class KvCache(C.Structure):
    _fields_ = [("K", C.c_void_p), ("V", C.c_void_p), ("capacity", C.c_int64), ("len", C.c_int32),
                ("split", C.c_int32), ("pending_k", C.c_int32), ("work", C.c_void_p), ("work_bytes", C.c_int64)]


class AttnInputs(C.Structure):
    _fields_ = [("q", C.c_void_p), ("ld_q", C.c_int64), ("gate", C.c_void_p), ("ld_gate", C.c_int64),
                ("k", C.c_void_p), ("ld_k", C.c_int64), ("v", C.c_void_p), ("ld_v", C.c_int64)]


class Layer(C.Structure):
    _fields_ = [("in_proj", Q4Weight), ("out_proj", Q4Weight), ("router", Q4Weight), ("gate_up", Q4Experts),
                ("down", Q4Experts), ("shared_gate_up", Q4Weight), ("shared_down", Q4Weight),
                ("gdn", GdnParams), ("norm1_w", C.c_void_p), ("norm2_w", C.c_void_p), ("norm_eps", C.c_float),
                ("top_k", C.c_int32)]


def load():
    """Loads libverify.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                           "`python -c 'import __graft_entry__ as g; g.build()'` (needs nvcc)")
    L = C.CDLL(LIB_PATH)
    p, i, i64, f = C.c_void_p, C.c_int, C.c_int64, C.c_float
    sig = {
        "verify_init": [i, C.POINTER(p)],
        "q4_tiled_bytes": [C.c_int32, C.c_int32, C.c_int32, C.c_int32],
        "q4_tile": [p, C.POINTER(Q4Weight), C.c_int32, C.c_int32, p, i64, C.POINTER(Q4Weight), p],
        "verify_destroy": [p],
        "verify_last_error": [p],
        "verify_device_status": [p, p, C.POINTER(C.c_int32)],
        "verify_launch_count": [p],
        "verify_selftest_stuck_wait": [p, p],
        "q4_qmv_k": [p, C.POINTER(Q4Weight), p, i, p, i, p],
        "q4_gather_experts_k": [p, C.POINTER(Q4Experts), C.POINTER(Q4Experts), p, i64, i, p, i, p, p, p, i,
                                C.POINTER(Q4Weight), C.POINTER(Q4Weight), p, p],
        "gdn_verify_k": [p, C.POINTER(GdnParams), C.POINTER(GdnState), C.POINTER(GdnInputs), i, p, i, p],
        "gdn_commit": [C.POINTER(GdnState), i],
        "verify_rmsnorm_k": [p, p, p, f, i, i, i, p, i, p],
        "verify_synth_q4": [p, p, p, p, i64, i64, C.c_uint64, C.c_uint64, C.c_uint64, f, f, f, f, i, p],
        "verify_layer_k": [p, C.POINTER(Layer), C.POINTER(GdnState), p, i, p, p],
        "verify_stack_k": [p, C.POINTER(Layer), C.POINTER(GdnState), i, p, i, p, p],
        "gdn_commit_all": [C.POINTER(GdnState), i, i],
        "verify_set_layer_events": [p, C.POINTER(p), i],
        "attn_workspace_bytes": [C.POINTER(AttnParams), i64, C.c_int32, C.c_int32],
        "attn_default_split": [i64],
        "attn_verify_k": [p, C.POINTER(AttnParams), C.POINTER(KvCache), C.POINTER(AttnInputs), i, p, i, p],
        "attn_commit": [C.POINTER(KvCache), i],
        "gdn_state_to_device": [p, C.POINTER(GdnState), i, p, p],
        "gdn_state_to_host": [p, C.POINTER(GdnState), i, p],
        "gdn_commit_dev": [p, C.POINTER(GdnState), i, p, p],
        "verify_accept_greedy": [p, p, i64, i, i, p, p, C.POINTER(GdnState), i, p],
        "verify_lm_head_accept": [p, C.POINTER(Q4Weight), p, i, p, p, C.POINTER(GdnState), i, p],
        "q4_gather_experts_k_noalloc": [C.POINTER(Q4Experts), C.POINTER(Q4Experts), p, i64, i, p, i, p, p, p, i,
                                        C.POINTER(Q4Weight), C.POINTER(Q4Weight), p, p, p],
    }
    for name, args in sig.items():
        fn = getattr(L, name)
        fn.argtypes = args
        fn.restype = C.c_int
    L.verify_last_error.restype = C.c_char_p
    L.verify_launch_count.restype = C.c_int64
    L.q4_tiled_bytes.restype = C.c_int64
    L.attn_workspace_bytes.restype = C.c_int64
    _lib = L
    return L


def _ptr(t):
    return None if t is None else C.c_void_p(t.data_ptr())


def q4_weight(packed, scales, biases) -> Q4Weight:
    """Row-layout Q4Weight over device tensors packed [N, K/8] (int32/uint32),
    scales/biases [N, K/64] (bf16 bits).  Compute calls take its tiled form
    (Verify.tile)."""
    n_out, k_in = packed.shape[-2], packed.shape[-1] * 8
    return Q4Weight(packed.data_ptr(), scales.data_ptr(), biases.data_ptr(), n_out, k_in, 64, 4, ROWS)


def q4_experts(packed, scales, biases) -> Q4Experts:
    """Row-layout Q4Experts over device tensors packed [E, N, K/8], scales/biases [E, N, K/64]."""
    E, n_out, k_in = packed.shape[0], packed.shape[1], packed.shape[2] * 8
    return Q4Experts(Q4Weight(packed.data_ptr(), scales.data_ptr(), biases.data_ptr(), n_out, k_in, 64, 4, ROWS), E)


class Tiled:
    """A tiled Q4 matrix (or expert stack): the device buffer and its struct
    (Q4Weight, or Q4Experts for a stack).  Keep it alive while calls use it."""

    def __init__(self, buf, struct):
        self.buf, self.struct = buf, struct


class Verify:
    """One library context (verify_ctx) on one device."""

    def __init__(self, device: int = 0):
        self.lib = load()
        self.ctx = C.c_void_p()
        st = self.lib.verify_init(device, C.byref(self.ctx))
        if st != OK:
            raise VerifyError(st, f"verify_init failed on device {device}")

    def close(self):
        if self.ctx:
            self.lib.verify_destroy(self.ctx)
            self.ctx = C.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def _check(self, st):
        if st != OK:
            raise VerifyError(st, self.lib.verify_last_error(self.ctx).decode())

    @staticmethod
    def _stream(stream):
        if stream is None:
            import torch
            stream = torch.cuda.current_stream().cuda_stream
        return C.c_void_p(int(stream))

    def launch_count(self) -> int:
        return int(self.lib.verify_launch_count(self.ctx))

    def selftest_stuck_wait(self, stream=None):
        """Launches the stuck-wait probe (verify_selftest_stuck_wait)."""
        self._check(self.lib.verify_selftest_stuck_wait(self.ctx, self._stream(stream)))

    def device_status(self, stream=None):
        code = C.c_int32(0)
        st = self.lib.verify_device_status(self.ctx, self._stream(stream), C.byref(code))
        return st, code.value

    # ------------------------------------------------------------ entry points

    def q4_qmv_k(self, W: Q4Weight, x, k: int, y, dtype_out: int = F32, stream=None):
        self._check(self.lib.q4_qmv_k(self.ctx, C.byref(W), _ptr(x), k, _ptr(y), dtype_out,
                                      self._stream(stream)))

    def q4_gather_experts_k(self, gate_up: Q4Experts, down: Q4Experts, logits, logits_ld: int, top_k: int,
                            x, k: int, idx_out, w_out, y, dtype_out: int = F32, shared_gate_up=None,
                            shared_down=None, shared_gate_logit=None, stream=None):
        self._check(self.lib.q4_gather_experts_k(
            self.ctx, C.byref(gate_up), C.byref(down), _ptr(logits), logits_ld, top_k, _ptr(x), k,
            _ptr(idx_out), _ptr(w_out), _ptr(y), dtype_out,
            C.byref(shared_gate_up) if shared_gate_up is not None else None,
            C.byref(shared_down) if shared_down is not None else None,
            _ptr(shared_gate_logit), self._stream(stream)))

    def gdn_verify_k(self, params: GdnParams, state: GdnState, inputs: GdnInputs, k: int, o,
                     dtype_out: int = F32, stream=None):
        self._check(self.lib.gdn_verify_k(self.ctx, C.byref(params), C.byref(state), C.byref(inputs), k,
                                          _ptr(o), dtype_out, self._stream(stream)))

    def gdn_commit(self, state: GdnState, accepted: int):
        st = self.lib.gdn_commit(C.byref(state), accepted)
        if st != OK:
            raise VerifyError(st, f"gdn_commit({accepted}) rejected")

    def verify_rmsnorm_k(self, x, w, eps: float, zero_centered: bool, n: int, k: int, out,
                         dtype_out: int = BF16, stream=None):
        self._check(self.lib.verify_rmsnorm_k(self.ctx, _ptr(x), _ptr(w), eps, int(bool(zero_centered)), n, k,
                                              _ptr(out), dtype_out, self._stream(stream)))

    def verify_layer_k(self, layer: Layer, state: GdnState, h, k: int, idx_out=None, stream=None):
        self._check(self.lib.verify_layer_k(self.ctx, C.byref(layer), C.byref(state), _ptr(h), k,
                                            _ptr(idx_out), self._stream(stream)))

    def verify_stack_k(self, layers, states, h, k: int, idx_out=None, stream=None):
        """One verify pass through every layer (verify_stack_k): layers and
        states are ctypes arrays of Layer and GdnState."""
        self._check(self.lib.verify_stack_k(self.ctx, layers, states, len(layers), _ptr(h), k,
                                            _ptr(idx_out) if idx_out is not None else None, self._stream(stream)))

    def gdn_commit_all(self, states, accepted: int):
        st = self.lib.gdn_commit_all(states, len(states), accepted)
        if st != OK:
            raise VerifyError(st, f"gdn_commit_all({accepted}) rejected")

    def attn_verify_k(self, params: AttnParams, cache: KvCache, inputs: AttnInputs, k: int, o,
                      dtype_out: int = F32, stream=None):
        self._check(self.lib.attn_verify_k(self.ctx, C.byref(params), C.byref(cache), C.byref(inputs), k,
                                           _ptr(o), dtype_out, self._stream(stream)))

    def attn_commit(self, cache: KvCache, accepted: int):
        st = self.lib.attn_commit(C.byref(cache), accepted)
        if st != OK:
            raise VerifyError(st, f"attn_commit({accepted}) rejected")

    def gdn_state_to_device(self, states, dev, stream=None):
        """Moves the committed slot of every state (a ctypes array of GdnState)
        to the device words dev (int32 [len(states), 2]); synchronises."""
        self._check(self.lib.gdn_state_to_device(self.ctx, states, len(states), _ptr(dev), self._stream(stream)))

    def gdn_state_to_host(self, states, stream=None):
        self._check(self.lib.gdn_state_to_host(self.ctx, states, len(states), self._stream(stream)))

    def gdn_commit_dev(self, states, accepted, stream=None):
        """Commits the device-held int32 accepted (a 1-element tensor) on every state."""
        self._check(self.lib.gdn_commit_dev(self.ctx, states, len(states), _ptr(accepted), self._stream(stream)))

    def accept_greedy(self, logits, k: int, draft, result, states=None, stream=None):
        """Greedy acceptance of a width-k block (verify_accept_greedy): logits
        fp32 [k, V] (row stride logits.stride(0)), draft int32 [k-1], result
        int32 [2 + k]; commits on the device-held states if given."""
        n = 0 if states is None else len(states)
        self._check(self.lib.verify_accept_greedy(
            self.ctx, _ptr(logits), logits.stride(0), logits.shape[1], k,
            _ptr(draft) if draft is not None and k > 1 else None, _ptr(result),
            states if n else None, n, self._stream(stream)))

    def lm_head_accept(self, W: Q4Weight, x, k: int, draft, result, states=None, stream=None):
        """The Q4 LM head with its argmax epilogue, then greedy acceptance and
        the commit (verify_lm_head_accept): x bf16 [k, H], draft int32
        [k-1], result int32 [2 + k]."""
        n = 0 if states is None else len(states)
        self._check(self.lib.verify_lm_head_accept(
            self.ctx, C.byref(W), _ptr(x), k, _ptr(draft) if draft is not None and k > 1 else None, _ptr(result),
            states if n else None, n, self._stream(stream)))

    def set_layer_events(self, events):
        """events: 8 torch.cuda.Event(enable_timing=True) (recorded once first) or None entries, or None."""
        if events is None:
            self._check(self.lib.verify_set_layer_events(self.ctx, None, 0))
            return
        arr = (C.c_void_p * 8)(*[None if e is None else e.cuda_event for e in events])
        self._check(self.lib.verify_set_layer_events(self.ctx, arr, 8))

    def tile(self, src, gate_up: bool = False, down: bool = False, stream=None) -> Tiled:
        """Tiled copy of a row-layout Q4Weight or Q4Experts (q4_tile): a new
        device buffer (torch uint8) and the struct describing it.  gate_up:
        an expert gate/up matrix; down: an expert down matrix; neither: a
        dense product's matrix."""
        import torch

        if gate_up and down:
            raise ValueError("a matrix is tiled as gate/up or as down, not both")
        kind = TILE_GATE_UP if gate_up else TILE_DOWN if down else TILE_DENSE
        experts = isinstance(src, Q4Experts)
        w, E = (src.w, src.n_experts) if experts else (src, 1)
        nbytes = int(self.lib.q4_tiled_bytes(w.n_out, w.k_in, E, kind))
        if nbytes < 0:
            raise VerifyError(EUNSUPPORTED, f"q4_tiled_bytes({w.n_out}, {w.k_in}, {E}, {kind}) rejected the shape")
        buf = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
        out = Q4Weight()
        self._check(self.lib.q4_tile(self.ctx, C.byref(w), E, kind, C.c_void_p(buf.data_ptr()), nbytes,
                                     C.byref(out), self._stream(stream)))
        return Tiled(buf, Q4Experts(out, E) if experts else out)

    def synth_q4(self, packed, scales, biases, seeds, scale_range, bias_range, centered=False, stream=None):
        self._check(self.lib.verify_synth_q4(self.ctx, _ptr(packed), _ptr(scales), _ptr(biases),
                                             packed.numel(), scales.numel(), *[C.c_uint64(s) for s in seeds],
                                             scale_range[0], scale_range[1], bias_range[0], bias_range[1],
                                             int(bool(centered)), self._stream(stream)))


def gdn_params(Hk, Hv, d, conv_w, A_log, dt_bias, norm_w, q_scale=None, l2_eps=1e-6, norm_eps=1e-6,
               gate_act=0) -> GdnParams:
    if q_scale is None:
        q_scale = d ** -0.5
    return GdnParams(Hk, Hv, d, d, 4, q_scale, l2_eps, norm_eps, gate_act, conv_w.data_ptr(), A_log.data_ptr(),
                     dt_bias.data_ptr(), norm_w.data_ptr())


def gdn_state(S_slots, conv_slots, cur=0) -> GdnState:
    st = GdnState()
    for s, (S, t) in enumerate(zip(S_slots, conv_slots)):
        st.S_slots[s] = S.data_ptr()
        st.conv_slots[s] = t.data_ptr()
    st.n_slots = len(S_slots)
    st.cur = cur
    st.pending_k = 0
    return st


def attn_params(Hq, Hkv, D, rope_dim=64, theta=1e7) -> AttnParams:
    return AttnParams(Hq, Hkv, D, rope_dim, theta)


def attn_workspace_bytes(params: AttnParams, capacity: int, split: int, max_k: int) -> int:
    return int(load().attn_workspace_bytes(C.byref(params), capacity, split, max_k))


def attn_default_split(capacity: int) -> int:
    return int(load().attn_default_split(capacity))


def kv_cache(K, V, work, length=0, split=256) -> KvCache:
    """K, V: int16 device tensors [Hkv, capacity, D] (binary16 bits); work: a
    device buffer of attn_workspace_bytes(...) bytes."""
    return KvCache(K.data_ptr(), V.data_ptr(), K.shape[1], length, split, 0, work.data_ptr(),
                   work.numel() * work.element_size())


def attn_inputs(q, gate, k, v) -> AttnInputs:
    """Row-major [rows, heads * D] (or [rows, heads, D]) bf16 tensors."""
    return AttnInputs(q.data_ptr(), q.stride(0), gate.data_ptr(), gate.stride(0), k.data_ptr(), k.stride(0),
                      v.data_ptr(), v.stride(0))


def gdn_inputs(qkv, z, a, b) -> GdnInputs:
    return GdnInputs(qkv.data_ptr(), qkv.stride(0), z.data_ptr(), z.stride(0), a.data_ptr(), a.stride(0),
                     b.data_ptr(), b.stride(0))
