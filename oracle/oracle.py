"""ctypes front end of the plain C oracle (oracle.c).

TEST INFRASTRUCTURE ONLY: used by the tests, the smoke check and the bench's
CPU baseline.  The product path (the CUDA library and its binding) never
imports this module, and this module imports nothing from the product.

The C file is compiled with gcc on first use (or by ``build()``), with
-ffp-contract=off so that no fused multiply-add changes its float64 rounding
between the x86 and Arm hosts.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "oracle.c")
LIB = os.path.join(HERE, "liboracle.so")
LIB_OMP = os.path.join(HERE, "liboracle_omp.so")  # the same source with -fopenmp, for timing only

_libs = {}
_threaded = False


def _compile(out, extra):
    if not os.path.exists(out) or os.path.getmtime(out) < os.path.getmtime(SRC):
        tmp = out + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", *extra,
                               "-o", tmp, SRC, "-lm"])
        os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    if force:
        for f in (LIB, LIB_OMP):
            if os.path.exists(f):
                os.remove(f)
    return _compile(LIB, [])


def build_threaded():
    """The OpenMP build (None if this host's gcc cannot build it)."""
    try:
        return _compile(LIB_OMP, ["-fopenmp"])
    except (subprocess.CalledProcessError, OSError):
        return None


def use_threads(on: bool) -> int:
    """Timing only: route every call below through the OpenMP build (on) or
    the plain single-threaded one; returns the threads the products use.
    Results are bit-identical either way."""
    global _threaded
    if on and build_threaded() is None:
        raise RuntimeError("the OpenMP build of the oracle is not available on this host")
    _threaded = bool(on)
    return int(lib().oracle_num_threads())


def lib():
    key = "omp" if _threaded else "plain"
    if key not in _libs:
        L = C.CDLL(build_threaded() if _threaded else build())
        p = C.c_void_p
        i, i64, d = C.c_int, C.c_int64, C.c_double
        L.oracle_q4_qmv.argtypes = [p, p, p, i, i, p, i64, i, p]
        L.oracle_route_topk.argtypes = [p, i64, i, i, i, p, p]
        L.oracle_gather_experts.argtypes = [p, p, p, p, p, p, i, i, i, p, i64, i, p, i, p, p, p,
                                            p, p, p, p, p, p, p, p]
        L.oracle_gdn_verify.argtypes = [i, i, i, i, i, d, d, d, i, p, p, p, p, p, p,
                                        p, i64, p, i64, p, i64, p, i64, i, p, p, p, p]
        L.oracle_rmsnorm.argtypes = [p, p, d, i, i, i, p]
        L.oracle_accept_greedy.argtypes = [p, i64, i, i, p, p]
        L.oracle_attn_verify.argtypes = [i, i, i, i, d, i, i, i64, p, p, p, p, p, p, p, p, p]
        L.oracle_round_f16.argtypes = [d]
        L.oracle_round_f16.restype = C.c_uint16
        L.oracle_round_bf16.argtypes = [d]
        L.oracle_round_bf16.restype = C.c_uint16
        L.oracle_num_threads.argtypes = []
        for f in ("oracle_q4_qmv", "oracle_route_topk", "oracle_gather_experts",
                  "oracle_gdn_verify", "oracle_rmsnorm", "oracle_accept_greedy", "oracle_attn_verify",
                  "oracle_num_threads"):
            getattr(L, f).restype = C.c_int
        _libs[key] = L
    return _libs[key]


def _ptr(a):
    return None if a is None else a.ctypes.data_as(C.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def _check(rc, name):
    if rc != 0:
        raise RuntimeError(f"{name} failed with code {rc}")


def round_bf16(v: float) -> int:
    return int(lib().oracle_round_bf16(float(v)))


def q4_qmv(packed, scales, biases, x) -> np.ndarray:
    """y[r, n] = sum_c (scale*q + bias)[n, c] * x[r, c]; x bf16 bits [k, K] -> float64 [k, N]."""
    packed, scales, biases = _c(packed, np.uint32), _c(scales, np.uint16), _c(biases, np.uint16)
    x = _c(np.atleast_2d(x), np.uint16)
    n_out, k_in = packed.shape[-2], packed.shape[-1] * 8
    k = x.shape[0]
    y = np.zeros((k, n_out), np.float64)
    _check(lib().oracle_q4_qmv(_ptr(packed), _ptr(scales), _ptr(biases), n_out, k_in,
                               _ptr(x), x.shape[1], k, _ptr(y)), "oracle_q4_qmv")
    return y


def route_topk(logits, T: int):
    logits = _c(np.atleast_2d(logits), np.float32)
    k, E = logits.shape
    idx = np.zeros((k, T), np.int32)
    w = np.zeros((k, T), np.float64)
    _check(lib().oracle_route_topk(_ptr(logits), E, k, E, T, _ptr(idx), _ptr(w)), "oracle_route_topk")
    return idx, w


def gather_experts(gate_up, down, logits, T: int, x, shared=None, shared_logit=None):
    """gate_up/down: (packed, scales, biases) stacks [E, 2I, H] / [E, H, I].
    shared: optional ((packed, scales, biases) of [2I, H], (...) of [H, I]) with
    shared_logit fp32 [k].  Returns idx [k,T], w [k,T], y float64 [k,H], h bf16 [k,T(+1),I]."""
    gp, gs, gb = (_c(gate_up[0], np.uint32), _c(gate_up[1], np.uint16), _c(gate_up[2], np.uint16))
    dp, ds, db = (_c(down[0], np.uint32), _c(down[1], np.uint16), _c(down[2], np.uint16))
    E, twoI, H8 = gp.shape
    I, H = twoI // 2, H8 * 8
    x = _c(np.atleast_2d(x), np.uint16)
    k = x.shape[0]
    logits = _c(np.atleast_2d(logits), np.float32)
    assert logits.shape == (k, E)
    slots = T + (1 if shared is not None else 0)
    idx = np.zeros((k, T), np.int32)
    w = np.zeros((k, T), np.float64)
    y = np.zeros((k, H), np.float64)
    h = np.zeros((k, slots, I), np.uint16)
    sg = [None] * 6
    sl = None
    if shared is not None:
        (sgp, sgs, sgb), (sdp, sds, sdb) = shared
        sg = [_c(sgp, np.uint32), _c(sgs, np.uint16), _c(sgb, np.uint16),
              _c(sdp, np.uint32), _c(sds, np.uint16), _c(sdb, np.uint16)]
        # the C side reads shared_logit[r * ld] with ld = E: lay it out that way
        sl = np.zeros((k, E), np.float32)
        sl[:, 0] = np.asarray(shared_logit, np.float32).reshape(k)
    _check(lib().oracle_gather_experts(_ptr(gp), _ptr(gs), _ptr(gb), _ptr(dp), _ptr(ds), _ptr(db),
                                       E, H, I, _ptr(logits), E, T, _ptr(x), k, _ptr(idx), _ptr(w),
                                       _ptr(y), *[_ptr(a) for a in sg], _ptr(sl), _ptr(h)),
           "oracle_gather_experts")
    return idx, w, y, h


def gdn_verify(Hk, Hv, d, params, S0, tail0, inputs, k, W=4, q_scale=None, l2_eps=1e-6,
               norm_eps=1e-6, gate_act=0, debug=False):
    """Returns o float64 [k, Hv*d], S_snap float64 [k, Hv, d, d], tail_snap bf16 [k, W-1, C]
    and, with debug=True, a dict of per-row intermediates."""
    if q_scale is None:
        q_scale = 1.0 / np.sqrt(d)
    C = 2 * Hk * d + Hv * d
    conv_w, A_log = _c(params["conv_w"], np.float32), _c(params["A_log"], np.float32)
    dt_bias, norm_w = _c(params["dt_bias"], np.float32), _c(params["norm_w"], np.float32)
    S0 = _c(S0, np.float64)
    tail0 = _c(tail0, np.uint16)
    qkv, z = _c(inputs["qkv"], np.uint16), _c(inputs["z"], np.uint16)
    a, b = _c(inputs["a"], np.uint16), _c(inputs["b"], np.uint16)
    o = np.zeros((k, Hv * d), np.float64)
    S_snap = np.zeros((k, Hv, d, d), np.float64)
    tail_snap = np.zeros((k, W - 1, C), np.uint16)
    per_row = 2 * Hk * d + 2 * Hv * d + 2 * Hv
    dbg = np.zeros((k, per_row), np.float64) if debug else None
    _check(lib().oracle_gdn_verify(Hk, Hv, d, d, W, float(q_scale), float(l2_eps), float(norm_eps),
                                   int(gate_act), _ptr(conv_w), _ptr(A_log), _ptr(dt_bias),
                                   _ptr(norm_w), _ptr(S0), _ptr(tail0),
                                   _ptr(qkv), qkv.shape[1], _ptr(z), z.shape[1], _ptr(a), a.shape[1],
                                   _ptr(b), b.shape[1], k, _ptr(o), _ptr(S_snap), _ptr(tail_snap),
                                   _ptr(dbg)), "oracle_gdn_verify")
    if not debug:
        return o, S_snap, tail_snap
    o1, o2, o3, o4, o5 = Hk * d, 2 * Hk * d, 2 * Hk * d + Hv * d, 2 * Hk * d + Hv * d + Hv, \
        2 * Hk * d + Hv * d + 2 * Hv
    info = dict(q=dbg[:, :o1].reshape(k, Hk, d), k=dbg[:, o1:o2].reshape(k, Hk, d),
                v=dbg[:, o2:o3].reshape(k, Hv, d), g=dbg[:, o3:o4], beta=dbg[:, o4:o5],
                y=dbg[:, o5:].reshape(k, Hv, d))
    return o, S_snap, tail_snap, info


def rmsnorm(x, w, eps=1e-6, zero_centered=True):
    x = _c(np.atleast_2d(x), np.float64)
    w = _c(w, np.float32)
    k, n = x.shape
    out = np.zeros_like(x)
    _check(lib().oracle_rmsnorm(_ptr(x), _ptr(w), float(eps), int(bool(zero_centered)), n, k, _ptr(out)),
           "oracle_rmsnorm")
    return out


def accept_greedy(logits, draft):
    """Greedy acceptance of a verify block: logits fp32 [k, V] (row 0 the
    pending token's, rows 1..k-1 the drafts'), draft int32 [k-1].
    Returns (a, next_token, t) with t the k greedy choices."""
    logits = _c(np.atleast_2d(logits), np.float32)
    k, V = logits.shape
    draft = _c(np.asarray(draft).reshape(-1), np.int32)
    if draft.size != k - 1:
        raise ValueError("draft must hold k - 1 tokens")
    out = np.zeros(2 + k, np.int32)
    _check(lib().oracle_accept_greedy(_ptr(logits), V, V, k, _ptr(draft) if k > 1 else None, _ptr(out)),
           "oracle_accept_greedy")
    return int(out[0]), int(out[1]), out[2:].copy()


def round_f16(v: float) -> int:
    return int(lib().oracle_round_f16(float(v)))


def attn_verify(Hq, Hkv, D, P, q, kn, vn, gate, Kc, Vc, rope_dim=64, theta=1e7):
    """Width-k attention verify over a binary16 KV cache.  q, gate: bf16 bits
    [k, Hq, D]; kn, vn: bf16 bits [k, Hkv, D]; Kc, Vc: binary16 bits
    [Hkv, cap, D] (positions 0..P-1 valid).  Returns o float64 [k, Hq, D] and
    the appended rows k_app, v_app (binary16 bits [k, Hkv, D])."""
    q, gate = _c(q, np.uint16), _c(gate, np.uint16)
    kn, vn = _c(kn, np.uint16), _c(vn, np.uint16)
    Kc, Vc = _c(Kc, np.uint16), _c(Vc, np.uint16)
    k = q.shape[0]
    cap = Kc.shape[1]
    o = np.zeros((k, Hq, D), np.float64)
    k_app = np.zeros((k, Hkv, D), np.uint16)
    v_app = np.zeros((k, Hkv, D), np.uint16)
    _check(lib().oracle_attn_verify(Hq, Hkv, D, rope_dim, float(theta), P, k, cap, _ptr(q), _ptr(kn), _ptr(vn),
                                    _ptr(gate), _ptr(Kc), _ptr(Vc), _ptr(o), _ptr(k_app), _ptr(v_app)),
           "oracle_attn_verify")
    return o, k_app, v_app


def to_bf16(v) -> np.ndarray:
    """Round float64 values to bf16 bit patterns (nearest-even), element by element."""
    v = np.asarray(v, np.float64)
    f = lib().oracle_round_bf16
    return np.array([f(float(t)) for t in v.ravel()], np.uint16).reshape(v.shape)


def stack_layer(w, h, S0, tail0, k, Hk, Hv, d, T, eps=1e-6):
    """One hybrid verify layer on the oracle, composed of the pinned pieces
    above in the order the layer defines ("QWEN38FLASH.md - Plan for
    supporting Qwen/Qwen3.8-Flash-Next", section 2: a Gated DeltaNet mixer,
    then a MoE with 10 routed + 1 shared expert; 2.4: zero-centred norms):

      xn = bf16(rmsnorm_zc(h));  p = bf16(in_proj . xn) = q|k|v, z, a, b
      o = bf16(gdn_verify(p));   h += out_proj . o
      xn2 = bf16(rmsnorm_zc(h)); l = fp32(router . xn2)   (E logits, then the shared gate)
      h += routed experts (top-T of l[:, :E]) + sigmoid(l[:, E]) * shared(xn2)

    READING: every activation that feeds a Q4 product is rounded to bf16 (the
    products take BF16 rows, "Flash-Next optimization transfer to Ornith and
    Qwen 27B", table "Shared architecture"), the residual stream h stays in
    the accumulation precision, router logits are fp32 (the routing input).

    w: provider with .in_proj/.out_proj/.router/.shared_gate_up/.shared_down
    as (packed, scales, biases), .gdn (params dict), .norm1/.norm2 (fp32) and
    .expert(e) -> ((gate_up packed, scales, biases), (down packed, scales, biases)).
    h: float64 [k, H].  Returns (h_out, S_snap, tail_snap, idx, logits).
    The routed sum uses only the selected experts: top-T of the full logits,
    then the same gather on the compacted stack of the distinct selected
    experts (same indices, weights and order as on the full stack).
    """
    H = h.shape[1]
    C = 2 * Hk * d + Hv * d
    Z = Hv * d
    xn = to_bf16(rmsnorm(h, w.norm1, eps, True))
    p = to_bf16(q4_qmv(*w.in_proj, xn))
    inp = dict(qkv=p[:, :C], z=p[:, C:C + Z], a=p[:, C + Z:C + Z + Hv], b=p[:, C + Z + Hv:C + Z + 2 * Hv])
    o, S_snap, tail_snap = gdn_verify(Hk, Hv, d, w.gdn, S0, tail0, inp, k)
    h = h + q4_qmv(*w.out_proj, to_bf16(o))
    xn2 = to_bf16(rmsnorm(h, w.norm2, eps, True))
    lg = q4_qmv(*w.router, xn2).astype(np.float32)
    E = lg.shape[1] - 1
    idx, _ = route_topk(lg[:, :E], T)
    U = np.unique(idx)
    ex = [w.expert(int(e)) for e in U]
    gu = tuple(np.stack([x[0][i] for x in ex]) for i in range(3))
    dn = tuple(np.stack([x[1][i] for x in ex]) for i in range(3))
    idx_c, _, y, _ = gather_experts(gu, dn, np.ascontiguousarray(lg[:, U]), T, xn2,
                                    shared=(w.shared_gate_up, w.shared_down), shared_logit=lg[:, E])
    assert np.array_equal(U[idx_c], idx)
    return h + y, S_snap, tail_snap, idx, lg
