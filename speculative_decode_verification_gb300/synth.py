"""Seeded synthetic inputs for the verify workloads.

This module only draws numbers.  It holds none of the verification arithmetic,
so both the CPU oracle side and the GPU side can take their inputs from it.

Generator: SplitMix64 (Steele, Lea, Flood, "Fast splittable pseudorandom
number generators", OOPSLA 2014; the finaliser constants are Vigna's).  It is
counter based: element i of a tensor is the i-th output of the SplitMix64
sequence started at that tensor's seed, i.e.  mix64(tseed + (i+1)*GAMMA).
Any element can be drawn on its own, so a device-side twin of the same
definition (``verify_synth_q4`` in the library) can fill multi-GB weight
tensors on the GPU and the host can still re-draw any sampled row bit for bit.

Value recipes (the shapes and distributions of the pages' workloads):
  * Q4 codes: the low 32 bits of each draw are one packed word, i.e. eight
    independent uniform codes 0..15.
  * uniform(lo, hi): u = (draw >> 40) * 2**-24 (exact in fp32), then
    v = fl32(fl32((hi - lo) * u) + lo), every step an fp32 IEEE operation.
  * normal(mean, std): Box-Muller in float64 from one draw, u1 = (hi32 + 1) *
    2**-32, u2 = lo32 * 2**-32, z = sqrt(-2 ln u1) cos(2 pi u2).  Host only.
  * bf16 tensors are drawn in fp32 and rounded to nearest-even on the host.
"""
from __future__ import annotations

import numpy as np

GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_MASK64 = (1 << 64) - 1


def _mix64_int(z: int) -> int:
    z &= _MASK64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _MASK64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _MASK64
    return z ^ (z >> 31)


def fnv1a64(name: str) -> int:
    h = 0xCBF29CE484222325
    for byte in name.encode():
        h ^= byte
        h = (h * 0x100000001B3) & _MASK64
    return h


def tensor_seed(seed: int, name: str) -> int:
    """Seed of one named tensor: mix64(fnv1a64(name) + seed*GAMMA)."""
    return _mix64_int(fnv1a64(name) + (seed * 0x9E3779B97F4A7C15))


def draws(tseed: int, start: int, count: int) -> np.ndarray:
    """uint64 draws start .. start+count-1 of the sequence seeded by tseed."""
    with np.errstate(over="ignore"):
        i = np.arange(start + 1, start + count + 1, dtype=np.uint64)
        z = np.uint64(tseed) + i * GAMMA
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
        return z ^ (z >> np.uint64(31))


# ------------------------------------------------------------------ bf16 bits

def f32_to_bf16(a: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (nearest, ties to even); returns uint16 bit patterns."""
    a = np.asarray(a, dtype=np.float32)
    b = np.ascontiguousarray(a).view(np.uint32)
    rounding = np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1))
    return ((b + rounding) >> np.uint32(16)).astype(np.uint16).reshape(a.shape)


def bf16_to_f32(h: np.ndarray) -> np.ndarray:
    return (np.asarray(h, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


# ------------------------------------------------------------- value recipes

def uniform_f32(tseed: int, count: int, lo: float, hi: float, start: int = 0) -> np.ndarray:
    z = draws(tseed, start, count)
    u = (z >> np.uint64(40)).astype(np.float32) * np.float32(2.0 ** -24)
    span = np.float32(hi) - np.float32(lo)
    return (span * u).astype(np.float32) + np.float32(lo)


def normal_f32(tseed: int, count: int, mean: float = 0.0, std: float = 1.0, start: int = 0) -> np.ndarray:
    z = draws(tseed, start, count)
    u1 = ((z >> np.uint64(32)).astype(np.float64) + 1.0) * 2.0 ** -32
    u2 = (z & np.uint64(0xFFFFFFFF)).astype(np.float64) * 2.0 ** -32
    n = np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2)
    return (mean + std * n).astype(np.float32)


def packed_words(tseed: int, count: int, start: int = 0) -> np.ndarray:
    return (draws(tseed, start, count) & np.uint64(0xFFFFFFFF)).astype(np.uint32)


# ----------------------------------------------------------- named tensors

SCALE_RANGE = (0.005, 0.02)
BIAS_RANGE = (-0.1, 0.1)


class Q4Matrix:
    """Host copy of one (or a stack of) affine Q4/g64 matrices.

    packed uint32 [E, N, K/8], scales/biases bf16 bits [E, N, K/64]; E = 1 for
    a dense matrix (then the arrays are 2-D).
    """

    def __init__(self, packed, scales, biases, n_out, k_in, n_experts=None):
        self.packed, self.scales, self.biases = packed, scales, biases
        self.n_out, self.k_in, self.n_experts = n_out, k_in, n_experts


def q4_seeds(seed: int, name: str):
    return (tensor_seed(seed, name + ".packed"), tensor_seed(seed, name + ".scales"),
            tensor_seed(seed, name + ".biases"))


# Centred recipe (the verify stack): bias = -scale * U(7, 8), i.e. the affine
# form of a roughly zero-mean weight group, so that projections are not
# dominated by a common offset and different rows route to different experts.
CENTERED_RANGE = (7.0, 8.0)


def q4_biases(sb: int, count: int, scales_bf16: np.ndarray, bias_range, centered: bool, start: int = 0):
    u = uniform_f32(sb, count, *bias_range, start=start)
    if not centered:
        return f32_to_bf16(u)
    return f32_to_bf16(-(bf16_to_f32(scales_bf16) * u).astype(np.float32))


def q4_matrix(seed: int, name: str, n_out: int, k_in: int, n_experts: int | None = None,
              scale_range=SCALE_RANGE, bias_range=BIAS_RANGE, centered: bool = False) -> Q4Matrix:
    """Random-init affine Q4/g64 weights: codes U{0..15}, scales U(0.005,0.02),
    biases U(-0.1,0.1) (or, centered, -scale * U(7, 8)), scales/biases bf16."""
    assert k_in % 64 == 0
    if centered:
        bias_range = CENTERED_RANGE
    e = 1 if n_experts is None else n_experts
    sp, ss, sb = q4_seeds(seed, name)
    nw, ng = n_out * (k_in // 8), n_out * (k_in // 64)
    packed = packed_words(sp, e * nw)
    scales = f32_to_bf16(uniform_f32(ss, e * ng, *scale_range))
    biases = q4_biases(sb, e * ng, scales, bias_range, centered)
    if n_experts is None:
        shape_w, shape_g = (n_out, k_in // 8), (n_out, k_in // 64)
    else:
        shape_w, shape_g = (e, n_out, k_in // 8), (e, n_out, k_in // 64)
    return Q4Matrix(packed.reshape(shape_w), scales.reshape(shape_g), biases.reshape(shape_g),
                    n_out, k_in, n_experts)


def q4_rows(seed: int, name: str, n_out: int, k_in: int, rows, expert: int = 0,
            scale_range=SCALE_RANGE, bias_range=BIAS_RANGE, centered: bool = False) -> Q4Matrix:
    """Re-draw only the given rows (of one expert) of a q4_matrix tensor.
    Bit-identical to slicing q4_matrix(...) but costs O(len(rows) * k_in)."""
    if centered:
        bias_range = CENTERED_RANGE
    sp, ss, sb = q4_seeds(seed, name)
    wpr, gpr = k_in // 8, k_in // 64
    rows = np.asarray(rows, dtype=np.int64)
    packed = np.empty((len(rows), wpr), np.uint32)
    scales = np.empty((len(rows), gpr), np.uint16)
    biases = np.empty((len(rows), gpr), np.uint16)
    for i, n in enumerate(rows):
        base = expert * n_out + int(n)
        packed[i] = packed_words(sp, wpr, start=base * wpr)
        scales[i] = f32_to_bf16(uniform_f32(ss, gpr, *scale_range, start=base * gpr))
        biases[i] = q4_biases(sb, gpr, scales[i], bias_range, centered, start=base * gpr)
    return Q4Matrix(packed, scales, biases, len(rows), k_in)


def q4_expert(seed: int, name: str, n_out: int, k_in: int, expert: int,
              scale_range=SCALE_RANGE, bias_range=BIAS_RANGE, centered: bool = False) -> Q4Matrix:
    """Re-draw one whole expert matrix of a q4_matrix(..., n_experts=E) stack."""
    if centered:
        bias_range = CENTERED_RANGE
    sp, ss, sb = q4_seeds(seed, name)
    wpr, gpr = k_in // 8, k_in // 64
    packed = packed_words(sp, n_out * wpr, start=expert * n_out * wpr)
    scales = f32_to_bf16(uniform_f32(ss, n_out * gpr, *scale_range, start=expert * n_out * gpr))
    biases = q4_biases(sb, n_out * gpr, scales, bias_range, centered, start=expert * n_out * gpr)
    return Q4Matrix(packed.reshape(n_out, wpr), scales.reshape(n_out, gpr), biases.reshape(n_out, gpr),
                    n_out, k_in)


def bf16_normal(seed: int, name: str, shape, mean=0.0, std=1.0) -> np.ndarray:
    n = int(np.prod(shape))
    return f32_to_bf16(normal_f32(tensor_seed(seed, name), n, mean, std)).reshape(shape)


def f32_normal(seed: int, name: str, shape, mean=0.0, std=1.0) -> np.ndarray:
    n = int(np.prod(shape))
    return normal_f32(tensor_seed(seed, name), n, mean, std).reshape(shape)


def f16_normal(seed: int, name: str, shape, mean=0.0, std=1.0) -> np.ndarray:
    """N(mean, std) rounded to IEEE binary16 (nearest-even), as bit patterns."""
    n = int(np.prod(shape))
    return normal_f32(tensor_seed(seed, name), n, mean, std).astype(np.float16).view(np.uint16).reshape(shape)


def f32_uniform(seed: int, name: str, shape, lo, hi) -> np.ndarray:
    n = int(np.prod(shape))
    return uniform_f32(tensor_seed(seed, name), n, lo, hi).reshape(shape)


# ------------------------------------------------------- workload shapes

# Dense projections of the Qwen-27B-shaped workload (hidden 5120, FFN 17408).
DENSE_SHAPES = [(5120, 5120), (17408, 5120), (5120, 17408)]  # (n_out, k_in)
DENSE_WIDTHS = [1, 4, 8, 9]

# Ornith-shaped routed MoE.
ORNITH_MOE = dict(E=256, T=8, H=2048, I=512)

# Flash-Next-shaped Gated DeltaNet layer.
FLASH_GDN = dict(n_qk_heads=16, n_v_heads=48, d=128, conv_kernel=4)

# 12-layer verify stack at hidden 2560 (GDN mixer + 512-expert MoE per layer).
STACK = dict(layers=12, H=2560, E=512, T=10, I=640, n_qk_heads=16, n_v_heads=48, d=128,
             conv_kernel=4)

# Flash-Next vocabulary (padded): the width of the target's logits per row,
# and the Q4 LM head that makes them from the hidden-2560 rows (n_out, k_in).
FLASH_VOCAB = 248_320
LM_HEAD = (FLASH_VOCAB, 2560)


def vocab_logits(seed: int, name: str, k: int, V: int, levels: int = 0) -> np.ndarray:
    """Target logits fp32 [k, V] ~ N(0, 1); with levels > 0 rounded to
    multiples of 1/levels, so that equal maxima occur."""
    x = f32_normal(seed, name, (k, V))
    if levels > 0:
        x = (np.round(x.astype(np.float64) * levels) / levels).astype(np.float32)
    return x


# Flash-Next-shaped attention layer (QSA below its sparse budget = dense GQA):
# 24 query heads, 2 KV heads, head dim 256, RoPE on the first 64 dims, base 1e7.
FLASH_ATTN = dict(n_q_heads=24, n_kv_heads=2, d=256, rope_dim=64, theta=1e7)


def attn_inputs(seed: int, prefix: str, k: int, Hq: int, Hkv: int, D: int):
    """The block's query, gate, key and value rows (bf16 bits): q and k with
    entries ~ N(0, 1) (unit-rms rows, as after the per-head norms), v and the
    gate ~ N(0, 1)."""
    return dict(q=bf16_normal(seed, prefix + ".q", (k, Hq, D)), gate=bf16_normal(seed, prefix + ".gate", (k, Hq, D)),
                k=bf16_normal(seed, prefix + ".k", (k, Hkv, D)), v=bf16_normal(seed, prefix + ".v", (k, Hkv, D)))


def attn_cache(seed: int, prefix: str, Hkv: int, cap: int, D: int, P: int):
    """A KV cache of capacity cap with P valid positions (binary16 bits
    [Hkv, cap, D], N(0, 1) keys and values; positions from P on zero).  Long
    caches are drawn from numpy's PCG64 stream seeded by the tensor name (the
    SplitMix64 Box-Muller stream is too slow for 10^8 values on the host)."""
    K = np.zeros((Hkv, cap, D), np.uint16)
    V = np.zeros((Hkv, cap, D), np.uint16)
    if P:
        if Hkv * P * D <= 1 << 20:
            K[:, :P] = f16_normal(seed, prefix + ".K", (Hkv, P, D))
            V[:, :P] = f16_normal(seed, prefix + ".V", (Hkv, P, D))
        else:
            for X, nm in ((K, ".K"), (V, ".V")):
                rng = np.random.default_rng(tensor_seed(seed, prefix + nm))
                X[:, :P] = rng.standard_normal((Hkv, P, D), dtype=np.float32).astype(np.float16).view(np.uint16)
    return K, V


# Tiny workload: one 512x512 projection and a 2/2-head, d=32 GDN step.
TINY_Q4 = (512, 512)
TINY_GDN = dict(n_qk_heads=2, n_v_heads=2, d=32, conv_kernel=4)


def gdn_params(seed: int, prefix: str, n_qk_heads: int, n_v_heads: int, d: int, conv_kernel: int = 4):
    """GDN parameters: conv_w U(-0.5,0.5), A_log U(-1,1), dt_bias U(-1,1),
    norm_w U(0.5,1.5), all fp32."""
    C = 2 * n_qk_heads * d + n_v_heads * d
    return dict(
        conv_w=f32_uniform(seed, prefix + ".conv_w", (C, conv_kernel), -0.5, 0.5),
        A_log=f32_uniform(seed, prefix + ".A_log", (n_v_heads,), -1.0, 1.0),
        dt_bias=f32_uniform(seed, prefix + ".dt_bias", (n_v_heads,), -1.0, 1.0),
        norm_w=f32_uniform(seed, prefix + ".norm_w", (d,), 0.5, 1.5),
    )


def gdn_inputs(seed: int, prefix: str, k: int, n_qk_heads: int, n_v_heads: int, d: int):
    """Per-row GDN inputs (bf16 bits): qkv [k, C], z [k, Hv*d], a, b [k, Hv], all N(0,1)."""
    C = 2 * n_qk_heads * d + n_v_heads * d
    return dict(
        qkv=bf16_normal(seed, prefix + ".qkv", (k, C)),
        z=bf16_normal(seed, prefix + ".z", (k, n_v_heads * d)),
        a=bf16_normal(seed, prefix + ".a", (k, n_v_heads)),
        b=bf16_normal(seed, prefix + ".b", (k, n_v_heads)),
    )


def gdn_initial_state(seed: int, prefix: str, n_qk_heads: int, n_v_heads: int, d: int,
                      conv_kernel: int = 4, s_std: float = 0.0, tail_std: float = 0.0):
    """Initial state: S fp32 [Hv, d, d] ~ N(0, s_std^2) (zeros if s_std == 0) and
    conv tail bf16 [conv_kernel-1, C] ~ N(0, tail_std^2) (zeros if 0)."""
    C = 2 * n_qk_heads * d + n_v_heads * d
    if s_std > 0:
        S = f32_normal(seed, prefix + ".S0", (n_v_heads, d, d), 0.0, s_std)
    else:
        S = np.zeros((n_v_heads, d, d), np.float32)
    if tail_std > 0:
        tail = bf16_normal(seed, prefix + ".tail0", (conv_kernel - 1, C), 0.0, tail_std)
    else:
        tail = np.zeros((conv_kernel - 1, C), np.uint16)
    return S, tail


class HostLayerWeights:
    """Host re-draw of one layer of the synthetic verify stack (the same named
    tensors the device stack draws): dense matrices eagerly, experts on demand."""

    def __init__(self, seed: int, l: int, H: int, NP: int, Z: int, E: int, I: int,
                 n_qk_heads: int, n_v_heads: int, d: int):
        p = f"stack.L{l}"
        self.seed, self.p, self.H, self.E, self.I = seed, p, H, E, I
        m = q4_matrix(seed, p + ".in_proj", NP, H, centered=True)
        self.in_proj = (m.packed, m.scales, m.biases)
        m = q4_matrix(seed, p + ".out_proj", H, Z, centered=True)
        self.out_proj = (m.packed, m.scales, m.biases)
        m = q4_matrix(seed, p + ".router", E + 1, H, centered=True)
        self.router = (m.packed, m.scales, m.biases)
        m = q4_matrix(seed, p + ".shared_gate_up", 2 * I, H, centered=True)
        self.shared_gate_up = (m.packed, m.scales, m.biases)
        m = q4_matrix(seed, p + ".shared_down", H, I, centered=True)
        self.shared_down = (m.packed, m.scales, m.biases)
        self.gdn = gdn_params(seed, p + ".gdn", n_qk_heads, n_v_heads, d)
        self.norm1 = f32_uniform(seed, p + ".norm1", (H,), -0.1, 0.1)
        self.norm2 = f32_uniform(seed, p + ".norm2", (H,), -0.1, 0.1)
        self._cache = {}

    def expert(self, e: int):
        if e not in self._cache:
            g = q4_expert(self.seed, self.p + ".gate_up", 2 * self.I, self.H, e, centered=True)
            dn = q4_expert(self.seed, self.p + ".down", self.H, self.I, e, centered=True)
            self._cache[e] = ((g.packed, g.scales, g.biases), (dn.packed, dn.scales, dn.biases))
        return self._cache[e]
