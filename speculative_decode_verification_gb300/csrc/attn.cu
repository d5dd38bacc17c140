// Width-k grouped-query attention over a binary16 KV cache ("QWEN38FLASH.md -
// Plan for supporting Qwen/Qwen3.8-Flash-Next" 2.2: 24 query and 2 KV heads of
// dim 256, partial RoPE, sigmoid output gate, F16 cache; "Red Lite dev45 -
// speculative decoding with the Qwen3-Next MTP block", "What it is": row r
// sees the earlier rows' keys and values).
//
// Three launches:
//  1. append: the block's keys (rotated at P + r) and values go into the
//     cache at P + r as binary16; the queries are rotated and scaled by
//     1/sqrt(D) and kept as binary16 pairs hi + lo.
//  2. partials: CTA (M tile, split s, KV head) takes 128 (row, query head)
//     pairs of that KV head's group and the key positions [s*split,
//     (s+1)*split) of the window, 64 at a time.  S = Q K^T and O += P V run on
//     the tcgen05 tensor cores with fp32 accumulators in tensor memory (the
//     query and the probabilities each as a binary16 pair hi + lo, two MMAs
//     against the same key or value tile, so that only the cache's own
//     binary16 rounding remains); each thread owns one pair's row of S and O,
//     masks positions after the pair's own (P + r) and keeps the running max
//     and sum.
//  3. combine: per (row, query head) the splits that hold the row's window are
//     merged in ascending order and gated.
// Launches 2 and 3 are programmatic dependents of the one before.
//
// Exactness: a row's arithmetic depends only on its own query, its window and
// the absolute cut of key positions (split and the 64-position sub-tiles), not
// on k or the other rows, so row r of a width-k call equals a width-1 call at
// P + r bit for bit.  Positions past a row's window add exact zeros, and
// splits past it are skipped.
//
// Bound: the cache read, 2 * Hkv * D * 2 bytes per position (2 KB at the
// Flash-Next shape), with 4 * k * Hq * D flops per key position (twice that
// on the tensor cores with the hi + lo pairs, and M padded to 128 pairs).
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "internal.h"

namespace vk {
namespace {

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

__device__ __forceinline__ uint32_t pack_half2(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }

// ---------------------------------------------------------------- append
// x rotated at pos on its first rope_dim entries, entry e.  The angle
// pos * inv_freq[j] is formed and reduced modulo 2 pi in float64 (two float64
// operations: the device's float64 rate is low), then sin and cos of the
// reduced angle in fp32, the rotation in float64.
__device__ __forceinline__ double rope_entry(const uint16_t* x, int e, int rope_dim, const double* inv_freq,
                                             long long pos) {
  const int half = rope_dim / 2;
  double y = (double)bf16f(x[e]);
  if (e < rope_dim) {
    const int j = e < half ? e : e - half;
    constexpr double kTwoPi = 6.283185307179586;
    const double ang = (double)pos * inv_freq[j];
    const float red = (float)fma(-kTwoPi, rint(ang * (1.0 / kTwoPi)), ang);
    float sn, cs;
    sincosf(red, &sn, &cs);
    y = e < half ? y * cs - (double)bf16f(x[e + half]) * sn : y * cs + (double)bf16f(x[e - half]) * sn;
  }
  return y;
}

// CTA (r, h): h < Hkv appends KV head h's key and value of row r to the cache;
// h >= Hkv rotates and scales query head h - Hkv of row r into its binary16
// pair (hi, lo).
__global__ void attn_append_kernel(const AttnArgs a) {
  griddep_launch();  // the split kernel may start its prefetch of committed positions
  const int r = blockIdx.x, h = blockIdx.y;
  const long long pos = (long long)a.P + r;
  if (h < a.Hkv) {
    const uint16_t* kr = a.kin + (long long)r * a.ld_k + (long long)h * a.D;
    const uint16_t* vr = a.vin + (long long)r * a.ld_v + (long long)h * a.D;
    for (int e = threadIdx.x; e < a.D; e += blockDim.x) {
      const long long dst = ((long long)h * a.cap + pos) * a.D + e;
      a.K[dst] = __half_as_ushort(__double2half(rope_entry(kr, e, a.rope_dim, a.inv_freq, pos)));
      a.V[dst] = __half_as_ushort(__float2half_rn(bf16f(vr[e])));
    }
    return;
  }
  const int hq = h - a.Hkv;
  const uint16_t* qr = a.q + (long long)r * a.ld_q + (long long)hq * a.D;
  const double scale = 1.0 / sqrt((double)a.D);
  for (int e = threadIdx.x; e < a.D; e += blockDim.x) {
    const double y = rope_entry(qr, e, a.rope_dim, a.inv_freq, pos) * scale;
    const __half hi = __double2half(y);
    const long long dst = ((long long)r * a.Hq + hq) * a.D + e;
    a.qh[dst] = __half_as_ushort(hi);
    a.ql[dst] = __half_as_ushort(__double2half(y - (double)__half2float(hi)));
  }
}

// ---------------------------------------------------------------- partials
// CTA (M tile, split s, KV head): the 128 (row, query head) pairs m0 .. m0+127
// of that KV head's group against the key positions [s*split, (s+1)*split),
// 64 at a time.  Thread t holds pair m0 + t: TMEM lane t.
//   S = Q K^T   tcgen05, M 128 x N 64, K = D in steps of 16: the query's
//               binary16 hi part, then its lo part, into one fp32 TMEM tile;
//   softmax     each thread reads its row of S from TMEM, masks positions
//               after its own (P + r), keeps the running max and sum, and
//               writes p as binary16 hi and lo parts to shared memory;
//   O += P V    tcgen05, M 128 x N D, K = 64 in steps of 16 (V MN-major),
//               O an fp32 TMEM tile, rescaled by exp(m_old - m_new) in place
//               (tcgen05.ld / st) when a row's max rises.
// Operands are in the canonical no-swizzle layouts (core matrices of 8 rows x
// 16 B): Q, K and P K-major, V MN-major, filled with 16-byte cp.async or
// stores.  Each load of the next key or value tile is issued as soon as the
// MMA that read the previous one has completed.  One CTA per SM (about
// 224 KB of shared memory at D = 256).
constexpr int kTcM = 128;        // pairs per CTA (TMEM lanes)
constexpr int kTcN = 64;         // key positions per sub-tile
constexpr int kTcThreads = 128;  // thread t <-> TMEM lane t

template <int D>
struct TcSmem {
  static constexpr int Q_BYTES = kTcM * D * 2;    // one of the query's hi / lo parts
  static constexpr int KV_BYTES = kTcN * D * 2;
  static constexpr int P_BYTES = kTcM * kTcN * 2;  // one of p's hi / lo parts
  static constexpr int QH = 0, QL = Q_BYTES, K = 2 * Q_BYTES, V = K + KV_BYTES, PH = V + KV_BYTES,
                       PL = PH + P_BYTES;
  static constexpr int BYTES = PL + P_BYTES;
  static constexpr uint32_t TMEM_COLS = D > 128 ? 512 : 256;  // S at column 0, O at O_COL
  static constexpr uint32_t O_COL = D > 128 ? 256 : 128;
};

// Byte offset of element (row, kidx) of a K-major operand with R rows:
// per k-step of 16, [row / 8][k half][row % 8][8 elements].
template <int R>
__device__ __forceinline__ uint32_t kmajor_off(int row, int kidx) {
  return (uint32_t)((kidx >> 4) * (R * 32) + (row >> 3) * 256 + ((kidx >> 3) & 1) * 128 + (row & 7) * 16 +
                    (kidx & 7) * 2);
}
// Byte offset of value (key, d) in the MN-major value tile: [key / 8][d / 8][key % 8][8 d].
template <int D>
__device__ __forceinline__ uint32_t vmajor_off(int key, int d) {
  return (uint32_t)(((key >> 3) * (D / 8) + (d >> 3)) * 128 + (key & 7) * 16 + (d & 7) * 2);
}

template <int D>
__global__ void __launch_bounds__(kTcThreads, 1) attn_partial_kernel(const AttnArgs a) {
  using L = TcSmem<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
  __shared__ __align__(8) uint64_t bars[2];  // S tile done, O tile done
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;
  volatile int* abort = &abort_flag;
  const uint32_t sb = smem_addr(smem);
  const uint32_t bar_s = smem_addr(&bars[0]), bar_o = smem_addr(&bars[1]);

  const int tid = threadIdx.x, warp = tid >> 5;
  const int s = blockIdx.y, hk = blockIdx.z;
  const int G = a.Hq / a.Hkv, M = a.k * G, Mpad = 16 * a.n_mtiles;
  const int m0 = blockIdx.x * kTcM;
  const int end = a.P + a.k;  // positions held by the cache after the append
  const int pos0 = s * a.split;
  const int pos_end = min(pos0 + a.split, end);
  const int nsub = (pos_end - pos0 + kTcN - 1) / kTcN;

  // keys and values of sub-tile `sub` (zero fill past the cache's end)
  auto load_kv = [&](int sub, bool values) {
    constexpr int CH = kTcN * (D / 8);
    for (int q = tid; q < CH; q += kTcThreads) {
      const int row = q / (D / 8), d0 = (q % (D / 8)) * 8;
      const int pos = pos0 + sub * kTcN + row;
      const bool ok = pos < end;
      const uint16_t* src = (values ? a.V : a.K) + ((long long)hk * a.cap + (ok ? pos : 0)) * D + d0;
      const uint32_t dst = values ? sb + L::V + vmajor_off<D>(row, d0) : sb + L::K + kmajor_off<kTcN>(row, d0);
      cp_async16(dst, src, ok ? 16u : 0u);
    }
    cp_async_commit();
  };

  if (tid == 0) {
    abort_flag = 0;
    mbar_init(bar_s, 1);
    mbar_init(bar_o, 1);
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(smem_addr(&tmem_slot), L::TMEM_COLS);
  // Launched as a programmatic dependent of the append kernel: a first
  // sub-tile of positions committed before this call (written at least two
  // launches back) is fetched before the dependency wait; the queries and the
  // block's own keys and values after it.
  const bool early = pos0 + kTcN <= a.P;
  if (early) {
    load_kv(0, false);
    load_kv(0, true);
  }
  griddep_wait();
  griddep_launch();
  // the queries of this CTA's 128 pairs, rotated at P + r and scaled by
  // 1/sqrt(D) by the append kernel: binary16 hi and lo parts (zeros past M)
  {
    constexpr int QCH = kTcM * (D / 8);
    for (int q = tid; q < 2 * QCH; q += kTcThreads) {
      const int part = q / QCH, cc = q % QCH;
      const int mm = cc / (D / 8), d0 = (cc % (D / 8)) * 8, m = m0 + mm;
      const bool ok = m < M;
      const long long row = ok ? (long long)(m / G) * a.Hq + hk * G + m % G : 0;
      cp_async16(sb + (part ? L::QL : L::QH) + kmajor_off<kTcM>(mm, d0), (part ? a.ql : a.qh) + row * D + d0,
                 ok ? 16u : 0u);
    }
    cp_async_commit();
  }
  if (!early) {
    load_kv(0, false);
    load_kv(0, true);
  }
  cp_async_wait<0>();
  fence_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  const uint32_t t_s = tmem + ((uint32_t)(32 * warp) << 16);  // this warp's lanes of S
  const uint32_t t_o = t_s + L::O_COL;                        // and of O
  const int m = m0 + tid;
  // last position this pair sees in this split (-1: none): its own window, and
  // no further than the split's end (a split need not be a multiple of 64)
  const int lim = m < M ? min(a.P + m / G, pos_end - 1) : -1;
  float m_run = -INFINITY, l_run = 0.f;
  constexpr uint32_t IDESC_S = umma_idesc_f16(kTcM, kTcN, false);
  constexpr uint32_t IDESC_O = umma_idesc_f16(kTcM, D, true);

  for (int sub = 0; sub < nsub; ++sub) {
    const uint32_t ph = (uint32_t)(sub & 1);
    // S = Q_hi K^T + Q_lo K^T
    if (tid == 0) {
      tc_fence_after();
#pragma unroll 1
      for (int part = 0; part < 2; ++part)
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks)
          umma_f16(tmem, umma_desc(sb + (part ? L::QL : L::QH) + ks * kTcM * 32, 128, 256),
                   umma_desc(sb + L::K + ks * kTcN * 32, 128, 256), IDESC_S, (part | ks) ? 1u : 0u);
      umma_commit(bar_s);
    }
    const bool ok_s = mbar_wait(bar_s, ph, abort, a.err);
    tc_fence_after();
    // the key tile is free: fetch the next one while this one's softmax and P V run
    if (sub + 1 < nsub) load_kv(sub + 1, false);
    // this pair's row of S; mask, running max and sum
    float sv[kTcN];
#pragma unroll
    for (int c0 = 0; c0 < kTcN; c0 += 32) {
      uint32_t v[32];
      tmem_ld32(t_s + (uint32_t)c0, v);
      tmem_ld_wait();
#pragma unroll
      for (int j = 0; j < 32; ++j) sv[c0 + j] = __uint_as_float(v[j]);
    }
    const int pbase = pos0 + sub * kTcN;
    float mx = -INFINITY;
#pragma unroll
    for (int j = 0; j < kTcN; ++j) {
      sv[j] = pbase + j <= lim ? sv[j] : -INFINITY;
      mx = fmaxf(mx, sv[j]);
    }
    const float mn = fmaxf(m_run, mx);
    const float alpha = mn == -INFINITY ? 1.f : expf(m_run - mn);
    const float msub = mn == -INFINITY ? 0.f : mn;
    m_run = mn;
    float ps = 0.f;
#pragma unroll
    for (int j0 = 0; j0 < kTcN; j0 += 8) {
      uint32_t hi[4], lo[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float p0 = expf(sv[j0 + 2 * e] - msub), p1 = expf(sv[j0 + 2 * e + 1] - msub);
        const __half2 h2 = __floats2half2_rn(p0, p1);
        hi[e] = pack_half2(h2);
        lo[e] = pack_half2(__floats2half2_rn(p0 - __low2float(h2), p1 - __high2float(h2)));
        ps += p0;
        ps += p1;
      }
      const uint32_t off = kmajor_off<kTcM>(tid, j0);
      asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(sb + L::PH + off), "r"(hi[0]), "r"(hi[1]),
                   "r"(hi[2]), "r"(hi[3])
                   : "memory");
      asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(sb + L::PL + off), "r"(lo[0]), "r"(lo[1]),
                   "r"(lo[2]), "r"(lo[3])
                   : "memory");
    }
    l_run = fmaf(l_run, alpha, ps);
    // O *= alpha for this pair (the whole warp when any of its rows changed)
    if (sub > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
      for (int c0 = 0; c0 < D; c0 += 32) {
        uint32_t v[32];
        tmem_ld32(t_o + (uint32_t)c0, v);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = __float_as_uint(__uint_as_float(v[j]) * alpha);
        tmem_st32(t_o + (uint32_t)c0, v);
      }
      tmem_st_wait();
    }
    // this sub-tile's values landed (the next key tile may still be in flight)
    if (sub + 1 < nsub) cp_async_wait<1>();
    else cp_async_wait<0>();
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    // O += P_hi V + P_lo V
    if (tid == 0 && ok_s) {
      tc_fence_after();
#pragma unroll 1
      for (int part = 0; part < 2; ++part)
#pragma unroll
        for (int ks = 0; ks < kTcN / 16; ++ks)
          umma_f16(tmem + L::O_COL, umma_desc(sb + (part ? L::PL : L::PH) + ks * kTcM * 32, 128, 256),
                   umma_desc(sb + L::V + 2 * ks * (D / 8) * 128, (D / 8) * 128, 128), IDESC_O,
                   (sub | part | ks) ? 1u : 0u);
      umma_commit(bar_o);
    } else if (tid == 0) {
      umma_commit(bar_o);  // nothing issued: the barrier still completes
    }
    mbar_wait(bar_o, ph, abort, a.err);
    tc_fence_after();
    // the value tile is free: fetch the next one
    if (sub + 1 < nsub) {
      load_kv(sub + 1, true);
      cp_async_wait<1>();  // the next key tile (the older group) has landed
      fence_async_smem();
      __syncthreads();
    }
  }

  // partial results of this split: the unnormalised O row, then (max, sum)
  const long long base = (long long)(hk * a.nsplit + s) * Mpad;
#pragma unroll 1
  for (int c0 = 0; c0 < D; c0 += 32) {
    uint32_t v[32];
    tmem_ld32(t_o + (uint32_t)c0, v);
    tmem_ld_wait();
    if (m < M && nsub > 0) {
      float4* dst = reinterpret_cast<float4*>(a.part_o + (base + m) * D + c0);
#pragma unroll
      for (int j = 0; j < 8; ++j)
        dst[j] = make_float4(__uint_as_float(v[4 * j]), __uint_as_float(v[4 * j + 1]), __uint_as_float(v[4 * j + 2]),
                             __uint_as_float(v[4 * j + 3]));
    }
  }
  if (m < M) a.part_ml[base + m] = make_float2(m_run, l_run);
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, L::TMEM_COLS);
}

// ---------------------------------------------------------------- combine
// One CTA per (row, query head).  The splits holding the row's window are
// merged in ascending order: weights exp(m_j - max) go to shared memory in
// chunks, and each thread sums its dims over the chunk, eight loads in
// flight, adding in split order.
constexpr int kCombineThreads = 256;
constexpr int kCombineChunk = 1024;

__global__ void __launch_bounds__(kCombineThreads) attn_combine_kernel(const AttnArgs a) {
  __shared__ float fs[kCombineChunk], ls[kCombineChunk];
  __shared__ float red[kCombineThreads / 32];
  const int G = a.Hq / a.Hkv, Mpad = 16 * a.n_mtiles;
  const int r = blockIdx.x / a.Hq, hq = blockIdx.x % a.Hq, hk = hq / G;
  const int m = r * G + hq % G;
  const int nsr = (a.P + r + a.split) / a.split;  // splits holding positions 0 .. P + r
  const long long row0 = (long long)hk * a.nsplit * Mpad + m;  // split j at row0 + j * Mpad
  const int tid = threadIdx.x;
  // the gate is an input of the call: read it before the dependency wait
  float gt[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int i = tid + h * kCombineThreads;
    gt[h] = i < a.D ? bf16f(a.gate[(long long)r * a.ld_gate + (long long)hq * a.D + i]) : 0.f;
  }
  griddep_wait();
  griddep_launch();
  float mx = -INFINITY;
  for (int j = tid; j < nsr; j += kCombineThreads) mx = fmaxf(mx, a.part_ml[row0 + (long long)j * Mpad].x);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
  if ((tid & 31) == 0) red[tid >> 5] = mx;
  __syncthreads();
  float mstar = red[0];
#pragma unroll
  for (int i = 1; i < kCombineThreads / 32; ++i) mstar = fmaxf(mstar, red[i]);
  constexpr int U = 8;
  float acc[2] = {0.f, 0.f}, l = 0.f;  // dims tid and tid + 256 (head_dim <= 512)
  for (int c0 = 0; c0 < nsr; c0 += kCombineChunk) {
    const int n = min(kCombineChunk, nsr - c0);
    __syncthreads();
    for (int j = tid; j < n; j += kCombineThreads) {
      const float2 ml = a.part_ml[row0 + (long long)(c0 + j) * Mpad];
      fs[j] = ml.x == -INFINITY ? 0.f : expf(ml.x - mstar);
      ls[j] = ml.y;
    }
    __syncthreads();
    for (int j = 0; j < n; ++j) l = fmaf(ls[j], fs[j], l);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int i = tid + h * kCombineThreads;
      if (i >= a.D) break;
      const float* src = a.part_o + (row0 + (long long)c0 * Mpad) * a.D + i;
      const long long stride = (long long)Mpad * a.D;
      int j = 0;
      for (; j + U <= n; j += U) {
        float x[U];
#pragma unroll
        for (int u = 0; u < U; ++u) x[u] = __ldcs(src + (j + u) * stride);
#pragma unroll
        for (int u = 0; u < U; ++u) acc[h] = fmaf(x[u], fs[j + u], acc[h]);
      }
      for (; j < n; ++j) acc[h] = fmaf(__ldcs(src + j * stride), fs[j], acc[h]);
    }
  }
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int i = tid + h * kCombineThreads;
    if (i >= a.D) break;
    const long long oi = (long long)r * a.Hq * a.D + (long long)hq * a.D + i;
    const float y = acc[h] / l * (1.f / (1.f + expf(-gt[h])));
    if (a.dtype == 1) reinterpret_cast<uint16_t*>(a.o)[oi] = f2bf16(y);
    else reinterpret_cast<float*>(a.o)[oi] = y;
  }
}

template <int D>
cudaError_t launch_attn_d(const AttnArgs& a, cudaStream_t s, int* launches) {
  attn_append_kernel<<<dim3(a.k, a.Hkv + a.Hq), 256, 0, s>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e) return e;
  ++*launches;
  // the partial and combine kernels are programmatic dependents: each may
  // start while the kernel before it finishes, and waits before reading its
  // results
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((a.k * (a.Hq / a.Hkv) + kTcM - 1) / kTcM, a.nsplit, a.Hkv);
  cfg.blockDim = dim3(kTcThreads);
  cfg.dynamicSmemBytes = TcSmem<D>::BYTES + 128;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if ((e = cudaLaunchKernelEx(&cfg, attn_partial_kernel<D>, a))) return e;
  ++*launches;
  cfg.gridDim = dim3(a.k * a.Hq);
  cfg.blockDim = dim3(kCombineThreads);
  cfg.dynamicSmemBytes = 0;
  if ((e = cudaLaunchKernelEx(&cfg, attn_combine_kernel, a))) return e;
  ++*launches;
  return cudaSuccess;
}

}  // namespace

cudaError_t attn_setup_kernels() {
  cudaError_t e = cudaFuncSetAttribute(attn_partial_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       TcSmem<128>::BYTES + 128);
  if (e) return e;
  return cudaFuncSetAttribute(attn_partial_kernel<256>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              TcSmem<256>::BYTES + 128);
}

cudaError_t launch_attn(const AttnArgs& a, cudaStream_t s, int* launches) {
  switch (a.D) {
    case 128: return launch_attn_d<128>(a, s, launches);
    case 256: return launch_attn_d<256>(a, s, launches);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace vk
