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
//  2. partials: CTA (M group, split s, KV head) takes 2 tiles of 16
//     (row, query head) pairs of that KV head's group and the key positions
//     [s*split, (s+1)*split) of the window, 32 at a time through a
//     double-buffered cp.async ring.  Warp (tile, D half) computes S = Q K^T on
//     the tensor cores (mma.sync m16n8k16, binary16 operands, fp32 sums; the
//     query and the probabilities each as a binary16 pair hi + lo, two MMAs
//     against the same key or value fragment, so that only the cache's own
//     binary16 rounding remains).  Each warp of a tile sums S over its half of
//     the head dim and the halves are added through shared memory; then both
//     mask positions after each row's own (P + r), keep the running max and
//     sum, and accumulate P V for their own half of the head dim.
//  3. combine: per (row, query head) the splits that hold the row's window are
//     merged in ascending order and gated.
// Launches 2 and 3 are programmatic dependents of the one before.
//
// Exactness: a row's arithmetic depends only on its own query, its window and
// the absolute cut of key positions (split and the 32-position sub-tiles), not
// on k or the other rows, so row r of a width-k call equals a width-1 call at
// P + r bit for bit.  Positions past a row's window add exact zeros, and
// splits past it are skipped.
//
// Bound: the cache read, 2 * Hkv * D * 2 bytes per position (2 KB at the
// Flash-Next shape), with 4 * k * Hq * D flops per key position.  The hi + lo
// pairs double the tensor work, and at k ~ 9 the mma.sync pipe, not HBM, is
// the limit: a capture at 65,536 positions shows the tensor pipe 37% busy,
// stalled on MMA dependencies, with DRAM 12% busy.
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "internal.h"

namespace vk {
namespace {

constexpr int kBN = 32;        // key positions per sub-tile
constexpr int kNS = kBN / 8;   // 8-position n-tiles of S per sub-tile
constexpr int kMT = 2;         // tiles of 16 (row, head) pairs per CTA
constexpr int kThreads = 128;  // 4 warps: (tile, D half)

template <int D>
struct AttnSmem {
  static constexpr int LD = D + 8;  // halves per row: 16 B of padding keeps ldmatrix conflict-free
  static constexpr int Q_BYTES = kMT * 16 * LD * 2;         // one of the query's hi / lo parts
  static constexpr int KV_BYTES = kBN * LD * 2;
  static constexpr int BYTES = 2 * Q_BYTES + 2 * 2 * KV_BYTES;  // q hi, q lo, 2 stages of (K, V)
};

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                        uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
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
template <int D>
__global__ void __launch_bounds__(kThreads) attn_partial_kernel(const AttnArgs a) {
  using SM = AttnSmem<D>;
  constexpr int LD = SM::LD;
  constexpr int NTO = D / 16;  // 8-wide output tiles per D half
  extern __shared__ __align__(16) uint8_t smem[];
  uint16_t* Qs = reinterpret_cast<uint16_t*>(smem);                  // q hi
  uint16_t* Qlo = reinterpret_cast<uint16_t*>(smem + SM::Q_BYTES);   // q - q hi
  uint16_t* KVs = reinterpret_cast<uint16_t*>(smem + 2 * SM::Q_BYTES);

  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int g = lane >> 2, c = lane & 3;
  const int s = blockIdx.y, hk = blockIdx.z;
  const int G = a.Hq / a.Hkv, M = a.k * G, Mpad = 16 * a.n_mtiles;
  const int m0 = blockIdx.x * (kMT * 16);
  const int end = a.P + a.k;  // positions held by the cache after the append
  const int pos0 = s * a.split;
  const int pos_end = min(pos0 + a.split, end);
  const int nsub = (pos_end - pos0 + kBN - 1) / kBN;

  auto load_sub = [&](int sub, int stage) {
    const int p0 = pos0 + sub * kBN;
    constexpr int CH = kBN * (D / 8);  // 16-byte chunks per K or V sub-tile
    for (int q = tid; q < 2 * CH; q += kThreads) {
      const int which = q / CH, cc = q % CH;
      const int row = cc / (D / 8), col = (cc % (D / 8)) * 8;
      const int pos = p0 + row;
      const bool ok = pos < end;
      const uint16_t* src = (which ? a.V : a.K) + ((long long)hk * a.cap + (ok ? pos : 0)) * D + col;
      uint16_t* dst = KVs + ((stage * 2 + which) * kBN + row) * LD + col;
      cp_async16(smem_addr(dst), src, ok ? 16u : 0u);  // zero fill past the cache's end
    }
    cp_async_commit();
  };
  // Launched as a programmatic dependent of the append kernel: a first
  // sub-tile of positions committed before this call (written at least two
  // launches back) is fetched before the dependency wait; the queries and the
  // block's own keys and values after it.
  const bool early = pos0 + kBN <= a.P;
  if (early) load_sub(0, 0);
  griddep_wait();
  griddep_launch();
  // queries of this CTA's 32 (row, head) pairs, rotated at P + r and scaled by
  // 1/sqrt(D) by the append kernel: two binary16 parts hi + lo (about 22
  // significant bits; zeros past M).
  {
    constexpr int QCH = kMT * 16 * (D / 8);
    for (int q = tid; q < 2 * QCH; q += kThreads) {
      const int part = q / QCH, cc = q % QCH;
      const int mm = cc / (D / 8), col = (cc % (D / 8)) * 8, m = m0 + mm;
      const bool ok = m < M;
      const long long row = ok ? (long long)(m / G) * a.Hq + hk * G + m % G : 0;
      cp_async16(smem_addr((part ? Qlo : Qs) + mm * LD + col), (part ? a.ql : a.qh) + row * D + col, ok ? 16u : 0u);
    }
  }
  if (early) cp_async_commit();  // the queries as a group of their own
  else load_sub(0, 0);           // the queries travel with the first tile

  const int mt = w >> 1, dh = w & 1;
  const int mrow = m0 + mt * 16;         // first pair of this warp's tile
  const bool live = mrow < M;            // uniform per warp
  int lim[2];                            // last visible position of rows g, g + 8 (-1: none)
#pragma unroll
  for (int ri = 0; ri < 2; ++ri) {
    const int m = mrow + g + 8 * ri;
    lim[ri] = m < M ? a.P + m / G : -1;
  }
  float o_acc[NTO][4];
#pragma unroll
  for (int nt = 0; nt < NTO; ++nt) o_acc[nt][0] = o_acc[nt][1] = o_acc[nt][2] = o_acc[nt][3] = 0.f;
  float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
  // this warp's D half of the query fragments
  const uint32_t q_base = smem_addr(Qs + (mt * 16 + (lane & 15)) * LD + dh * (D / 2) + (lane >> 4) * 8);
  const uint32_t qlo_base = q_base + SM::Q_BYTES;
  __shared__ float xs[4][kNS * 4][32];  // partial scores of each warp, in fragment order

  for (int sub = 0; sub < nsub; ++sub) {
    if (sub + 1 < nsub) {
      load_sub(sub + 1, (sub + 1) & 1);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    if (live) {
      const uint16_t* Ks = KVs + ((sub & 1) * 2) * kBN * LD;
      const uint16_t* Vs = Ks + kBN * LD;
      // S = Q K^T: 16 pairs x kBN positions.  Each warp of the tile sums over
      // its D half (hi and lo query parts in separate accumulators), then the
      // two halves are added through shared memory, half 0 first.
      float sh[kNS][4], sl[kNS][4];
#pragma unroll
      for (int nt = 0; nt < kNS; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) sh[nt][e] = sl[nt][e] = 0.f;
      // lanes 0-7 / 8-15: rows of n-tile 2j at columns +0 / +8; lanes 16-31: n-tile 2j+1
      const uint32_t k_base =
          smem_addr(Ks + ((lane >> 4) * 8 + (lane & 7)) * LD + dh * (D / 2) + ((lane >> 3) & 1) * 8);
#pragma unroll
      for (int kk = 0; kk < D / 32; ++kk) {
        uint32_t a0, a1, a2, a3, l0, l1, l2, l3, b[2 * kNS];
        ldsm_x4(q_base + kk * 32, a0, a1, a2, a3);
        ldsm_x4(qlo_base + kk * 32, l0, l1, l2, l3);
#pragma unroll
        for (int j = 0; j < kNS / 2; ++j)
          ldsm_x4(k_base + j * 16 * LD * 2 + kk * 32, b[4 * j], b[4 * j + 1], b[4 * j + 2], b[4 * j + 3]);
#pragma unroll
        for (int nt = 0; nt < kNS; ++nt) mma_f16(sh[nt], a0, a1, a2, a3, b[2 * nt], b[2 * nt + 1]);
#pragma unroll
        for (int nt = 0; nt < kNS; ++nt) mma_f16(sl[nt], l0, l1, l2, l3, b[2 * nt], b[2 * nt + 1]);
      }
      float sacc[kNS][4];
#pragma unroll
      for (int nt = 0; nt < kNS; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float part = sh[nt][e] + sl[nt][e];
          xs[w][nt * 4 + e][lane] = part;
          sacc[nt][e] = part;
        }
      if (mt == 0) named_bar(1, 64);  // the tile's two warps (constant ids)
      else named_bar(2, 64);
#pragma unroll
      for (int nt = 0; nt < kNS; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float other = xs[w ^ 1][nt * 4 + e][lane];
          sacc[nt][e] = dh == 0 ? sacc[nt][e] + other : other + sacc[nt][e];
        }
      // mask, running max and sum; p rounded to binary16 feeds P V and the sum
      const int pbase = pos0 + sub * kBN;
      float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
      for (int nt = 0; nt < kNS; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int ri = e >> 1, pos = pbase + nt * 8 + 2 * c + (e & 1);
          const float v = pos <= lim[ri] ? sacc[nt][e] : -INFINITY;
          sacc[nt][e] = v;
          mx[ri] = fmaxf(mx[ri], v);
        }
      float alpha[2], msub[2];
#pragma unroll
      for (int ri = 0; ri < 2; ++ri) {
        mx[ri] = fmaxf(mx[ri], __shfl_xor_sync(0xffffffffu, mx[ri], 1));
        mx[ri] = fmaxf(mx[ri], __shfl_xor_sync(0xffffffffu, mx[ri], 2));
        const float mn = fmaxf(m_run[ri], mx[ri]);
        alpha[ri] = mn == -INFINITY ? 1.f : expf(m_run[ri] - mn);
        msub[ri] = mn == -INFINITY ? 0.f : mn;
        m_run[ri] = mn;
      }
      uint32_t pa[kNS][2], pl[kNS][2];  // p as binary16 pairs hi, lo: [n-tile][row g / g + 8]
      float ps[2] = {0.f, 0.f};
#pragma unroll
      for (int nt = 0; nt < kNS; ++nt)
#pragma unroll
        for (int ri = 0; ri < 2; ++ri) {
          const float p0 = expf(sacc[nt][2 * ri] - msub[ri]), p1 = expf(sacc[nt][2 * ri + 1] - msub[ri]);
          const __half2 h2 = __floats2half2_rn(p0, p1);
          pa[nt][ri] = pack_half2(h2);
          pl[nt][ri] = pack_half2(__floats2half2_rn(p0 - __low2float(h2), p1 - __high2float(h2)));
          ps[ri] += p0;
          ps[ri] += p1;
        }
#pragma unroll
      for (int ri = 0; ri < 2; ++ri) {
        ps[ri] += __shfl_xor_sync(0xffffffffu, ps[ri], 1);
        ps[ri] += __shfl_xor_sync(0xffffffffu, ps[ri], 2);
        l_run[ri] = fmaf(l_run[ri], alpha[ri], ps[ri]);
      }
#pragma unroll
      for (int nt = 0; nt < NTO; ++nt) {
        o_acc[nt][0] *= alpha[0];
        o_acc[nt][1] *= alpha[0];
        o_acc[nt][2] *= alpha[1];
        o_acc[nt][3] *= alpha[1];
      }
      // O += P V over this warp's half of the head dim; lanes 0-15 address the
      // 16 positions of a k-step, lanes 16-31 the same for the next n-tile
      const uint32_t v_base = smem_addr(Vs + (lane & 15) * LD + dh * (D / 2) + (lane >> 4) * 8);
#pragma unroll
      for (int kk = 0; kk < kBN / 16; ++kk) {
        const uint32_t a0 = pa[2 * kk][0], a1 = pa[2 * kk][1], a2 = pa[2 * kk + 1][0], a3 = pa[2 * kk + 1][1];
        const uint32_t l0 = pl[2 * kk][0], l1 = pl[2 * kk][1], l2 = pl[2 * kk + 1][0], l3 = pl[2 * kk + 1][1];
#pragma unroll
        for (int nt = 0; nt < NTO; nt += 2) {
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(v_base + (kk * 16 * LD + nt * 8) * 2, b0, b1, b2, b3);
          mma_f16(o_acc[nt], a0, a1, a2, a3, b0, b1);
          mma_f16(o_acc[nt], l0, l1, l2, l3, b0, b1);
          mma_f16(o_acc[nt + 1], a0, a1, a2, a3, b2, b3);
          mma_f16(o_acc[nt + 1], l0, l1, l2, l3, b2, b3);
        }
      }
    }
    __syncthreads();  // the next load reuses this stage
  }

  // partial results of this split
  if (!live) return;
  const long long base = (long long)(hk * a.nsplit + s) * Mpad;
#pragma unroll
  for (int ri = 0; ri < 2; ++ri) {
    const int m = mrow + g + 8 * ri;
    if (m >= M) continue;
    if (dh == 0 && c == 0) a.part_ml[base + m] = make_float2(m_run[ri], l_run[ri]);
    float* dst = a.part_o + (base + m) * D + dh * (D / 2) + 2 * c;
#pragma unroll
    for (int nt = 0; nt < NTO; ++nt)
      *reinterpret_cast<float2*>(dst + nt * 8) = make_float2(o_acc[nt][2 * ri], o_acc[nt][2 * ri + 1]);
  }
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
  cfg.gridDim = dim3((a.n_mtiles + kMT - 1) / kMT, a.nsplit, a.Hkv);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = AttnSmem<D>::BYTES;
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
                                       AttnSmem<128>::BYTES);
  if (e) return e;
  return cudaFuncSetAttribute(attn_partial_kernel<256>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              AttnSmem<256>::BYTES);
}

cudaError_t launch_attn(const AttnArgs& a, cudaStream_t s, int* launches) {
  switch (a.D) {
    case 128: return launch_attn_d<128>(a, s, launches);
    case 256: return launch_attn_d<256>(a, s, launches);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace vk
