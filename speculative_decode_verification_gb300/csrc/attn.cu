// Width-k grouped-query attention over a binary16 KV cache ("QWEN38FLASH.md -
// Plan for supporting Qwen/Qwen3.8-Flash-Next" 2.2: 24 query and 2 KV heads of
// dim 256, partial RoPE, sigmoid output gate, F16 cache; "Red Lite dev45 -
// speculative decoding with the Qwen3-Next MTP block", "What it is": row r
// sees the earlier rows' keys and values).
//
// Three launches:
//  1. append: the block's keys (rotated at P + r, angles in float64) and
//     values go into the cache at P + r as binary16; CTA (r, 0) also writes
//     the (cos, sin) table of row r for the queries.
//  2. partials: CTA (M group, split s, KV head) takes 2 tiles of 16
//     (row, query head) pairs of that KV head's group and the key positions
//     [s*split, (s+1)*split) of the window, 32 at a time through a
//     double-buffered cp.async ring.  Warp (tile, D half) computes S = Q K^T on
//     the tensor cores (mma.sync m16n8k16, binary16 operands, fp32 sums; the
//     query and the probabilities each as a binary16 pair hi + lo, two MMAs
//     against the same key or value fragment, so that only the cache's own
//     binary16 rounding remains), masks
//     positions after each row's own (P + r), keeps the running max and sum,
//     and accumulates P V for its half of the head dim.  Both warps of a tile
//     compute the same S.
//  3. combine: per (row, query head) the splits that hold the row's window are
//     merged in ascending order and gated.
//
// Exactness: a row's arithmetic depends only on its own query, its window and
// the absolute cut of key positions (split and the 32-position sub-tiles), not
// on k or the other rows, so row r of a width-k call equals a width-1 call at
// P + r bit for bit.  Positions past a row's window add exact zeros, and
// splits past it are skipped.
//
// Bound: the cache read, 2 * Hkv * D * 2 bytes per position (2 KB at the
// Flash-Next shape), with the work of k * Hq / Hkv query rows per key; at long
// windows and k ~ 9 the mma.sync pipe, not HBM, is the limit.
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "internal.h"

namespace vk {
namespace {

constexpr int kBN = 32;        // key positions per sub-tile
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
__global__ void attn_append_kernel(const AttnArgs a) {
  const int r = blockIdx.x, h = blockIdx.y, i = threadIdx.x;
  const int half = a.rope_dim / 2;
  const long long pos = (long long)a.P + r;
  const uint16_t* kr = a.kin + (long long)r * a.ld_k + (long long)h * a.D;
  const uint16_t* vr = a.vin + (long long)r * a.ld_v + (long long)h * a.D;
  for (int e = i; e < a.D; e += blockDim.x) {
    double y = (double)bf16f(kr[e]);
    if (e < a.rope_dim) {
      const int j = e < half ? e : e - half;
      double sn, cs;
      sincos((double)pos * pow((double)a.theta, -2.0 * j / a.rope_dim), &sn, &cs);
      y = e < half ? y * cs - (double)bf16f(kr[e + half]) * sn : y * cs + (double)bf16f(kr[e - half]) * sn;
      if (h == 0 && e < half) a.rot[r * half + e] = make_float2((float)cs, (float)sn);
    }
    const long long dst = ((long long)h * a.cap + pos) * a.D + e;
    a.K[dst] = __half_as_ushort(__double2half(y));
    a.V[dst] = __half_as_ushort(__float2half_rn(bf16f(vr[e])));
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
  load_sub(0, 0);

  // queries of this CTA's 32 (row, head) pairs: rotated at P + r, scaled by
  // 1/sqrt(D), held as two binary16 parts hi + lo (about 22 significant bits;
  // zeros past M)
  const float scale = 1.f / sqrtf((float)D);
  const int half = a.rope_dim / 2;
  for (int e = tid; e < kMT * 16 * D; e += kThreads) {
    const int mm = e / D, i = e % D, m = m0 + mm;
    float y = 0.f;
    if (m < M) {
      const int r = m / G, hq = hk * G + m % G;
      const uint16_t* qr = a.q + (long long)r * a.ld_q + (long long)hq * D;
      y = bf16f(qr[i]);
      if (i < a.rope_dim) {
        const float2 cs = a.rot[r * half + (i < half ? i : i - half)];
        y = i < half ? fmaf(y, cs.x, -bf16f(qr[i + half]) * cs.y) : fmaf(y, cs.x, bf16f(qr[i - half]) * cs.y);
      }
    }
    const float ys = y * scale;
    const __half hi = __float2half_rn(ys);
    Qs[mm * LD + i] = __half_as_ushort(hi);
    Qlo[mm * LD + i] = __half_as_ushort(__float2half_rn(ys - __half2float(hi)));
  }

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
  const uint32_t q_base = smem_addr(Qs + (mt * 16 + (lane & 15)) * LD + (lane >> 4) * 8);
  const uint32_t qlo_base = q_base + SM::Q_BYTES;

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
      // S = Q K^T: 16 pairs x 32 positions
      float sacc[4][4];
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) sacc[nt][0] = sacc[nt][1] = sacc[nt][2] = sacc[nt][3] = 0.f;
      // lanes 0-7 / 8-15: rows of n-tile 2j at columns +0 / +8; lanes 16-31: n-tile 2j+1
      const uint32_t k_base = smem_addr(Ks + ((lane >> 4) * 8 + (lane & 7)) * LD + ((lane >> 3) & 1) * 8);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        uint32_t a0, a1, a2, a3, l0, l1, l2, l3;
        ldsm_x4(q_base + kk * 32, a0, a1, a2, a3);
        ldsm_x4(qlo_base + kk * 32, l0, l1, l2, l3);
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          uint32_t b0, b1, b2, b3;
          ldsm_x4(k_base + j * 16 * LD * 2 + kk * 32, b0, b1, b2, b3);
          mma_f16(sacc[2 * j], a0, a1, a2, a3, b0, b1);
          mma_f16(sacc[2 * j], l0, l1, l2, l3, b0, b1);
          mma_f16(sacc[2 * j + 1], a0, a1, a2, a3, b2, b3);
          mma_f16(sacc[2 * j + 1], l0, l1, l2, l3, b2, b3);
        }
      }
      // mask, running max and sum; p rounded to binary16 feeds P V and the sum
      const int pbase = pos0 + sub * kBN;
      float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
      for (int nt = 0; nt < 4; ++nt)
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
      uint32_t pa[4][2], pl[4][2];  // p as binary16 pairs hi, lo: [n-tile][row g / g + 8]
      float ps[2] = {0.f, 0.f};
#pragma unroll
      for (int nt = 0; nt < 4; ++nt)
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
      for (int kk = 0; kk < 2; ++kk) {
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
__global__ void attn_combine_kernel(const AttnArgs a) {
  const int G = a.Hq / a.Hkv, Mpad = 16 * a.n_mtiles;
  const int r = blockIdx.x / a.Hq, hq = blockIdx.x % a.Hq, hk = hq / G;
  const int m = r * G + hq % G;
  const int nsr = (a.P + r + a.split) / a.split;  // splits holding positions 0 .. P + r
  float mstar = -INFINITY;
  for (int j = 0; j < nsr; ++j) mstar = fmaxf(mstar, a.part_ml[(long long)(hk * a.nsplit + j) * Mpad + m].x);
  for (int i = threadIdx.x; i < a.D; i += blockDim.x) {
    float acc = 0.f, l = 0.f;
    for (int j = 0; j < nsr; ++j) {
      const long long row = (long long)(hk * a.nsplit + j) * Mpad + m;
      const float2 ml = a.part_ml[row];
      if (ml.x == -INFINITY) continue;
      const float f = expf(ml.x - mstar);
      acc = fmaf(a.part_o[row * a.D + i], f, acc);
      l = fmaf(ml.y, f, l);
    }
    const long long oi = (long long)r * a.Hq * a.D + (long long)hq * a.D + i;
    const float gt = bf16f(a.gate[(long long)r * a.ld_gate + (long long)hq * a.D + i]);
    const float y = acc / l * (1.f / (1.f + expf(-gt)));
    if (a.dtype == 1) reinterpret_cast<uint16_t*>(a.o)[oi] = f2bf16(y);
    else reinterpret_cast<float*>(a.o)[oi] = y;
  }
}

template <int D>
cudaError_t launch_attn_d(const AttnArgs& a, cudaStream_t s, int* launches) {
  attn_append_kernel<<<dim3(a.k, a.Hkv), 256, 0, s>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e) return e;
  ++*launches;
  const dim3 grid((a.n_mtiles + kMT - 1) / kMT, a.nsplit, a.Hkv);
  attn_partial_kernel<D><<<grid, kThreads, AttnSmem<D>::BYTES, s>>>(a);
  if ((e = cudaGetLastError())) return e;
  ++*launches;
  attn_combine_kernel<<<a.k * a.Hq, 256, 0, s>>>(a);
  if ((e = cudaGetLastError())) return e;
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
