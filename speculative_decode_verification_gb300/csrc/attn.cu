// Width-k grouped-query attention over a binary16 KV cache ("QWEN38FLASH.md -
// Plan for supporting Qwen/Qwen3.8-Flash-Next" 2.2: 24 query and 2 KV heads of
// dim 256, partial RoPE, sigmoid output gate, F16 cache; "Red Lite dev45 -
// speculative decoding with the Qwen3-Next MTP block", "What it is": row r
// sees the earlier rows' keys and values).
//
// Three launches:
//  1. append: the block's keys (rotated at P + r) and values go into the
//     cache at P + r as binary16; the queries are rotated and scaled by
//     log2(e)/sqrt(D) and kept as binary16 pairs hi + lo.
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
#include <cudaTypedefs.h>
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
// pos * inv_freq[j] is formed and reduced modulo 2 pi in float64 (a handful of
// float64 operations: the device's float64 rate is low), then sin and cos of
// the reduced angle and the rotation in fp32 (a few fp32 ulps, well inside
// the binary16 rounding that follows).
__device__ __forceinline__ float rope_entry(const uint16_t* x, int e, int rope_dim, const double* inv_freq,
                                            long long pos) {
  const float xe = bf16f(x[e]);
  if (e >= rope_dim) return xe;
  const int half = rope_dim / 2;
  const int j = e < half ? e : e - half;
  constexpr double kTwoPi = 6.283185307179586;
  const double ang = (double)pos * inv_freq[j];
  const float red = (float)fma(-kTwoPi, rint(ang * (1.0 / kTwoPi)), ang);
  float sn, cs;
  sincosf(red, &sn, &cs);
  return e < half ? fmaf(xe, cs, -bf16f(x[e + half]) * sn) : fmaf(xe, cs, bf16f(x[e - half]) * sn);
}

// CTA (r, h): h < Hkv appends KV head h's key and value of row r to the cache;
// h >= Hkv rotates and scales query head h - Hkv of row r into its binary16
// pair (hi, lo), stored as pair r * G + g of its KV head.
__global__ void attn_append_kernel(const AttnArgs a) {
  griddep_launch();  // the split kernel may start its prefetch of committed positions
  const int r = blockIdx.x, h = blockIdx.y;
  const long long pos = (long long)a.P + r;
  if (h < a.Hkv) {
    const uint16_t* kr = a.kin + (long long)r * a.ld_k + (long long)h * a.D;
    const uint16_t* vr = a.vin + (long long)r * a.ld_v + (long long)h * a.D;
    for (int e = threadIdx.x; e < a.D; e += blockDim.x) {
      const long long dst = ((long long)h * a.cap + pos) * a.D + e;
      a.K[dst] = __half_as_ushort(__float2half_rn(rope_entry(kr, e, a.rope_dim, a.inv_freq, pos)));
      a.V[dst] = __half_as_ushort(__float2half_rn(bf16f(vr[e])));
    }
    return;
  }
  const int hq = h - a.Hkv, G = a.Hq / a.Hkv;
  const uint16_t* qr = a.q + (long long)r * a.ld_q + (long long)hq * a.D;
  const float qscale = (float)a.qscale;
  // pair r * G + g of KV head hq / G, g = hq % G
  const long long qrow = (long long)(hq / G) * a.q_rows + (long long)r * G + hq % G;
  for (int e = threadIdx.x; e < a.D; e += blockDim.x) {
    const float y = rope_entry(qr, e, a.rope_dim, a.inv_freq, pos) * qscale;
    const __half hi = __float2half_rn(y);
    const long long dst = qrow * a.D + e;
    a.qh[dst] = __half_as_ushort(hi);
    a.ql[dst] = __half_as_ushort(__float2half_rn(y - __half2float(hi)));
  }
}

// ---------------------------------------------------------------- partials
// CTA (M tile, split s, KV head): the 128 (row, query head) pairs m0 .. m0+127
// of that KV head's group against the key positions [s*split, (s+1)*split),
// 64 at a time (sub-tile j: positions s*split + 64 j ..).  Three roles:
//   loads     (warp 4): TMA tile loads of each sub-tile's keys and values,
//             128-byte swizzled, into a ring of shared-memory slots, in the
//             order the MMAs consume them (K0, K1, V0, K2, V1, ...);
//   MMAs      (warp 5): S_j = Q K_j^T into TMEM tile j % 2 (the query's
//             binary16 hi part from TMEM, then its lo part from shared
//             memory), and O += P_j V_j with P_j read from the same TMEM tile
//             (hi part, then lo part), issued as S_0, S_1, PV_0, S_2, PV_1, ...
//             so that the tensor cores run S_{j+1} and PV_{j-1} while the
//             softmax of sub-tile j does;
//   softmax   (warps 0-3, thread t <-> TMEM lane t <-> pair m0 + t): reads its
//             row of S_j, masks positions after the pair's own (P + r) and at
//             or past the split's end, and writes p = 2^(s - m) as binary16 hi
//             and lo parts over S_j.  The scores are in log2 units (the
//             queries carry log2(e) / sqrt(D)).  m is the row's running
//             maximum, raised only when a sub-tile's maximum exceeds it by more
//             than 8: O (an fp32 TMEM tile) and the running sum are then
//             rescaled by 2^(m_old - m_new), otherwise p may reach 2^8 and
//             nothing is rescaled; the result, O / sum, is the same.
// TMEM: S / P tiles at columns 0 and 64, the query's hi part at 128, O at
// 256 (the hi part arrives by TMA in ring slots 3 and 4 and is moved to TMEM
// before those slots take their first tiles).  With fewer than 128 pairs only
// the pairs' rows, rounded up to 8, are loaded; the other rows of the query
// tiles hold whatever shared memory held, and their scores are masked and
// their outputs never stored.  Shared memory: the query's lo part (K-major) and the ring of key and
// value tiles, all 1 KB-aligned 128-byte-swizzle layouts (keys K-major,
// values MN-major: their rows are the cache's rows).  At the end each O row
// goes through shared memory to a bulk copy.  Every wait is a bounded
// mbarrier wait; before the CTA exits, every copy and MMA it issued has
// completed.
constexpr int kTcM = 128;          // pairs per CTA (TMEM lanes)
constexpr int kTcN = 64;           // key positions per sub-tile
constexpr int kSoftThreads = 128;  // warps 0-3
constexpr int kTcThreads = 192;    // + the load warp and the MMA warp
constexpr int kLoadWarp = 4, kMmaWarp = 5;
constexpr int kSBufs = 2;          // S / P tiles in TMEM, 64 columns each
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kQCol = 128;    // the query's hi part: D / 2 columns
constexpr uint32_t kOCol = 256;    // O: D columns
constexpr float kRaiseLog2 = 8.f;  // a row's max is raised when exceeded by more than this (log2 units)

template <int D>
struct TcSmem {
  static constexpr int BLOCK_Q = kTcM * 128;       // one 64-column block of the query (128 rows x 128 B)
  static constexpr int BLOCK_KV = kTcN * 128;      // one 64-column block of a key or value tile
  static constexpr int Q_BYTES = (D / 64) * BLOCK_Q;   // the query's lo part
  static constexpr int TILE_BYTES = (D / 64) * BLOCK_KV;
  static constexpr int SLOTS = D == 256 ? 5 : 10;
  static constexpr int QL = 0, RING = Q_BYTES;
  static constexpr int QH_STAGE = RING + 3 * TILE_BYTES;  // slots 3 and 4 hold the hi part first
  static constexpr int BYTES = RING + SLOTS * TILE_BYTES;
  static constexpr int ALLOC = BYTES + 1024;  // + alignment of the base to 1 KB
  static_assert(SLOTS * TILE_BYTES >= kTcM * (D * 4 + 16), "the O tile is staged in the ring");
  static_assert(SLOTS >= 5 && 2 * TILE_BYTES == Q_BYTES, "the query's hi part is staged in slots 3 and 4");
};

// Rows of one query tile load: the M pairs of a KV head rounded up to 8, at
// most 128 (rows past it stay unloaded: pairs past M, never stored).
__host__ __device__ constexpr int query_box_rows(int M) { return M < kTcM ? (M + 7) / 8 * 8 : kTcM; }

// ring item i -> sub-tile and operand, in the order the MMAs consume them:
// K_0, K_1, V_0, K_2, V_1, ..., K_{n-1}, V_{n-2}, V_{n-1}
__device__ __forceinline__ int k_item(int j) { return j == 0 ? 0 : 2 * j - 1; }
__device__ __forceinline__ int v_item(int j, int n) { return j == n - 1 ? 2 * n - 1 : 2 * j + 2; }

template <int D>
__global__ void __launch_bounds__(kTcThreads, 1) attn_partial_kernel(const __grid_constant__ AttnArgs a) {
  using L = TcSmem<D>;
  constexpr int NS = L::SLOTS;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ __align__(8) uint64_t bars[2 * NS + 2 * kSBufs + 4];
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;
  volatile int* abort = &abort_flag;
  const uint32_t sb = smem_addr(smem);
  const uint32_t bar0 = smem_addr(&bars[0]);
  auto full = [&](int i) { return bar0 + 8u * (uint32_t)i; };                    // slot i landed
  auto empty = [&](int i) { return bar0 + 8u * (uint32_t)(NS + i); };           // slot i read by its MMAs
  auto s_full = [&](int b) { return bar0 + 8u * (uint32_t)(2 * NS + b); };      // S tile b computed
  auto pv_done = [&](int b) { return bar0 + 8u * (uint32_t)(2 * NS + kSBufs + b); };  // P tile b consumed
  const uint32_t p_full = bar0 + 8u * (2 * NS + 2 * kSBufs);      // a sub-tile's P written, O rescaled
  const uint32_t q_full = p_full + 8u;                             // the query's hi part is in TMEM
  const uint32_t mma_drain = q_full + 8u;
  const uint32_t q_lo = mma_drain + 8u;                            // both parts landed in shared memory

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int s = blockIdx.y, hk = blockIdx.z;
  const int G = a.Hq / a.Hkv, M = a.k * G, Mpad = 16 * a.n_mtiles;
  const int m0 = blockIdx.x * kTcM;
  const int end = a.P + a.k;  // positions held by the cache after the append
  const int pos0 = s * a.split;
  const int pos_end = min(pos0 + a.split, end);
  const int n = (pos_end - pos0 + kTcN - 1) / kTcN;  // >= 1: split s starts below the cache's end

  if (tid == 0) {
    abort_flag = 0;
    for (int i = 0; i < NS; ++i) {
      mbar_init(full(i), 1);
      mbar_init(empty(i), 1);
    }
    for (int b = 0; b < kSBufs; ++b) {
      mbar_init(s_full(b), 1);
      mbar_init(pv_done(b), 1);
    }
    mbar_init(p_full, kSoftThreads);
    mbar_init(q_full, kSoftThreads);
    mbar_init(mma_drain, 1);
    mbar_init(q_lo, 1);
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(smem_addr(&tmem_slot), kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;

  if (warp == kLoadWarp) {
    if (lane == 0) {
      // Launched as a programmatic dependent of the append kernel: tiles of
      // positions committed before this call (written at least two launches
      // back) are fetched before the dependency wait, the rest after it.
      // The query (written by the append kernel) follows the dependency wait,
      // which comes right after the first key tile (fetching more before it
      // measured slower: the query then shares the bandwidth with every CTA's
      // prefetch): its lo part into its own region, its hi part into ring
      // slots 3 and 4, from where the softmax warps move it to TMEM before
      // those slots take tiles.
      bool waited = false;
      int issued = 0;
      auto wait_then_query = [&]() {
        griddep_wait();
        waited = true;
        mbar_arrive_expect_tx(q_lo, (uint32_t)(2 * (D / 64) * query_box_rows(M) * 128));
#pragma unroll
        for (int c = 0; c < D / 64; ++c) {
          tma_load_2d(sb + L::QL + c * L::BLOCK_Q, &a.tm_ql, q_lo, 64 * c, hk * a.q_rows + m0);
          tma_load_2d(sb + L::QH_STAGE + c * L::BLOCK_Q, &a.tm_qh, q_lo, 64 * c, hk * a.q_rows + m0);
        }
      };
      for (int i = 0; i < 2 * n; ++i) {
        int j;
        bool values;
        if (i == 2 * n - 1) j = n - 1, values = true;
        else if (i == 0) j = 0, values = false;
        else if (i & 1) j = (i + 1) / 2, values = false;
        else j = i / 2 - 1, values = true;
        const int p0 = pos0 + j * kTcN;
        if (!waited && (p0 + kTcN > a.P || i >= 1)) wait_then_query();
        if (i == 3 && !mbar_wait(q_full, 0, abort, a.err)) break;  // the staged hi part was read
        const int slot = i % NS, use = i / NS;
        if (use > 0 && !mbar_wait(empty(slot), (uint32_t)((use - 1) & 1), abort, a.err)) break;
        mbar_arrive_expect_tx(full(slot), (uint32_t)L::TILE_BYTES);
        const uint32_t dst = sb + L::RING + (uint32_t)slot * L::TILE_BYTES;
#pragma unroll
        for (int c = 0; c < D / 64; ++c)
          tma_load_3d(dst + c * L::BLOCK_KV, values ? &a.tm_v : &a.tm_k, full(slot), 64 * c, p0, hk);
        ++issued;
      }
      if (!waited) wait_then_query();
      // every issued tile has landed before the CTA exits
      for (int i = max(0, issued - NS); i < issued; ++i) mbar_wait_drain(full(i % NS), (uint32_t)((i / NS) & 1), a.err);
      mbar_wait_drain(q_lo, 0, a.err);
    }
  } else if (warp == kMmaWarp) {
    if (lane == 0) {
      constexpr uint32_t IDESC_S = umma_idesc_f16(kTcM, kTcN, false);
      constexpr uint32_t IDESC_O = umma_idesc_f16(kTcM, D, true);
      // O += P_t V_t: P_t from TMEM tile t % 2, V_t MN-major (LBO: 64-column
      // block stride, SBO: 8-key group stride)
      auto issue_pv = [&](int t) -> bool {
        if (!mbar_wait(p_full, (uint32_t)(t & 1), abort, a.err)) return false;
        const int iv = v_item(t, n);
        if (!mbar_wait(full(iv % NS), (uint32_t)((iv / NS) & 1), abort, a.err)) return false;
        tc_fence_after();
        const uint32_t vt = sb + L::RING + (uint32_t)(iv % NS) * L::TILE_BYTES;
        const uint32_t pt = tmem + (uint32_t)(t % kSBufs) * kTcN;
#pragma unroll 1
        for (int part = 0; part < 2; ++part)
#pragma unroll
          for (int ks = 0; ks < kTcN / 16; ++ks)
            umma_f16_ts(tmem + kOCol, pt + (uint32_t)(part * (kTcN / 2) + ks * 8),
                        umma_desc_sw128(vt + ks * 2048, L::BLOCK_KV, 1024), IDESC_O, (t | part | ks) ? 1u : 0u);
        umma_commit(pv_done(t % kSBufs));
        umma_commit(empty(iv % NS));
        return true;
      };
      bool ok = mbar_wait(q_lo, 0, abort, a.err) && mbar_wait(q_full, 0, abort, a.err);
      tc_fence_after();
      for (int j = 0; ok && j < n; ++j) {
        const int b = j % kSBufs;
        // tile b still holds P_{j-2}, read by PV_{j-2}: MMAs issued by one
        // thread execute in issue order, so S_j is issued behind it without
        // waiting for its completion
        const int ik = k_item(j);
        if (!mbar_wait(full(ik % NS), (uint32_t)((ik / NS) & 1), abort, a.err)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t kt = sb + L::RING + (uint32_t)(ik % NS) * L::TILE_BYTES;
        const uint32_t st = tmem + (uint32_t)b * kTcN;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)  // the query's hi part, from TMEM
          umma_f16_ts(st, tmem + kQCol + (uint32_t)(kk * 8),
                      umma_desc_sw128(kt + (kk >> 2) * L::BLOCK_KV + (kk & 3) * 32, 16, 1024), IDESC_S,
                      kk ? 1u : 0u);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)  // its lo part, from shared memory
          umma_f16(st, umma_desc_sw128(sb + L::QL + (kk >> 2) * L::BLOCK_Q + (kk & 3) * 32, 16, 1024),
                   umma_desc_sw128(kt + (kk >> 2) * L::BLOCK_KV + (kk & 3) * 32, 16, 1024), IDESC_S, 1u);
        umma_commit(s_full(b));
        umma_commit(empty(ik % NS));
        if (j >= 1 && !issue_pv(j - 1)) ok = false;
      }
      if (ok) issue_pv(n - 1);
      // every MMA issued above has completed before the CTA exits
      umma_commit(mma_drain);
      mbar_wait_drain(mma_drain, 0, a.err);
    }
  } else {
    const uint32_t t_lane = tmem + ((uint32_t)(32 * warp) << 16);
    const int m = m0 + tid;
    griddep_wait();
    griddep_launch();
    // the hi part of this thread's query (rotated at P + r and scaled by
    // log2(e) / sqrt(D) by the append kernel; rows past M unused) from its
    // staging slots into its TMEM lane; 16-byte chunk c of row t at chunk
    // (c % 8) ^ (t % 8) of its row in 64-column block c / 8
    if (__all_sync(0xffffffffu, mbar_wait(q_lo, 0, abort, a.err))) {
      uint32_t v[D / 64][32];
#pragma unroll
      for (int c = 0; c < D / 8; ++c) {
        const uint32_t src = sb + L::QH_STAGE + (uint32_t)((c >> 3) * L::BLOCK_Q + tid * 128 + (((c & 7) ^ (tid & 7)) << 4));
        asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(v[c >> 3][4 * (c & 7)]), "=r"(v[c >> 3][4 * (c & 7) + 1]), "=r"(v[c >> 3][4 * (c & 7) + 2]),
                       "=r"(v[c >> 3][4 * (c & 7) + 3])
                     : "r"(src));
      }
#pragma unroll
      for (int c = 0; c < D / 64; ++c) tmem_st32(t_lane + kQCol + (uint32_t)(32 * c), v[c]);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(q_full);
    }
    // last position this pair sees in this split (-1: none): its own window,
    // and no further than the split's end
    const int lim = m < M ? min(a.P + m / G, pos_end - 1) : -1;
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    for (int j = 0; j < n; ++j) {
      const int b = j % kSBufs;
      // waits are made warp-uniform: the TMEM loads and stores below are warp-wide
      if (!__all_sync(0xffffffffu, mbar_wait(s_full(b), (uint32_t)((j / kSBufs) & 1), abort, a.err))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t t_s = t_lane + (uint32_t)b * kTcN;
      float sv[kTcN];
      {
        uint32_t v0[32], v1[32];
        tmem_ld32(t_s, v0);
        tmem_ld32(t_s + 32, v1);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          sv[i] = __uint_as_float(v0[i]);
          sv[32 + i] = __uint_as_float(v1[i]);
        }
      }
      const int pbase = pos0 + j * kTcN;
      float mx = -INFINITY;
#pragma unroll
      for (int i = 0; i < kTcN; ++i) {
        sv[i] = pbase + i <= lim ? sv[i] : -INFINITY;
        mx = fmaxf(mx, sv[i]);
      }
      const bool raise = mx > m_run + kRaiseLog2;  // (any finite mx when m_run is -inf)
      const float alpha = raise ? exp2f(m_run - mx) : 1.f;
      if (raise) m_run = mx;
      const float msub = m_run == -INFINITY ? 0.f : m_run;
      float ps = 0.f;
      {
        uint32_t hi[32], lo[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const float p0 = exp2f(sv[2 * e] - msub), p1 = exp2f(sv[2 * e + 1] - msub);
          const __half2 h2 = __floats2half2_rn(p0, p1);
          hi[e] = pack_half2(h2);
          lo[e] = pack_half2(__floats2half2_rn(p0 - __low2float(h2), p1 - __high2float(h2)));
          ps += p0;
          ps += p1;
        }
        tmem_st32(t_s, hi);
        tmem_st32(t_s + 32, lo);
      }
      l_run = fmaf(l_run, alpha, ps);
      // O *= alpha once PV_{j-1} has completed (the whole warp when any of
      // its rows raised its max)
      if (j > 0) {
        if (!__all_sync(0xffffffffu,
                        mbar_wait(pv_done((j - 1) % kSBufs), (uint32_t)(((j - 1) / kSBufs) & 1), abort, a.err))) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (__any_sync(0xffffffffu, raise)) {
#pragma unroll 1
          for (int c0 = 0; c0 < D; c0 += 64) {
            uint32_t v0[32], v1[32];
            tmem_ld32(t_lane + kOCol + (uint32_t)c0, v0);
            tmem_ld32(t_lane + kOCol + (uint32_t)c0 + 32, v1);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              v0[i] = __float_as_uint(__uint_as_float(v0[i]) * alpha);
              v1[i] = __float_as_uint(__uint_as_float(v1[i]) * alpha);
            }
            tmem_st32(t_lane + kOCol + (uint32_t)c0, v0);
            tmem_st32(t_lane + kOCol + (uint32_t)c0 + 32, v1);
          }
        }
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(p_full);
    }
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(pv_done((n - 1) % kSBufs), (uint32_t)(((n - 1) / kSBufs) & 1),
                                                  abort, a.err));
    // partial results of this split: the unnormalised O row (through shared
    // memory, then one bulk copy per row), then (max, sum)
    if (ok) {
      tc_fence_after();
      // every MMA has completed and every tile was consumed: the ring is free.
      // Row t at t * (4D + 16) bytes, so that a warp's 16-byte stores of one
      // column chunk spread over the banks.
      const uint32_t stage = sb + L::RING + (uint32_t)tid * (uint32_t)(D * 4 + 16);
#pragma unroll 1
      for (int c0 = 0; c0 < D; c0 += 32) {
        uint32_t v[32];
        tmem_ld32(t_lane + kOCol + (uint32_t)c0, v);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 8; ++i)
          asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(stage + (uint32_t)(c0 * 4 + i * 16)),
                       "r"(v[4 * i]), "r"(v[4 * i + 1]), "r"(v[4 * i + 2]), "r"(v[4 * i + 3])
                       : "memory");
      }
      if (m < M) {
        const long long base = (long long)(hk * a.nsplit + s) * Mpad;
        fence_async_smem();
        bulk_store(a.part_o + (base + m) * D, stage, (uint32_t)(D * 4));
        bulk_commit();
        a.part_ml[base + m] = make_float2(m_run, l_run);
        bulk_wait_read_all();
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ---------------------------------------------------------------- combine
// One CTA per (row, query head), 8 warps.  Warp w merges the partials of the
// splits w, w + 8, w + 16, ... that hold the row's window, in ascending
// order, in batches whose loads are all in flight at once (lane l holds dims
// 4l .. 4l + 3 and 128 + 4l .. 128 + 4l + 3), keeping its own running
// maximum: O_w and L_w are sums of 2^(m_j - m_w) O_j and 2^(m_j - m_w) l_j.
// The eight warps' sums are then rescaled to the largest m_w and added in
// warp order.
constexpr int kCombineThreads = 256;
constexpr int kCombineWarps = kCombineThreads / 32;
constexpr int kCombineU = 5;  // splits per warp per batch: 40 splits per round of loads

__global__ void __launch_bounds__(kCombineThreads, 2) attn_combine_kernel(const AttnArgs a) {
  __shared__ float4 red_o[kCombineWarps][64];
  __shared__ float red_l[kCombineWarps], red_m[kCombineWarps];
  const int G = a.Hq / a.Hkv, Mpad = 16 * a.n_mtiles;
  const int r = blockIdx.x / a.Hq, hq = blockIdx.x % a.Hq, hk = hq / G;
  const int m = r * G + hq % G;
  const int nsr = (a.P + r + a.split) / a.split;  // splits holding positions 0 .. P + r
  const long long row0 = (long long)hk * a.nsplit * Mpad + m;  // split j at row0 + j * Mpad
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nv = a.D / 128;  // float4 per lane: 2 at D = 256, 1 at D = 128
  // the gate is an input of the call: read it before the dependency wait
  const float gt = tid < a.D ? bf16f(a.gate[(long long)r * a.ld_gate + (long long)hq * a.D + tid]) : 0.f;
  griddep_wait();
  griddep_launch();
  float4 acc[2] = {make_float4(0.f, 0.f, 0.f, 0.f), make_float4(0.f, 0.f, 0.f, 0.f)};
  float l = 0.f, mw = -INFINITY;
  const long long rstride = (long long)Mpad * a.D / 4;  // float4 between consecutive splits
  const float4* src = reinterpret_cast<const float4*>(a.part_o + row0 * a.D) + lane;
  for (int j0 = warp; j0 < nsr; j0 += kCombineWarps * kCombineU) {
    float2 ml[kCombineU];
    float4 x[kCombineU][2];
#pragma unroll
    for (int u = 0; u < kCombineU; ++u) {
      const int j = j0 + u * kCombineWarps;
      const bool in = j < nsr;
      ml[u] = in ? a.part_ml[row0 + (long long)j * Mpad] : make_float2(-INFINITY, 0.f);
#pragma unroll
      for (int h = 0; h < 2; ++h)
        x[u][h] = in && h < nv ? __ldcs(src + j * rstride + h * 32) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    float mb = mw;
#pragma unroll
    for (int u = 0; u < kCombineU; ++u) mb = fmaxf(mb, ml[u].x);
    if (mb == -INFINITY) continue;  // nothing in this batch or before it
    const float sc = mw == -INFINITY ? 0.f : exp2f(mw - mb);
    mw = mb;
    l *= sc;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      acc[h].x *= sc;
      acc[h].y *= sc;
      acc[h].z *= sc;
      acc[h].w *= sc;
    }
#pragma unroll
    for (int u = 0; u < kCombineU; ++u) {
      const float f = ml[u].x == -INFINITY ? 0.f : exp2f(ml[u].x - mb);
      l = fmaf(ml[u].y, f, l);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        acc[h].x = fmaf(x[u][h].x, f, acc[h].x);
        acc[h].y = fmaf(x[u][h].y, f, acc[h].y);
        acc[h].z = fmaf(x[u][h].z, f, acc[h].z);
        acc[h].w = fmaf(x[u][h].w, f, acc[h].w);
      }
    }
  }
  red_o[warp][lane] = acc[0];
  red_o[warp][lane + 32] = acc[1];
  if (lane == 0) {
    red_l[warp] = l;
    red_m[warp] = mw;
  }
  __syncthreads();
  if (tid < a.D) {
    float mstar = red_m[0];
#pragma unroll
    for (int w = 1; w < kCombineWarps; ++w) mstar = fmaxf(mstar, red_m[w]);
    const int q4 = tid >> 2, c = tid & 3;
    float y = 0.f, lt = 0.f;
#pragma unroll
    for (int w = 0; w < kCombineWarps; ++w) {
      const float f = red_m[w] == -INFINITY ? 0.f : exp2f(red_m[w] - mstar);
      const float4 v = red_o[w][q4];
      y = fmaf(c == 0 ? v.x : c == 1 ? v.y : c == 2 ? v.z : v.w, f, y);
      lt = fmaf(red_l[w], f, lt);
    }
    const long long oi = (long long)r * a.Hq * a.D + (long long)hq * a.D + tid;
    const float out = y / lt * (1.f / (1.f + expf(-gt)));
    if (a.dtype == 1) reinterpret_cast<uint16_t*>(a.o)[oi] = f2bf16(out);
    else reinterpret_cast<float*>(a.o)[oi] = out;
  }
}

// Host: the tensor map of one cache (K or V) for the partial kernel's tile
// loads: {D, P + k, Hkv} binary16 with the cache's strides, boxes of 64
// dims x 64 positions, 128-byte swizzle; positions at or past P + k read as
// zeros.
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

cudaError_t encode_cache_map(CUtensorMap* m, uint16_t* base, const AttnArgs& a) {
  if (!g_encode) return cudaErrorInitializationError;
  const cuuint64_t dims[3] = {(cuuint64_t)a.D, (cuuint64_t)(a.P + a.k), (cuuint64_t)a.Hkv};
  const cuuint64_t strides[2] = {(cuuint64_t)a.D * 2, (cuuint64_t)a.cap * a.D * 2};
  const cuuint32_t box[3] = {64, (cuuint32_t)kTcN, 1}, es[3] = {1, 1, 1};
  const CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, base, dims, strides, box, es,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// Host: the tensor map of the queries' hi or lo parts: {D, Hkv * q_rows}
// binary16, boxes of 64 dims x query_box_rows(M) rows, 128-byte swizzle.
cudaError_t encode_query_map(CUtensorMap* m, uint16_t* base, const AttnArgs& a) {
  if (!g_encode) return cudaErrorInitializationError;
  const cuuint64_t dims[2] = {(cuuint64_t)a.D, (cuuint64_t)a.Hkv * a.q_rows};
  const cuuint64_t strides[1] = {(cuuint64_t)a.D * 2};
  const cuuint32_t box[2] = {64, (cuuint32_t)query_box_rows(a.k * (a.Hq / a.Hkv))}, es[2] = {1, 1};
  const CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, base, dims, strides, box, es,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <int D>
cudaError_t launch_attn_d(const AttnArgs& a0, cudaStream_t s, int* launches) {
  AttnArgs a = a0;
  cudaError_t e;
  if ((e = encode_cache_map(&a.tm_k, a.K, a)) || (e = encode_cache_map(&a.tm_v, a.V, a)) ||
      (e = encode_query_map(&a.tm_ql, a.ql, a)) || (e = encode_query_map(&a.tm_qh, a.qh, a)))
    return e;
  attn_append_kernel<<<dim3(a.k, a.Hkv + a.Hq), 256, 0, s>>>(a);
  if ((e = cudaGetLastError())) return e;
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
  cfg.dynamicSmemBytes = TcSmem<D>::ALLOC;
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
  cudaError_t e;
  if (!g_encode) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if ((e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q))) return e;
    if (q != cudaDriverEntryPointSuccess || !fn) return cudaErrorSymbolNotFound;
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  if ((e = cudaFuncSetAttribute(attn_partial_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                TcSmem<128>::ALLOC)))
    return e;
  return cudaFuncSetAttribute(attn_partial_kernel<256>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              TcSmem<256>::ALLOC);
}

cudaError_t launch_attn(const AttnArgs& a, cudaStream_t s, int* launches) {
  switch (a.D) {
    case 128: return launch_attn_d<128>(a, s, launches);
    case 256: return launch_attn_d<256>(a, s, launches);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace vk
