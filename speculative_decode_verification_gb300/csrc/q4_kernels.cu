// q4_kernels.cu - affine Q4/g64 weight x k BF16 rows on the GB300 tensor cores.
//
// What is computed (pages, by title): "Flash-Next optimization transfer to
// Ornith and Qwen 27B", table "Shared architecture and implemented paths"
// (affine Q4, group 64, BF16) and section "Exact verification kernels"
// (width-k equals serial QMV; gathered top-8 experts with fused gate/up);
// "Red Lite dev45 - speculative decoding with the Qwen3-Next MTP block",
// "What it is" (decode each weight once for all rows, each row in the 1-row
// order; all (expert,row) pairs in one dispatch, one tail).
//
// Design (GB300, sm_103a):
//  * Weights are read in the tiled layout of tile.cu: per (128-row tile,
//    256-column chunk) one contiguous block of scales, biases and codes in MMA
//    fragment order.  A CTA is one producer warp plus four consumer warps.  The
//    producer fills a ring of stages in shared memory: one bulk copy per weight
//    block and cp.async of the activation rows, both completing on the stage's
//    mbarrier.  Each weight byte crosses HBM once per call.
//  * Consumers read each fragment with one 16-byte shared load, decode the
//    nibbles to bf16 code values 128 + q (exact) with one lop3 per pair and
//    feed them to mma.sync m16n8k16 as the A operand; the k activation rows
//    are the N columns (8 per MMA; a second column block for k > 8).  Per
//    64-column group the fp32 result C = sum (128 + q) x is folded as
//        acc += s*C + (b - 128 s) * sum(x),
//    the group sums sum(x) added up once per stage.  Products of the integer
//    codes with bf16 x are exact; the accumulation is fp32.
//  * Every output column is an independent dot product, the group order is
//    fixed and the split of K across CTAs depends only on (N, K, SM count):
//    row r of a width-k call is bit-identical to a width-1 call.
//  * Dense: two CTAs per SM, four stages; RB row tiles x S K-splits, the S
//    CTAs of a tile form a thread block cluster and add their partial tiles
//    through distributed shared memory in rank order (no global scratch, no
//    atomics).
//  * Routed MoE: a one-CTA kernel routes every row (a warp per row) and
//    writes the routes.  Then four CTAs per SM, a four-stage ring of 9 KB
//    blocks: each CTA reads the routes, builds the list of work units and works
//    through items: first the gate/up items (expert, row chunk, 64 gate + 64
//    up rows; SwiGLU into the h rows), then the down items (expert, row chunk, 128 output rows;
//    one partial output per (row, rank)).  A down item starts once every
//    gate/up item of its unit is counted done; the items come from two
//    in-order counters such that every such wait ends without assuming
//    that all CTAs are resident.  A second small kernel combines every row's
//    experts in rank order.
#include "argmax.cuh"
#include "common.cuh"
#include "internal.h"

namespace vk {

// A stage: [scales, biases][codes][activation rows].  The first two parts are
// one block of a tiled weight layout (tile.cu: GPU 64-column groups per
// block), copied with one bulk copy.
template <int NT, int ST = kStages, int GPU = kGroupsPerUnit>
struct Q4Layout {
  static constexpr int STAGES = ST;                          // pipeline depth
  static constexpr int GROUPS = GPU;                         // 64-column groups per stage
  static constexpr int NB = 8 * NT;                          // activation rows held per stage
  static constexpr int SB_BYTES = tile_sb_bytes(GPU);        // scales then biases, [row][GPU groups]
  static constexpr int W_BYTES = GPU * kTileGroupBytes;      // codes, fragment order, [group][16-row block][lane]
  static constexpr int X_BYTES = GPU * NB * 128;             // [group][row][64 bf16]
  static constexpr int STAGE = SB_BYTES + W_BYTES + X_BYTES;
  static constexpr int SX_BYTES = GPU * NB * 4;              // fp32 group sums [group][row]
  static constexpr int SX_OFF = ST * STAGE;                  // one slot per stage, after the stages
  static constexpr int BAR_OFF = SX_OFF + ST * SX_BYTES;
  static constexpr int MISC_OFF = BAR_OFF + 2 * ST * 8;
  static constexpr int MISC_BYTES = 64 + 16 * 8;             // flags, then the producer's row-pointer table
  static constexpr int BASE_BYTES = MISC_OFF + MISC_BYTES;
  static_assert(STAGE % 128 == 0, "stages keep 128-byte alignment");
};

// Where a stage of GPU groups holding NBL activation rows keeps them (the
// consumer's view).
template <int NBL, int GPU = kGroupsPerUnit>
struct XLayout {
  static constexpr int NB = NBL;
  static constexpr int SB_BYTES = tile_sb_bytes(GPU);
  static constexpr int W_BYTES = GPU * kTileGroupBytes;
  static constexpr int X_BYTES = GPU * NBL * 128;
};

template <int CW>
struct Warps {
  static constexpr int MT = kBM / 16 / CW;       // 16-row MMA tiles per consumer warp
  static constexpr int THREADS = (CW + 1) * 32;  // + the producer warp
};

// Routing tables kept in shared memory by the MoE kernels.
struct RouteSmem {
  uint32_t mask[kMaxExperts];      // bit r set: row r selected the expert
  int16_t ulist[kMaxExperts];      // distinct selected experts, ascending
  int16_t vlist[2 * kMaxExperts + 2];  // work units: expert slot u (< U, or U = shared) | row chunk << 12
  int32_t idx[16 * kMaxTopK];      // [r][j]
  int U;
  int V;
};

// ---------------------------------------------------------------- producer

// A stage is filled in two parts that both complete on its full barrier: the
// weight block (scales, biases and the gcount groups of codes: one bulk copy,
// expected bytes) and the activation rows (cp.async, then one arrival per
// producer lane).  Only what the consumers read is copied: activation rows
// below nb, groups below gcount.  Anything else in the stage is stale and only
// reaches output columns that are never stored (an MMA column depends on its
// own activation row alone).

// Weight block kc of a row tile (tile: the row tile's first block; GPU
// groups per block).  Reads only static data, with the evict-first L2 policy
// (every weight byte is read once per call).
template <int GPU = kGroupsPerUnit>
__device__ __forceinline__ void produce_w(uint8_t* stage_ptr, uint32_t full_bar, const uint8_t* tile, int kc,
                                          int gcount) {
  const uint32_t bytes = tile_sb_bytes(GPU) + gcount * kTileGroupBytes;
  mbar_arrive_expect_tx(full_bar, bytes);
  bulk_load_hint(smem_addr(stage_ptr), tile + (long long)kc * tile_chunk_bytes(GPU), bytes, full_bar,
                 l2_evict_first_policy());
}

// Activation rows b < nb (brow: their pointers, in shared memory), then this
// lane's arrival once all its copies have landed.
template <int NT, int GPU = kGroupsPerUnit>
__device__ __forceinline__ void produce_x(uint8_t* stage_ptr, uint32_t full_bar, int kc, int gcount,
                                          const uint16_t* const* brow, int nb, int lane) {
  using L = XLayout<8 * NT, GPU>;
  const uint32_t x_dst = smem_addr(stage_ptr) + L::SB_BYTES + L::W_BYTES;
  // [group][row][8 chunks of 16 B], chunk index xor (row & 7)
#pragma unroll
  for (int idx = lane; idx < L::NB * 8 * GPU; idx += 32) {
    const int b = idx / (8 * GPU);
    if (b >= nb) break;
    const int G = (idx >> 3) % GPU;
    const int ch = idx & 7;
    if (G < gcount)
      cp_async16(x_dst + G * (L::NB * 128) + b * 128 + ((ch ^ (b & 7)) << 4),
                 brow[b] + kc * (64 * GPU) + G * 64 + ch * 8, 16u);
  }
  cp_async_mbar_arrive_noinc(full_bar);
}

// Fills one stage.
template <int NT, int GPU = kGroupsPerUnit>
__device__ __forceinline__ void produce_stage(uint8_t* stage_ptr, uint32_t full_bar, const uint8_t* tile, int kc,
                                              int gcount, const uint16_t* const* brow, int nb, int lane) {
  if (lane == 0) produce_w<GPU>(stage_ptr, full_bar, tile, kc, gcount);
  produce_x<NT, GPU>(stage_ptr, full_bar, kc, gcount, brow, nb, lane);
}

// On abort the producer keeps the CTA alive until its bulk copies have landed.
template <int ST = kStages>
__device__ __forceinline__ void producer_drain(uint32_t bar_base, long long fills) {
  for (long long f = (fills > ST ? fills - ST : 0); f < fills; ++f) {
    const int s = (int)(f % ST);
    const uint32_t ph = (uint32_t)((f / ST) & 1);
    const long long t0 = clock64();
    while (!mbar_try_wait(bar_base + 8 * s, ph) && clock64() - t0 < kWaitTimeoutCycles) {
    }
  }
}

// ---------------------------------------------------------------- consumer

// Accumulates group G of a stage into acc for this warp's MT row tiles: NT
// MMA column blocks (activation rows 0 .. 8 NT - 1) of a stage laid out for
// NBL activation rows.
template <int NT, int MT, int NBL, bool MMASUM = false, int GPU = kGroupsPerUnit>
__device__ __forceinline__ void consume_group(uint32_t w_src, uint32_t x_src, uint32_t sx_src, int G,
                                              const uint2 (&sw)[MT][2], const uint2 (&bw)[MT][2],
                                              const int (&rbase)[MT], int lane, float (&acc)[MT][NT][4]) {
  using L = XLayout<NBL, GPU>;
  const int g = lane >> 2, c = lane & 3;
  // B fragments: activation row 8t+g, columns 16c .. 16c+15 of the group
  uint32_t bf[NT][8];
  float sx[NT][2];
#pragma unroll
  for (int t = 0; t < NT; ++t) {
    const int b = 8 * t + g;
    const uint32_t rowa = x_src + G * (L::NB * 128) + b * 128;
    const uint4 xa = lds128(rowa + (((2 * c) ^ (b & 7)) << 4));
    const uint4 xb = lds128(rowa + (((2 * c + 1) ^ (b & 7)) << 4));
    bf[t][0] = xa.x; bf[t][1] = xa.y; bf[t][2] = xa.z; bf[t][3] = xa.w;
    bf[t][4] = xb.x; bf[t][5] = xb.y; bf[t][6] = xb.z; bf[t][7] = xb.w;
    if (MMASUM) {  // sums of activation rows 8t + 2c, 8t + 2c + 1: an MMA with A = 1
      float cs[4] = {0.f, 0.f, 0.f, 0.f};
      constexpr uint32_t ONE2 = 0x3F803F80u;
#pragma unroll
      for (int j = 0; j < 4; ++j) mma_bf16_16816(cs, ONE2, ONE2, ONE2, ONE2, bf[t][2 * j], bf[t][2 * j + 1]);
      sx[t][0] = cs[0];
      sx[t][1] = cs[1];
    } else {
      const uint2 s2 = lds64(sx_src + (G * L::NB + 8 * t + 2 * c) * 4);  // sums of columns 2c, 2c+1
      sx[t][0] = __uint_as_float(s2.x);
      sx[t][1] = __uint_as_float(s2.y);
    }
  }
#pragma unroll
  for (int m = 0; m < MT; ++m) {
    // This lane's four code words of the 16-row block: rows g and g+8, words
    // W0 (columns 16c .. 16c+7 of the group) and W1 (16c+8 .. 16c+15).
    const uint4 w4 = lds128(w_src + ((G * 8 + (rbase[m] >> 4)) * 32 + lane) * 16);
    // Nibble pairs (p, p+4) of a word: lop3 of the word shifted by 4p bits
    // with mask 0x000F000F and the bf16 exponent of 128 -> (128 + q_p, 128 + q_{p+4}).
    // The tiled layout orders the nibbles so that pair p of word Ww is the A
    // fragment of MMA j = 2w + (p & 1), k-slots 2c + 8 (p >> 1) and the next,
    // i.e. activation columns 16c + 4j + 2 (p >> 1) and the next.
    uint32_t A[4][4];
    {
      const uint32_t v[4] = {w4.x, w4.y, w4.z, w4.w};  // row g W0, row g+8 W0, row g W1, row g+8 W1
      uint32_t q[4][4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        q[i][0] = and_or(v[i], 0x000F000Fu, 0x43004300u);
        q[i][1] = and_or(v[i] >> 4, 0x000F000Fu, 0x43004300u);
        q[i][2] = and_or(v[i] >> 8, 0x000F000Fu, 0x43004300u);
        q[i][3] = and_or(v[i] >> 12, 0x000F000Fu, 0x43004300u);
      }
#pragma unroll
      for (int wd = 0; wd < 2; ++wd)
#pragma unroll
        for (int odd = 0; odd < 2; ++odd) {
          const int j = 2 * wd + odd;
          A[j][0] = q[2 * wd][odd];          // row g,   k-slots 2c, 2c+1
          A[j][1] = q[2 * wd + 1][odd];      // row g+8
          A[j][2] = q[2 * wd][odd + 2];      // row g,   k-slots 2c+8, 2c+9
          A[j][3] = q[2 * wd + 1][odd + 2];  // row g+8
        }
    }
    const uint32_t s_lo = (G & 2) ? sw[m][0].y : sw[m][0].x;
    const uint32_t s_hi = (G & 2) ? sw[m][1].y : sw[m][1].x;
    const uint32_t b_lo = (G & 2) ? bw[m][0].y : bw[m][0].x;
    const uint32_t b_hi = (G & 2) ? bw[m][1].y : bw[m][1].x;
    const float sA = (G & 1) ? bf16hi(s_lo) : bf16lo(s_lo);
    const float sB = (G & 1) ? bf16hi(s_hi) : bf16lo(s_hi);
    const float bA = fmaf(-128.f, sA, (G & 1) ? bf16hi(b_lo) : bf16lo(b_lo));
    const float bB = fmaf(-128.f, sB, (G & 1) ? bf16hi(b_hi) : bf16lo(b_hi));
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      float cg[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int j = 0; j < 4; ++j)
        mma_bf16_16816(cg, A[j][0], A[j][1], A[j][2], A[j][3], bf[t][2 * j], bf[t][2 * j + 1]);
      acc[m][t][0] = fmaf(bA, sx[t][0], fmaf(sA, cg[0], acc[m][t][0]));
      acc[m][t][1] = fmaf(bA, sx[t][1], fmaf(sA, cg[1], acc[m][t][1]));
      acc[m][t][2] = fmaf(bB, sx[t][0], fmaf(sB, cg[2], acc[m][t][2]));
      acc[m][t][3] = fmaf(bB, sx[t][1], fmaf(sB, cg[3], acc[m][t][3]));
    }
  }
}

// Accumulates one stage (gcount groups) for NT MMA column blocks; the stage
// holds NBL activation rows (NBL >= 8 NT).  ok = false: the stage never filled
// (abort) - keep the named-barrier count, skip the math.  The activation
// group sums come either from consumer warp w < 4 adding up group w once per
// stage (then a named barrier), or with MMASUM from one MMA with an all-ones
// A operand in every warp, with no barrier (the routed-expert kernel).
template <int NT, int CW, int NBL, bool MMASUM = false, int GPU = kGroupsPerUnit>
__device__ __forceinline__ void consume_stage(const uint8_t* stage_ptr, uint32_t sx_src, int gcount,
                                              const int (&rbase)[Warps<CW>::MT], int lane,
                                              float (&acc)[Warps<CW>::MT][NT][4], bool ok) {
  static_assert(NBL >= 8 * NT, "stage holds too few activation rows");
  static_assert(MMASUM || GPU == 4, "per-warp group sums need one consumer warp per group");
  using L = XLayout<NBL, GPU>;
  constexpr int MT = Warps<CW>::MT;
  const uint32_t sb_src = smem_addr(stage_ptr);
  const uint32_t w_src = sb_src + L::SB_BYTES;
  const uint32_t x_src = w_src + L::W_BYTES;
  const int g = lane >> 2, c = lane & 3;
  const int w = threadIdx.x >> 5;
  if (!ok) {
    if (!MMASUM) named_bar(2, CW * 32);
    return;
  }
  // Consumer warp w < 4 adds up activation group w of the stage: each thread
  // its 16 values, then the four threads of a row.
  if (!MMASUM && w < gcount) {
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      const int b = 8 * t + g;
      const uint32_t rowa = x_src + w * (L::NB * 128) + b * 128;
      const uint32_t ca = rowa + (((2 * c) ^ (b & 7)) << 4), cb = rowa + (((2 * c + 1) ^ (b & 7)) << 4);
      const uint4 xa = lds128(ca);
      const uint4 xb = lds128(cb);
      float part = (bf16lo(xa.x) + bf16hi(xa.x)) + (bf16lo(xa.y) + bf16hi(xa.y));
      part += (bf16lo(xa.z) + bf16hi(xa.z)) + (bf16lo(xa.w) + bf16hi(xa.w));
      part += (bf16lo(xb.x) + bf16hi(xb.x)) + (bf16lo(xb.y) + bf16hi(xb.y));
      part += (bf16lo(xb.z) + bf16hi(xb.z)) + (bf16lo(xb.w) + bf16hi(xb.w));
      part += __shfl_xor_sync(0xffffffffu, part, 1);
      part += __shfl_xor_sync(0xffffffffu, part, 2);
      if (c == 0) asm volatile("st.shared.f32 [%0], %1;" ::"r"(sx_src + (w * L::NB + b) * 4), "f"(part) : "memory");
    }
  }
  // scales / biases of this thread's rows, GPU groups each ([row][GPU] bf16;
  // with two groups the pair sits in .x)
  uint2 sw[MT][2], bw[MT][2];
#pragma unroll
  for (int m = 0; m < MT; ++m)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int row = rbase[m] + g + 8 * h;
      if (GPU == 4) {
        sw[m][h] = lds64(sb_src + row * 8);
        bw[m][h] = lds64(sb_src + kBM * 8 + row * 8);
      } else {
        static_assert(GPU == 4 || GPU == 2, "two or four groups per stage");
        sw[m][h] = make_uint2(lds32(sb_src + row * 4), 0u);
        bw[m][h] = make_uint2(lds32(sb_src + kBM * 4 + row * 4), 0u);
      }
    }
  if (!MMASUM) named_bar(2, CW * 32);
  if (gcount == GPU) {
#pragma unroll
    for (int G = 0; G < GPU; ++G)
      consume_group<NT, MT, NBL, MMASUM, GPU>(w_src, x_src, sx_src, G, sw, bw, rbase, lane, acc);
  } else {
#pragma unroll 1
    for (int G = 0; G < gcount; ++G)
      consume_group<NT, MT, NBL, MMASUM, GPU>(w_src, x_src, sx_src, G, sw, bw, rbase, lane, acc);
  }
}

__device__ __forceinline__ void store_out(void* y, int dtype, long long i, float v) {
  if (dtype == 1) {
    reinterpret_cast<uint16_t*>(y)[i] = f2bf16(v);
  } else if (dtype == 2) {
    reinterpret_cast<float*>(y)[i] += v;
  } else {
    reinterpret_cast<float*>(y)[i] = v;
  }
}

template <int MT, int NT>
__device__ __forceinline__ void zero_acc(float (&acc)[MT][NT][4]) {
#pragma unroll
  for (int m = 0; m < MT; ++m)
#pragma unroll
    for (int t = 0; t < NT; ++t)
#pragma unroll
      for (int q = 0; q < 4; ++q) acc[m][t][q] = 0.f;
}

template <int CW, int ST = kStages>
__device__ __forceinline__ void init_barriers(uint32_t bar_base) {
  if (threadIdx.x == 0) {
    for (int s = 0; s < ST; ++s) {
      mbar_init(bar_base + 8 * s, 33);         // full: lane 0's tx arrival + 32 cp.async arrivals
      mbar_init(bar_base + 8 * (ST + s), CW);  // empty: one arrival per consumer warp
    }
    fence_mbar_init();
  }
}

// ================================================================== dense

// Argmax epilogue of the dense product (the LM head's greedy choice): each
// consumer warp takes the largest key of its output rows per column, the CTA
// merges its warps in shared memory and each column with one 64-bit atomicMax
// (no fence, no ticket: a one-CTA launch of the acceptance kernel reads the
// merged keys after this kernel).  Consumer threads only; the keys are those
// of the fp32 values the plain product would store.
template <int NT, int MT>
__device__ void dense_argmax_epilogue(const DenseArgs& a, const float (&acc)[MT][NT][4], const bool (&mine)[MT],
                                      int tile, const int (&rbase)[MT], int warp, int lane, uint8_t* scratch,
                                      bool aborted) {
  constexpr int CW = kDenseWarps, NTH = CW * 32;
  constexpr uint32_t FULL = 0xffffffffu;
  const int g = lane >> 2, c = lane & 3;
  unsigned long long* red = reinterpret_cast<unsigned long long*>(scratch);  // [CW][16]
  unsigned long long kb[NT][2];
#pragma unroll
  for (int t = 0; t < NT; ++t) kb[t][0] = kb[t][1] = 0ull;
#pragma unroll
  for (int m = 0; m < MT; ++m)
#pragma unroll
    for (int t = 0; t < NT; ++t)
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int row = tile * kBM + rbase[m] + g + 8 * (q >> 1);
        const int col = 8 * t + 2 * c + (q & 1);
        if (mine[m] && row < a.N && col < a.k) kb[t][q & 1] = umax64(kb[t][q & 1], argmax_key(acc[m][t][q], row));
      }
#pragma unroll
  for (int t = 0; t < NT; ++t)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) kb[t][e] = umax64(kb[t][e], __shfl_xor_sync(FULL, kb[t][e], off));
      if (g == 0) red[warp * 16 + 8 * t + 2 * c + e] = kb[t][e];
    }
  named_bar(2, NTH);
  if (warp == 0 && lane < a.k && !aborted) {
    unsigned long long mk = 0ull;
#pragma unroll
    for (int w = 0; w < CW; ++w) mk = umax64(mk, red[w * 16 + lane]);
    if (mk) atomicMax(a.best + a.r0 + lane, mk);
  }
}

template <int NT, bool ARGMAX = false>
__global__ void __launch_bounds__(Warps<kDenseWarps>::THREADS, kQ4CtasPerSm)
    q4_dense_kernel(const DenseArgs a) {
  using L = Q4Layout<NT>;
  constexpr int CW = kDenseWarps, MT = Warps<CW>::MT;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t bar_base = smem_addr(smem + L::BAR_OFF);
  volatile int* abort = reinterpret_cast<volatile int*>(smem + L::MISC_OFF);
  if (threadIdx.x == 0) *abort = 0;
  init_barriers<CW>(bar_base);
  __syncthreads();

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int S = a.S;
  const int tile = blockIdx.x / S, split = blockIdx.x % S;
  const int kc0 = split * a.KC / S, kc1 = (split + 1) * a.KC / S;

  if (warp == CW) {
    // ------------------------------------------------------------ producer
    const uint16_t** brow = reinterpret_cast<const uint16_t**>(smem + L::MISC_OFF + 64);
    if (lane < L::NB) brow[lane] = a.x + (long long)(lane < a.k ? lane : 0) * a.K;
    __syncwarp();
    const uint8_t* ts = a.tiles + (long long)tile * a.rt_bytes;
    // The first stages' weights are static: fetch them before the previous
    // kernel has finished (the ring is empty, no wait), the activations after.
    const int n_pre = min(kStages, kc1 - kc0);
    if (lane == 0)
      for (int f = 0; f < n_pre; ++f)
        produce_w(smem + f * L::STAGE, bar_base + 8 * f, ts, kc0 + f, min(kGroupsPerUnit, a.KG - 4 * (kc0 + f)));
    griddep_wait();
    griddep_launch();
    for (int f = 0; f < n_pre; ++f)
      produce_x<NT>(smem + f * L::STAGE, bar_base + 8 * f, kc0 + f, min(kGroupsPerUnit, a.KG - 4 * (kc0 + f)), brow,
                    a.k, lane);
    long long fills = n_pre;
    for (int kc = kc0 + n_pre; kc < kc1; ++kc, ++fills) {
      const int s = (int)(fills % kStages);
      const uint32_t ph = (uint32_t)((fills / kStages) & 1);
      if (!mbar_wait(bar_base + 8 * (kStages + s), ph ^ 1, abort, a.err)) break;
      const int gcount = min(kGroupsPerUnit, a.KG - 4 * kc);
      produce_stage<NT>(smem + s * L::STAGE, bar_base + 8 * s, ts, kc, gcount, brow, a.k, lane);
    }
    if (*abort) producer_drain(bar_base, fills);
    if (S > 1) {  // the producer warp takes part in the cluster barriers
      cluster_sync();
      cluster_arrive();
      cluster_wait();
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  griddep_wait();
  griddep_launch();
  const int g = lane >> 2, c = lane & 3;
  int rbase[MT];
#pragma unroll
  for (int m = 0; m < MT; ++m) rbase[m] = 16 * (warp * MT + m);
  float acc[MT][NT][4];
  zero_acc<MT, NT>(acc);
  long long fills = 0;
  for (int kc = kc0; kc < kc1; ++kc, ++fills) {
    const int s = (int)(fills % kStages);
    const uint32_t ph = (uint32_t)((fills / kStages) & 1);
    const bool ok = mbar_wait(bar_base + 8 * s, ph, abort, a.err);
    const int gcount = min(kGroupsPerUnit, a.KG - 4 * kc);
    consume_stage<NT, CW, L::NB>(smem + s * L::STAGE, smem_addr(smem + L::SX_OFF + s * L::SX_BYTES), gcount, rbase,
                                 lane, acc, ok);
    __syncwarp();
    if (lane == 0) mbar_arrive(bar_base + 8 * (kStages + s));
  }
  // Which of this warp's row tiles does this CTA write?  With S > 1, 16-row
  // tile mt of the 128-row tile belongs to rank mt % S, which sums the S
  // partial tiles in rank order.
  bool mine[MT];
#pragma unroll
  for (int m = 0; m < MT; ++m) mine[m] = S == 1 || ((warp * MT + m) % S) == split;
  // y += result: the old values this CTA adds to, loaded now so that the
  // loads overlap the cluster reduction
  float old[MT][NT][4];
#pragma unroll
  for (int m = 0; m < MT; ++m)
#pragma unroll
    for (int t = 0; t < NT; ++t)
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int row = tile * kBM + rbase[m] + g + 8 * (q >> 1);
        const int col = 8 * t + 2 * c + (q & 1);
        old[m][t][q] = (a.dtype == 2 && mine[m] && row < a.N && col < a.k)
                           ? reinterpret_cast<const float*>(a.y)[(long long)col * a.N + row]
                           : 0.f;
      }
  if (S > 1) {
    // Stage 0 now holds this CTA's partial tile: once every consumer warp is
    // done with the last stage, which may itself be stage 0.
    named_bar(2, CW * 32);
    float4* part = reinterpret_cast<float4*>(smem);
#pragma unroll
    for (int m = 0; m < MT; ++m)
#pragma unroll
      for (int t = 0; t < NT; ++t)
        part[((warp * MT + m) * NT + t) * 32 + lane] = make_float4(acc[m][t][0], acc[m][t][1], acc[m][t][2], acc[m][t][3]);
    cluster_sync();
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      if (!mine[m]) continue;  // warp-uniform
      // up to 8 ranks' four-float loads in flight at once, then their adds; in rank order
      constexpr int QB = 8;
#pragma unroll
      for (int t = 0; t < NT; ++t) acc[m][t][0] = acc[m][t][1] = acc[m][t][2] = acc[m][t][3] = 0.f;
      for (int q0 = 0; q0 < S; q0 += QB) {
        float4 pv[QB][NT];
#pragma unroll
        for (int q = 0; q < QB; ++q)
#pragma unroll
          for (int t = 0; t < NT; ++t)
            if (q0 + q < S) pv[q][t] = ld_dsmem_f32x4(part + ((warp * MT + m) * NT + t) * 32 + lane, (uint32_t)(q0 + q));
#pragma unroll
        for (int t = 0; t < NT; ++t)
#pragma unroll
          for (int q = 0; q < QB; ++q)
            if (q0 + q < S) {
              acc[m][t][0] += pv[q][t].x;
              acc[m][t][1] += pv[q][t].y;
              acc[m][t][2] += pv[q][t].z;
              acc[m][t][3] += pv[q][t].w;
            }
      }
    }
    cluster_arrive();  // this CTA has read its peers' partial tiles
  }
  if constexpr (ARGMAX) {
    // stage 1's space is free (stage 0 may still hold the partial tile peers read)
    dense_argmax_epilogue<NT, MT>(a, acc, mine, tile, rbase, warp, lane, smem + L::STAGE, *abort != 0);
  } else if (!*abort) {
#pragma unroll
    for (int m = 0; m < MT; ++m)
#pragma unroll
      for (int t = 0; t < NT; ++t)
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int row = tile * kBM + rbase[m] + g + 8 * (q >> 1);
          const int col = 8 * t + 2 * c + (q & 1);
          if (!mine[m] || row >= a.N || col >= a.k) continue;
          const long long i = (long long)col * a.N + row;
          if (a.dtype == 2) reinterpret_cast<float*>(a.y)[i] = old[m][t][q] + acc[m][t][q];
          else store_out(a.y, a.dtype, i, acc[m][t][q]);
        }
  }
  if (S > 1) cluster_wait();  // peers keep their shared memory until every rank has read it
}

// ================================================================== MoE

// Top-T routing (deterministic): descending logit, equal logits -> lower
// index; weights = softmax over the T selected logits (fp32).
//
// One warp takes R rows at once, interleaved so that their latencies overlap.
// A logit becomes an order-preserving key (0 = no expert; -0 counts as +0).
// Each lane keeps its four best keys in descending order (equal keys: lower
// index first), updated with compares and selects rather than branches.  A
// round takes the warp maximum key and, among the lanes holding it, the lowest
// expert index; the winning lane shifts its list and, once its four are taken,
// rescans its remaining keys (rare).
template <int R>
__device__ __forceinline__ void route_warp_rows(const float* logits, long long ld, int E, int T, const int (&row)[R],
                                                int lane, int (&e_out)[R], float (&w_out)[R]) {
  constexpr int NI = kMaxExperts / 32;
  constexpr uint32_t FULL = 0xffffffffu;
  uint32_t key[R][NI];
  {
    float v[R][NI];
#pragma unroll
    for (int q = 0; q < R; ++q) {
      const float* l = logits + (long long)(row[q] < 0 ? 0 : row[q]) * ld;
#pragma unroll
      for (int i = 0; i < NI; ++i) {
        const int e = lane + 32 * i;
        v[q][i] = (row[q] >= 0 && e < E) ? __ldcg(l + e) : 0.f;  // L2: written by the kernel before
      }
    }
#pragma unroll
    for (int q = 0; q < R; ++q)
#pragma unroll
      for (int i = 0; i < NI; ++i) {
        const uint32_t b = __float_as_uint(v[q][i] == 0.f ? 0.f : v[q][i]);
        key[q][i] = (row[q] >= 0 && lane + 32 * i < E) ? ((b & 0x80000000u) ? ~b : (b | 0x80000000u)) : 0u;
      }
  }
  uint32_t taken[R], tk[R][4];
  int ti[R][4];
  // this lane's four best keys not yet taken, descending
  auto scan = [&](int q) {
    uint32_t k0 = 0u, k1 = 0u, k2 = 0u, k3 = 0u;
    int i0 = 0, i1 = 0, i2 = 0, i3 = 0;
#pragma unroll
    for (int i = 0; i < NI; ++i) {
      const uint32_t kv = ((taken[q] >> i) & 1u) ? 0u : key[q][i];
      const bool c0 = kv > k0, c1 = kv > k1, c2 = kv > k2, c3 = kv > k3;  // c0 => c1 => c2 => c3
      k3 = c2 ? k2 : (c3 ? kv : k3);
      i3 = c2 ? i2 : (c3 ? i : i3);
      k2 = c1 ? k1 : (c2 ? kv : k2);
      i2 = c1 ? i1 : (c2 ? i : i2);
      k1 = c0 ? k0 : (c1 ? kv : k1);
      i1 = c0 ? i0 : (c1 ? i : i1);
      k0 = c0 ? kv : k0;
      i0 = c0 ? i : i0;
    }
    tk[q][0] = k0; tk[q][1] = k1; tk[q][2] = k2; tk[q][3] = k3;
    ti[q][0] = i0; ti[q][1] = i1; ti[q][2] = i2; ti[q][3] = i3;
  };
#pragma unroll
  for (int q = 0; q < R; ++q) {
    taken[q] = 0u;
    scan(q);
  }
  float myv[R];
  int mye[R];
#pragma unroll
  for (int q = 0; q < R; ++q) { myv[q] = 0.f; mye[q] = -1; }
  for (int j = 0; j < T; ++j) {
    // the R rows' reductions back to back (independent), then the updates
    uint32_t m[R], we[R];
#pragma unroll
    for (int q = 0; q < R; ++q) m[q] = __reduce_max_sync(FULL, tk[q][0]);
#pragma unroll
    for (int q = 0; q < R; ++q)
      we[q] = __reduce_min_sync(FULL, tk[q][0] == m[q] ? (uint32_t)(lane + 32 * ti[q][0]) : FULL);
    bool rescan[R];
#pragma unroll
    for (int q = 0; q < R; ++q) {
      const bool win = row[q] >= 0 && lane == (int)(we[q] & 31u);
      taken[q] |= win ? (1u << ti[q][0]) : 0u;
      tk[q][0] = win ? tk[q][1] : tk[q][0]; ti[q][0] = win ? ti[q][1] : ti[q][0];
      tk[q][1] = win ? tk[q][2] : tk[q][1]; ti[q][1] = win ? ti[q][2] : ti[q][1];
      tk[q][2] = win ? tk[q][3] : tk[q][2]; ti[q][2] = win ? ti[q][3] : ti[q][2];
      tk[q][3] = win ? 0u : tk[q][3];
      rescan[q] = win && tk[q][0] == 0u;  // four taken from this lane: look at the rest
      if (lane == j) {
        myv[q] = __uint_as_float((m[q] & 0x80000000u) ? (m[q] & 0x7fffffffu) : ~m[q]);
        mye[q] = (int)we[q];
      }
    }
#pragma unroll
    for (int q = 0; q < R; ++q)
      if (rescan[q]) scan(q);
  }
#pragma unroll
  for (int q = 0; q < R; ++q) {
    const float top = __shfl_sync(FULL, myv[q], 0);
    const float ex = lane < T ? expf(myv[q] - top) : 0.f;
    float sum = ex;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(FULL, sum, off);
    sum = __shfl_sync(FULL, sum, 0);
    e_out[q] = mye[q];
    w_out[q] = ex / sum;
  }
}

// The routing of a call, once: warp r routes row r (up to 16 rows) and lane
// j < T writes the row's j-th expert and weight to idx_out / w_out, which the
// expert kernel and the combine then read.
__global__ void __launch_bounds__(32 * 16) moe_route_kernel(const MoeArgs a) {
  griddep_wait();  // the routing logits come from the kernel before
  griddep_launch();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp >= a.k) return;
  const int row[1] = {warp};
  int e[1];
  float w[1];
  route_warp_rows<1>(a.logits, a.logits_ld, a.E, a.T, row, lane, e, w);
  if (lane < a.T) {
    a.idx_out[warp * a.T + lane] = e[0];
    a.w_out[warp * a.T + lane] = w[0];
  }
}

// Reads the routes of rows 0 .. k-1 (idx, [k, T], written by the routing
// kernel) into rs: per row its experts, per expert the bitmask of its rows.
// Then one pass over the masks gives the distinct experts and the work units.
// Every thread of the CTA calls it, after rs->mask has been zeroed and a CTA
// barrier; it ends with __syncthreads.
__device__ void load_routes(const int32_t* idx, int T, int k, int has_shared, RouteSmem* rs) {
  const int tid = threadIdx.x, nthr = blockDim.x;
  const int warp = tid >> 5, lane = tid & 31;
  for (int t = tid; t < k * T; t += nthr) {
    const int r = t / T, j = t - r * T;
    const int e = __ldcg(idx + t);  // L2: written by the kernel before
    rs->idx[r * kMaxTopK + j] = e;
    atomicOr(&rs->mask[e], 1u << r);
  }
  __syncthreads();
  if (warp == 0) {
    // One pass over the masks gives the distinct experts (ascending) and the
    // work units: (expert slot u, chunk c of 8 of its rows), the chunks of one
    // expert adjacent so that its weights are read back to back.  At most 16
    // rows, so an expert has one chunk, or two when more than 8 rows chose it.
    // Lane l takes experts 16 l .. 16 l + 15: it counts its experts and units,
    // a warp scan gives its first slots, then it writes its own entries.
    constexpr int PER = kMaxExperts / 32;
    uint32_t mk[PER];
    const uint4* m4 = reinterpret_cast<const uint4*>(rs->mask + PER * lane);
#pragma unroll
    for (int i = 0; i < PER / 4; ++i) {
      const uint4 t = m4[i];
      mk[4 * i] = t.x; mk[4 * i + 1] = t.y; mk[4 * i + 2] = t.z; mk[4 * i + 3] = t.w;
    }
    uint32_t fm = 0u, tm = 0u;  // bit i: expert 16 l + i selected; selected by more than 8 rows
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      fm |= (mk[i] != 0u ? 1u : 0u) << i;
      tm |= (__popc(mk[i]) > 8 ? 1u : 0u) << i;
    }
    const int packed = __popc(fm) | ((__popc(fm) + __popc(tm)) << 16);  // the halves never carry
    int incl = packed;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += t;
    }
    int u = (incl - packed) & 0xFFFF, vp = (incl - packed) >> 16;
    for (; fm; fm &= fm - 1u) {
      const int i = __ffs(fm) - 1;
      rs->ulist[u] = (int16_t)(PER * lane + i);
      rs->vlist[vp++] = (int16_t)u;
      if ((tm >> i) & 1u) rs->vlist[vp++] = (int16_t)(u | (1 << 12));
      ++u;
    }
    const int tot = __shfl_sync(0xffffffffu, incl, 31);
    const int running = tot & 0xFFFF;
    int vrun = tot >> 16;
    if (lane == 0) {
      if (has_shared) {  // slot U: the shared expert, every row
        for (int c = 0; c < (k + 7) / 8; ++c) rs->vlist[vrun + c] = (int16_t)(running | (c << 12));
        vrun += (k + 7) / 8;
      }
      rs->U = running;
      rs->V = vrun;
    }
  }
  __syncthreads();
}

// Row r and rank j of the b-th (ascending row) pair routed to expert slot u.
__device__ __forceinline__ void pair_of(const RouteSmem* rs, const MoeArgs& a, int u, int b, int& r, int& j) {
  if (u >= rs->U) {  // shared expert: every row, slot T
    r = b;
    j = a.T;
    return;
  }
  const int e = rs->ulist[u];
  uint32_t m = rs->mask[e];
  for (int i = 0; i < b; ++i) m &= m - 1u;
  r = __ffs(m) - 1;
  j = 0;
  for (int jj = 0; jj < a.T; ++jj)
    if (rs->idx[r * kMaxTopK + jj] == e) j = jj;
}

__device__ __forceinline__ int pairs_of(const RouteSmem* rs, const MoeArgs& a, int u) {
  return u >= rs->U ? a.k : __popc(rs->mask[rs->ulist[u]]);
}

// One item of a MoE kernel on the consumer side: the stage loop and the
// epilogue.  The item covers rows 8 rc .. 8 rc + nb - 1 of expert slot u.
template <int CW, bool GATEUP, int ST, int GPU>
__device__ __forceinline__ void moe_item(const MoeArgs& a, const RouteSmem* rs, uint8_t* smem, uint32_t bar_base,
                                         volatile int* abort, int u, int rc, int tile, int nb, int KC, int KG, int TS,
                                         const int (&rbase)[Warps<CW>::MT], int lane, long long& fills) {
  using L = Q4Layout<1, ST, GPU>;
  constexpr int MT = Warps<CW>::MT;
  const int warp = threadIdx.x >> 5, g = lane >> 2, c = lane & 3;
  float acc[MT][1][4];
  zero_acc<MT, 1>(acc);
  for (int kc = 0; kc < KC; ++kc, ++fills) {
    const int s = (int)(fills % ST);
    const uint32_t ph = (uint32_t)((fills / ST) & 1);
    const bool ok = mbar_wait(bar_base + 8 * s, ph, abort, a.err);
    const int gcount = min(GPU, KG - GPU * kc);
    consume_stage<1, CW, L::NB, true, GPU>(smem + s * L::STAGE, smem_addr(smem + L::SX_OFF + s * L::SX_BYTES), gcount,
                                           rbase, lane, acc, ok);
    __syncwarp();
    if (lane == 0) mbar_arrive(bar_base + 8 * (ST + s));
  }
  // pair ids of this thread's columns
  long long pid[1][2];
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    const int b = 2 * c + q;
    int r = 0, j = 0;
    if (b < nb) pair_of(rs, a, u, 8 * rc + b, r, j);
    pid[0][q] = b < nb ? (long long)r * TS + j : -1;
  }
  constexpr int NTC = 1;
  if (GATEUP) {
    if (*abort) return;
#pragma unroll
    for (int t = 0; t < NTC; ++t)
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const long long p = pid[t][q & 1];
        if (p < 0) continue;
        const int i = 64 * tile + 16 * warp + g + 8 * (q >> 1);
        const float gate = acc[0][t][q], up = acc[MT - 1][t][q];
        const float h = gate / (1.f + expf(-gate)) * up;
        a.hbuf[p * a.I + i] = f2bf16(h);
      }
  } else {
#pragma unroll
    for (int m = 0; m < MT; ++m)
#pragma unroll
      for (int t = 0; t < NTC; ++t)
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const long long p = pid[t][q & 1];
          const int n = kBM * tile + rbase[m] + g + 8 * (q >> 1);
          if (p >= 0 && n < a.H) a.part[p * a.H + n] = acc[m][t][q];
        }
  }
}

// y[r][n] = sum_j w[r][j] p[r][j][n] in rank order j, then + sigmoid(shared
// gate logit) x the shared expert's partial: one thread per output, every
// partial loaded before the sum.
__global__ void __launch_bounds__(256) moe_combine_kernel(const MoeArgs a) {
  // Before the dependency wait: the old residual (y += result) and the shared
  // expert's gate logit, written at least two kernels earlier.
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const bool live = i < (long long)a.k * a.H;
  const int r = live ? (int)(i / a.H) : 0, n = live ? (int)(i % a.H) : 0;
  const float yo = live && a.dtype == 2 ? reinterpret_cast<const float*>(a.y)[(long long)r * a.H + n] : 0.f;
  const float sg = live && a.has_shared ? __ldcg(a.shared_logit + (long long)r * a.logits_ld) : 0.f;
  // the kernel after the combine (the next layer's norm) reads only static
  // data before its own wait: it may start now
  griddep_launch();
  griddep_wait();
  if (blockIdx.x == 0) {  // the routed-expert kernel is done: reset its counters and unit counts
    for (int i = threadIdx.x; i < kMoeSchedWords; i += blockDim.x) a.work[i] = 0;
  }
  if (!live) return;
  const int TS = a.T + a.has_shared;
  const float* pr = a.part + (long long)r * TS * a.H + n;
  float v[kMaxTopK], wj[kMaxTopK];
#pragma unroll
  for (int j = 0; j < kMaxTopK; ++j) {
    v[j] = j < a.T ? __ldcg(pr + (long long)j * a.H) : 0.f;
    wj[j] = j < a.T ? __ldcg(a.w_out + r * a.T + j) : 0.f;
  }
  const float vs = a.has_shared ? __ldcg(pr + (long long)a.T * a.H) : 0.f;
  float y = 0.f;
#pragma unroll
  for (int j = 0; j < kMaxTopK; ++j)
    if (j < a.T) y = fmaf(wj[j], v[j], y);
  if (a.has_shared) y = fmaf(1.f / (1.f + expf(-sg)), vs, y);
  if (a.dtype == 2) reinterpret_cast<float*>(a.y)[(long long)r * a.H + n] = yo + y;
  else store_out(a.y, a.dtype, (long long)r * a.H + n, y);
}

// The routed-expert products as one persistent kernel (a second kernel, the
// combine, follows).  Work items:
//   [0, n_gu)         gate/up items (unit v, 64 outputs of I): gate rows and
//                     up rows of the same outputs go to the same warp, the
//                     epilogue applies SwiGLU and writes h (bf16) for the
//                     unit's rows, then counts the item in done[v];
//   [n_gu, n_gu+n_dn) down items (unit v, 128 rows of H): one fp32 partial
//                     per (row, rank); its h rows are read only once
//                     done[v] == I / 64, all gate/up tiles of the unit.
// A unit is (distinct expert or the shared expert, chunk of up to 8 of its
// rows).  Items are unit-major: concurrent CTAs stream consecutive slices of
// one expert.  Gate/up items come in order from one counter, down items from
// a second; a CTA draws from the gate/up counter while it has items, except
// that its first draw may go to the down counter: only the first
// ceil(est / n_sm) CTAs to arrive on an SM start on a gate/up item (est: an
// upper bound of the gate/up item count), so that when gate/up items are
// fewer than the CTAs they fall on distinct SMs.  The first CTA on every SM
// always starts on the gate/up counter.
// Progress without co-residency: a gate/up item waits for nothing.  A down
// item of unit v waits for v's gate/up items; each of those is claimed by a
// CTA that is running (claims happen at run time) or unclaimed.  If one is
// unclaimed, the gate/up counter is not exhausted, and the first CTA of the
// waiting CTA's SM (which arrived before it, so it runs) still draws from
// that counter: it never waits while gate/up items remain.  So every
// gate/up item is eventually claimed and done, and every wait ends, however
// many CTAs are resident (bounded waits besides).
__device__ __forceinline__ void moe_decode(const MoeArgs& a, const RouteSmem* rs, int item, int n_gu, int ntg,
                                           int ntd, bool& gu, int& v, int& u, int& rc, int& tile, int& nb) {
  gu = item < n_gu;
  const int rel = gu ? item : item - n_gu;
  const int nt = gu ? ntg : ntd;
  v = rel / nt;
  tile = rel % nt;
  const int unit = rs->vlist[v];
  u = unit & 0xFFF;
  rc = unit >> 12;
  nb = min(8, pairs_of(rs, a, u) - 8 * rc);
}

__global__ void __launch_bounds__(Warps<kGateUpWarps>::THREADS, kMoeCtasPerSm) moe_kernel(const MoeArgs a) {
  static_assert(kGateUpWarps == kDownWarps, "both item kinds share one CTA shape");
  constexpr int ST = kMoeStages, GPU = kExpertGroups;
  using L = Q4Layout<1, ST, GPU>;
  constexpr int CW = kGateUpWarps, MT = Warps<CW>::MT;
  static_assert(MT == 2, "gate/up pairs the gate and up row tiles in one warp");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t bar_base = smem_addr(smem + L::BAR_OFF);
  volatile int* abort = reinterpret_cast<volatile int*>(smem + L::MISC_OFF);
  volatile int* slot_item = abort + 4;  // item id of the item starting in stage s (-1: no more work)
  RouteSmem* rs = reinterpret_cast<RouteSmem*>(smem + L::BASE_BYTES);
  static_assert(L::BASE_BYTES % 16 == 0, "the routing tables are read with 16-byte loads");
  if (threadIdx.x == 0) *abort = 0;
  init_barriers<CW, ST>(bar_base);
  for (int e = threadIdx.x; e < kMaxExperts; e += blockDim.x) rs->mask[e] = 0u;  // shared memory only
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // The first draw: this CTA's arrival slot on its SM, then the gate/up or
  // the down counter (read as an item once the routes give n_gu).  Issued
  // before the dependency wait, so that the two atomics' latency overlaps it:
  // the scheduling words are touched only by this kernel and its combine,
  // and the combine that last reset them ran at least two kernels back.
  bool first_gu = true;
  int first_raw = 0;
  if (warp == CW && lane == 0) {
    unsigned smid;
    asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
    const int est = (min(a.k * a.T, a.E) + a.has_shared) * (a.I / 64);
    if (smid < (unsigned)kMoeSmSlots) first_gu = (long long)atomicAdd(a.work + 2 + smid, 1) * a.n_sm < est;
    first_raw = atomicAdd(a.work + (first_gu ? 0 : 1), 1);
  }
  griddep_wait();  // the routes come from the routing kernel before
  griddep_launch();
  load_routes(a.idx_out, a.T, a.k, a.has_shared, rs);  // ends with __syncthreads

  const int TS = a.T + a.has_shared;
  const int ntg = a.I / 64, ntd = (a.H + kBM - 1) / kBM;
  const int n_gu = rs->V * ntg, n_all = n_gu + rs->V * ntd;
  const int KGg = a.H / 64, KCg = (KGg + GPU - 1) / GPU;
  const int KGd = a.I / 64, KCd = (KGd + GPU - 1) / GPU;

  if (warp == CW) {
    // ------------------------------------------------------------ producer
    const uint16_t** brow = reinterpret_cast<const uint16_t**>(smem + L::MISC_OFF + 64);
    long long fills = 0;
    // lane 0 draws; gu_open: the gate/up counter may still hold items
    bool gu_open = true;
    int next = 0;
    if (lane == 0) {
      if (!first_gu) {
        next = n_gu + first_raw;
      } else if (first_raw < n_gu) {
        next = first_raw;
      } else {
        gu_open = false;
        next = n_gu + atomicAdd(a.work + 1, 1);
      }
    }
    next = __shfl_sync(0xffffffffu, next, 0);
    for (;;) {
      const int item = next;
      const int s0 = (int)(fills % ST);
      if (!mbar_wait(bar_base + 8 * (ST + s0), (uint32_t)(((fills / ST) & 1) ^ 1), abort, a.err)) break;
      if (item >= n_all || *abort) {
        // end mark: a stage without data whose item id tells the consumers to stop
        if (lane == 0) {
          slot_item[s0] = -1;
          mbar_arrive_expect_tx(bar_base + 8 * s0, 0);
        }
        cp_async_mbar_arrive_noinc(bar_base + 8 * s0);
        ++fills;
        break;
      }
      bool gu;
      int v, u, rc, tile, nb;
      moe_decode(a, rs, item, n_gu, ntg, ntd, gu, v, u, rc, tile, nb);
      const bool shared = u >= rs->U;
      const int e = shared ? 0 : rs->ulist[u];
      __syncwarp();
      if (lane < L::NB) {
        int r = 0, j = 0;
        if (lane < nb) pair_of(rs, a, u, 8 * rc + lane, r, j);
        brow[lane] = gu ? a.x + (long long)r * a.H : a.hbuf + ((long long)r * TS + j) * a.I;
      }
      __syncwarp();
      const uint8_t* ts =
          gu ? (shared ? a.sgu_tiles : a.gu_tiles + (long long)e * ntg * a.gu_rt_bytes) + tile * a.gu_rt_bytes
             : (shared ? a.sdn_tiles : a.dn_tiles + (long long)e * ntd * a.dn_rt_bytes) + tile * a.dn_rt_bytes;
      const int KG = gu ? KGg : KGd, KC = gu ? KCg : KCd;
      int kc = 0;
      if (!gu) {
        int ok = 1;
        if (lane == 0) ok = wait_count(a.done + v, ntg, abort, a.err);
        if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      }
      for (; kc < KC; ++kc, ++fills) {
        const int s = (int)(fills % ST);
        const uint32_t ph = (uint32_t)((fills / ST) & 1);
        if (kc > 0 && !mbar_wait(bar_base + 8 * (ST + s), ph ^ 1, abort, a.err)) break;
        if (kc == 0 && lane == 0) slot_item[s] = item;
        produce_stage<1, GPU>(smem + s * L::STAGE, bar_base + 8 * s, ts, kc, min(GPU, KG - GPU * kc), brow, nb,
                              lane);
      }
      // The next item, fetched once this item's stages are all issued: an
      // atomic still in flight would hold up this lane's next barrier arrival
      // (a release).  Gate/up items first, while there are any.
      if (lane == 0) {
        int i = n_gu;
        if (gu_open) {
          i = atomicAdd(a.work, 1);
          gu_open = i < n_gu;
        }
        next = i < n_gu ? i : n_gu + atomicAdd(a.work + 1, 1);
      }
      next = __shfl_sync(0xffffffffu, next, 0);
      if (*abort) break;
    }
    if (*abort) producer_drain<ST>(bar_base, fills);
    return;
  }

  // -------------------------------------------------------------- consumers
  long long fills = 0;
  for (;;) {
    const int s = (int)(fills % ST);
    if (!mbar_wait(bar_base + 8 * s, (uint32_t)((fills / ST) & 1), abort, a.err)) break;
    const int item = slot_item[s];
    if (item < 0) break;
    bool gu;
    int v, u, rc, tile, nb;
    moe_decode(a, rs, item, n_gu, ntg, ntd, gu, v, u, rc, tile, nb);
    if (gu) {
      const int rbase[MT] = {16 * warp, 64 + 16 * warp};
      moe_item<CW, true, ST, GPU>(a, rs, smem, bar_base, abort, u, rc, tile, nb, KCg, KGg, TS, rbase, lane, fills);
      // publish this tile of the unit's h rows
      named_bar(3, CW * 32);
      if (threadIdx.x == 0) {
        __threadfence();
        atomicAdd(a.done + v, 1);
      }
    } else {
      const int rbase[MT] = {16 * (warp * MT), 16 * (warp * MT + 1)};
      moe_item<CW, false, ST, GPU>(a, rs, smem, bar_base, abort, u, rc, tile, nb, KCd, KGd, TS, rbase, lane, fills);
    }
  }
}

// ================================================================ launchers

template <int NT>
static size_t dense_smem() { return Q4Layout<NT>::BASE_BYTES + 1024; }
template <int NT>
static size_t moe_smem() { return Q4Layout<NT, kMoeStages, kExpertGroups>::BASE_BYTES + sizeof(RouteSmem) + 1024; }

template <typename F>
static cudaError_t setup_one(F* kernel, int threads, size_t smem, int* ctas_per_sm) {
  cudaError_t e;
  if ((e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem))) return e;
  if ((e = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                (int)cudaSharedmemCarveoutMaxShared)))
    return e;
  int n = 0;
  if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, threads, smem))) return e;
  *ctas_per_sm = n < *ctas_per_sm ? n : *ctas_per_sm;
  return cudaSuccess;
}

// Sets the launch attributes of every Q4 kernel and reports how many CTAs of
// the dense and of the MoE kernels fit on one SM (the minimum over the two
// tile widths, so that the grid - and with it the split of K across CTAs -
// does not depend on k).
cudaError_t q4_setup_kernels(int* dense_ctas_per_sm, int* moe_ctas_per_sm) {
  cudaError_t e;
  constexpr int TD = Warps<kDenseWarps>::THREADS, TG = Warps<kGateUpWarps>::THREADS;
  *dense_ctas_per_sm = kQ4CtasPerSm;
  if ((e = setup_one(q4_dense_kernel<1>, TD, dense_smem<1>(), dense_ctas_per_sm))) return e;
  if ((e = setup_one(q4_dense_kernel<2>, TD, dense_smem<2>(), dense_ctas_per_sm))) return e;
  // clusters of up to 16 CTAs (sizes above 8 are not portable)
  if ((e = cudaFuncSetAttribute(q4_dense_kernel<1>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1))) return e;
  if ((e = cudaFuncSetAttribute(q4_dense_kernel<2>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1))) return e;
  // the argmax-epilogue instances (LM head): same shape, their occupancy checked alike
  int argmax_ctas = kQ4CtasPerSm;
  if ((e = setup_one(q4_dense_kernel<1, true>, TD, dense_smem<1>(), &argmax_ctas))) return e;
  if ((e = setup_one(q4_dense_kernel<2, true>, TD, dense_smem<2>(), &argmax_ctas))) return e;
  if ((e = cudaFuncSetAttribute(q4_dense_kernel<1, true>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1)))
    return e;
  if ((e = cudaFuncSetAttribute(q4_dense_kernel<2, true>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1)))
    return e;
  if (argmax_ctas < *dense_ctas_per_sm) return cudaErrorInvalidConfiguration;
  *moe_ctas_per_sm = kMoeCtasPerSm;
  if ((e = setup_one(moe_kernel, TG, moe_smem<1>(), moe_ctas_per_sm))) return e;
  if (*dense_ctas_per_sm < 1 || *moe_ctas_per_sm < 1) return cudaErrorInvalidConfiguration;
  return cudaSuccess;
}

// For every cluster size S = 1 .. kMaxSplits: how many clusters of S dense
// CTAs the GPU runs at once (the smaller of the two column-block widths, so
// that the split of K, chosen from it, does not depend on k).
cudaError_t q4_dense_cluster_limits(int* max_clusters) {
  constexpr int TD = Warps<kDenseWarps>::THREADS;
  max_clusters[0] = 0;
  for (int S = 1; S <= kMaxSplits; ++S) {
    int best = 1 << 30;
    for (int nt = 1; nt <= 2; ++nt) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(S * 64);
      cfg.blockDim = dim3(TD);
      cfg.dynamicSmemBytes = nt == 1 ? dense_smem<1>() : dense_smem<2>();
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = S;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      int n = 0;
      cudaError_t e = nt == 1 ? cudaOccupancyMaxActiveClusters(&n, q4_dense_kernel<1>, &cfg)
                              : cudaOccupancyMaxActiveClusters(&n, q4_dense_kernel<2>, &cfg);
      if (e && S > 8) {  // a GPU without clusters this large: never chosen
        (void)cudaGetLastError();
        n = 0;
      } else if (e) {
        return e;
      }
      best = n < best ? n : best;
    }
    max_clusters[S] = best;
  }
  return cudaSuccess;
}

cudaError_t launch_q4_dense(const DenseArgs& a, int nt, bool pdl, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.RB * a.S);
  cfg.blockDim = dim3(Warps<kDenseWarps>::THREADS);
  cfg.dynamicSmemBytes = nt == 1 ? dense_smem<1>() : dense_smem<2>();
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = a.S;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 2 : 1;
  if (nt == 1) return cudaLaunchKernelEx(&cfg, q4_dense_kernel<1>, a);
  return cudaLaunchKernelEx(&cfg, q4_dense_kernel<2>, a);
}

cudaError_t launch_q4_dense_argmax(const DenseArgs& a, int nt, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.RB * a.S);
  cfg.blockDim = dim3(Warps<kDenseWarps>::THREADS);
  cfg.dynamicSmemBytes = nt == 1 ? dense_smem<1>() : dense_smem<2>();
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = a.S;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (nt == 1) return cudaLaunchKernelEx(&cfg, q4_dense_kernel<1, true>, a);
  return cudaLaunchKernelEx(&cfg, q4_dense_kernel<2, true>, a);
}

// Three kernels: the routing kernel (after everything the caller enqueued
// before it, or, with pdl, during the tail of the kernel before it), then the
// routed-expert kernel and the combine, each a programmatic dependent of the
// kernel before it.  The expert kernel's first draw, before its dependency
// wait, touches scheduling words that the previous call's combine reset: that
// combine ran before the routing kernel, two kernels back.
cudaError_t launch_moe(const MoeArgs& a, bool pdl, cudaStream_t s, int* launches) {
  cudaLaunchAttribute pdl_attr[1];
  pdl_attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl_attr[0].val.programmaticStreamSerializationAllowed = 1;
  {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1);
    cfg.blockDim = dim3(32 * a.k);
    cfg.stream = s;
    cfg.attrs = pdl_attr;
    cfg.numAttrs = pdl ? 1 : 0;
    cudaError_t e = cudaLaunchKernelEx(&cfg, moe_route_kernel, a);
    if (e) return e;
    ++*launches;
  }
  {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(a.G);
    cfg.blockDim = dim3(Warps<kGateUpWarps>::THREADS);
    cfg.dynamicSmemBytes = moe_smem<1>();
    cfg.stream = s;
    cfg.attrs = pdl_attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, moe_kernel, a);
    if (e) return e;
    ++*launches;
  }
  cudaError_t e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(((long long)a.k * a.H + 255) / 256));
  cfg.blockDim = dim3(256);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, moe_combine_kernel, a);
  if (!e) ++*launches;
  return e;
}

}  // namespace vk
