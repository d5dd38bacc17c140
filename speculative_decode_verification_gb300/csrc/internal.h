// internal.h - declarations shared by the library's translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace vk {

// Q4 engine geometry (see q4_kernels.cu).
constexpr int kBM = 128;           // weight rows per tile
constexpr int kGroupsPerUnit = 4;  // 64-column groups per pipeline stage (256 columns)
constexpr int kStages = 4;         // pipeline depth
constexpr int kDenseWarps = 4;     // consumer warps of the dense kernel: two 16-row MMA tiles each
constexpr int kGateUpWarps = 4;    // fused gate/up: a gate tile and its up tile per warp
constexpr int kDownWarps = 4;      // routed down projection: two 16-row MMA tiles each
constexpr int kQ4CtasPerSm = 2;    // dense kernels
constexpr int kMaxSplits = 16;      // K-splits of a dense row tile (one cluster; 16 = largest non-portable size)
constexpr int kMoeCtasPerSm = 4;   // routed-expert kernel: 8 activation rows per stage, four stages
constexpr int kMoeStages = 4;
constexpr int kExpertGroups = 2;   // routed experts: 64-column groups per stage (128 columns)
constexpr int kMoeUnits = 2 * 512 + 2;  // work units of one call: (expert, chunk of 8 rows), at most
constexpr int kMoeSmSlots = 256;        // per-SM arrival counters of the routed-expert kernel (SM ids below this)
// Scheduling words of the routed-expert kernel, zero between calls: the
// gate/up item counter, the down item counter, one arrival counter per SM,
// then one gate/up tile count per unit.
constexpr int kMoeSchedWords = 2 + kMoeSmSlots + kMoeUnits;
constexpr int kMaxExperts = 512;
constexpr int kMaxTopK = 16;

// Tiled weight layouts (tile.cu): per (128-row tile, chunk of G 64-column
// groups) a block of scales and biases followed by the chunk's groups of
// codes.  Dense matrices: G = kGroupsPerUnit (256 columns); routed and shared
// experts: G = kExpertGroups (128 columns).
constexpr int kTileGroupBytes = kBM * 32;                                 // 4096: 128 rows x 64 codes
__host__ __device__ constexpr int tile_sb_bytes(int groups) { return 2 * kBM * 2 * groups; }
__host__ __device__ constexpr int tile_chunk_bytes(int groups) {
  return tile_sb_bytes(groups) + groups * kTileGroupBytes;
}
constexpr int kTileSbBytes = tile_sb_bytes(kGroupsPerUnit);               // 2048
constexpr int kTileChunkBytes = tile_chunk_bytes(kGroupsPerUnit);         // 18432
// Groups per chunk of a tiled layout (verify_q4_layout), 0 if not tiled.
__host__ __device__ constexpr int layout_groups(int layout) {
  return layout == 1 ? kGroupsPerUnit : (layout == 2 || layout == 3) ? kExpertGroups : 0;
}
// Bytes of one 128-row tile of a tiled matrix with k_in columns.
__host__ __device__ constexpr long long tile_row_bytes(int k_in, int groups) {
  return (long long)tile_sb_bytes(groups) * ((k_in / 64 + groups - 1) / groups) + (long long)kTileGroupBytes * (k_in / 64);
}

// Dense product: RB row tiles x S K-splits, one cluster of S CTAs per tile.
struct DenseArgs {
  const uint8_t* tiles;  // tiled weights
  long long rt_bytes;    // bytes of one row tile
  const uint16_t* x;     // [k, K] bf16
  void* y;            // [k, N]
  int* err;
  int N, K, k, dtype;
  int KG, KC, RB;     // groups per row, 256-column chunks per row, 128-row tiles
  int S;              // K-splits per tile (cluster size, 1..16)
  // Argmax epilogue (the LM head's greedy choice; y unused): per output
  // column r (block row r0 + r) the 64-bit argmax key over the N outputs is
  // merged into best[r0 + r] (zero before the first pass).
  unsigned long long* best;
  int r0;
};

// Routed experts: the routing kernel, the expert kernel and the combine.
struct MoeArgs {
  const float* logits;
  long long logits_ld;
  const float* shared_logit;  // NULL: no shared expert
  const uint16_t* x;          // [k, H]
  const uint8_t* gu_tiles;    // tiled [E, 2I, H], gate/up pairing: I/64 row tiles per expert
  const uint8_t* dn_tiles;    // tiled [E, H, I]: ceil(H/128) row tiles per expert
  const uint8_t* sgu_tiles;   // shared expert, same layouts (NULL: none)
  const uint8_t* sdn_tiles;
  long long gu_rt_bytes, dn_rt_bytes;
  uint16_t* hbuf;             // scratch [k, TS, I] bf16 (TS = T + has_shared)
  float* part;                // scratch [k, TS, H] fp32
  int* work;                  // scratch [kMoeSchedWords] (zero before a call; the combine kernel resets it):
                              // gate/up counter, down counter, per-SM arrivals, then the unit counts
  int* done;                  // = work + 2 + kMoeSmSlots: gate/up tiles written per unit
  int32_t* idx_out;
  float* w_out;
  void* y;
  int* err;
  int E, T, H, I, k, dtype;
  int has_shared;
  int G;                      // CTAs of the routed-expert kernel
  int n_sm;                   // SMs of the GPU
};

// CTAs per SM of the routed-expert grid: three when an upper bound of the
// gate/up items fits one wave of four per SM (fewer CTAs per SM stream
// faster each), else all that fit (more CTAs shorten the waves of large
// expert sets).  The grid changes no result: an item's arithmetic is the same
// on any CTA.
inline int moe_ctas_per_sm_for(int k, int top_k, int E, int has_shared, int I, int num_sms, int max_per_sm) {
  const int est = ((k * top_k < E ? k * top_k : E) + has_shared) * (I / 64);
  return est <= 4 * num_sms && max_per_sm > 3 ? 3 : max_per_sm;
}

// Shape rules of the routed-expert call, shared by q4_gather_experts_k and
// its no-allocation twin so that both accept the same calls: 0 (fine) or the
// verify_status to return, with a message.
int moe_shape_status(int k, int max_k, int E_gate_up, int E_down, int top_k, int gu_n_out, int gu_k_in,
                     int dn_n_out, int dn_k_in, const char** msg);

// State slots: S_slots[s] fp32 [Hv, dv, dk], tail_slots[s] bf16 [W-1, C].  The
// kernel reads slot cur and writes the state after row r to slot r + (r >= cur),
// the r+1-th slot other than cur in ascending order (r counted from the
// block's first row: a launch with r0 > 0 continues from the slot of row r0-1).  cur is the argument, or,
// with dev_state, dev_state[0] read when the kernel runs (written by a device
// commit at least two launches earlier); the kernel then stores k in
// dev_state[1] (the rows now pending).
struct GdnArgs {
  float* S_slots[33];
  uint16_t* tail_slots[33];
  int n_slots, cur;
  int* dev_state;
  int r0;  // block row of this launch's first row: it starts from the state after r0 rows
  const uint16_t* qkv; long long ld_qkv;
  const uint16_t* z;   long long ld_z;
  const uint16_t* a;   long long ld_a;
  const uint16_t* b;   long long ld_b;
  const float* conv_w;
  const float* A_log;
  const float* dt_bias;
  const float* norm_w;
  void* o;
  int* err;
  int Hk, Hv, d, W, k, dtype, gate_act;
  float q_scale, l2_eps, norm_eps;
};

// Launchers (return the first CUDA error; *launches counts kernels launched).
cudaError_t q4_setup_kernels(int* dense_ctas_per_sm, int* moe_ctas_per_sm);
// max_clusters[S], S = 1 .. kMaxSplits: dense-kernel clusters of S CTAs resident at once.
cudaError_t q4_dense_cluster_limits(int* max_clusters);
// pdl: launch with programmatic stream serialization (the kernel may start
// while the previous kernel on the stream runs; see griddep_wait).
cudaError_t launch_q4_dense(const DenseArgs& a, int nt, bool pdl, cudaStream_t s);
// The same product with the argmax epilogue (one pass of up to 16 rows).
cudaError_t launch_q4_dense_argmax(const DenseArgs& a, int nt, cudaStream_t s);
cudaError_t launch_moe(const MoeArgs& a, bool pdl, cudaStream_t s, int* launches);
// Tiled layouts: bytes of E matrices [N, K] of a tile kind (0 dense, 1
// gate/up: tiles pair gate and up rows, 2 expert down), and the conversion
// from the row-major layout.
long long tiled_bytes(int N, int K, int E, int kind);
cudaError_t launch_tile(const uint32_t* packed, const uint16_t* scales, const uint16_t* biases, uint8_t* dst, int N,
                        int K, int E, int kind, cudaStream_t s);
cudaError_t gdn_setup_kernels();
// One kernel whose two bounded waits (a barrier and a counter that nothing
// completes) run out and record VERIFY_DEV_ETIMEOUT in *err.
cudaError_t launch_stuck_wait_probe(int* err, cudaStream_t s);
cudaError_t launch_gdn(const GdnArgs& a, bool pdl, cudaStream_t s);
cudaError_t launch_rmsnorm(const float* x, const float* w, float eps, int zc, int n, int k, void* out,
                           int dtype, bool pdl, cudaStream_t s);

// Width-k grouped-query attention over a binary16 KV cache: append (the
// block's rotated keys and values into the cache, the rotation table), split
// partials (one CTA per (M group, key split, KV head)), combine.
struct AttnArgs {
  // tensor maps of the K and V caches for the split kernel's tile loads (set
  // by the launcher): {D, P + k, Hkv} binary16, boxes of 64 x 64 x 1,
  // 128-byte swizzle, zeros past P + k
  CUtensorMap tm_k, tm_v;
  // tensor maps of the queries' lo and hi parts for the same kernel:
  // {D, Hkv * q_rows} binary16, boxes of 64 x 128, 128-byte swizzle
  CUtensorMap tm_ql, tm_qh;
  const uint16_t* q;    long long ld_q;
  const uint16_t* gate; long long ld_gate;
  const uint16_t* kin;  long long ld_k;
  const uint16_t* vin;  long long ld_v;
  uint16_t* K;          // [Hkv, cap, D]
  uint16_t* V;
  long long cap;
  int Hq, Hkv, D, rope_dim;
  double inv_freq[128];  // theta^(-2j / rope_dim), j < rope_dim / 2, computed on the host in float64
  double qscale;         // log2(e) / sqrt(D): scores in log2 units
  int P, k, split;
  int nsplit;           // ceil((P + k) / split)
  int n_mtiles;         // ceil(k * Hq / Hkv / 16): 16 (row, head) pairs per tile
  int q_rows;           // query rows per KV head: k * Hq / Hkv rounded up to 128
  uint16_t* qh;         // [Hkv][q_rows][D] binary16: rotated, scaled queries (hi part), row r * G + g
                        // of KV head h for query head h * G + g of block row r (rows past k * G unused)
  uint16_t* ql;         // the remainders (lo part), same layout
  float* part_o;        // [Hkv][nsplit][16 n_mtiles][D] unnormalised outputs
  float2* part_ml;      // [Hkv][nsplit][16 n_mtiles] (running max in log2 units, sum)
  void* o;              // [k, Hq * D]
  int dtype;
  int* err;             // device error word (a pipeline wait that ran out)
};
constexpr int kAttnMaxM = 512;   // k * (Hq / Hkv) per call
cudaError_t attn_setup_kernels();
cudaError_t launch_attn(const AttnArgs& a, cudaStream_t s, int* launches);

// Greedy acceptance fused with the device commit (V > 0), the device commit
// alone of the accepted count *accepted (V == 0, one CTA), or the acceptance
// and commit from keys already merged in best (V < 0, one CTA: after the LM
// head's argmax epilogue).
struct AcceptArgs {
  const float* logits;        // [k, V], row r at logits + r * ld
  long long ld;
  int V, k;
  int vec;                    // rows are 16-byte aligned: float4 loads
  int blocks_per_row;
  const int* draft;           // [k-1]
  int* result;                // [2 + k]
  const int* accepted;        // V == 0: the accepted row count
  int* dev_state;             // [n_states][2] {committed slot, pending rows}
  int n_states;
  int need_k;                 // > 0: every state's pending rows must equal it
  unsigned long long* best;   // scratch [kMaxAcceptK], zero between calls
  unsigned int* ticket;       // scratch, zero between calls
  int* err;
};
constexpr int kMaxAcceptK = 32;
constexpr int kAcceptThreads = 256;
// Grid of the acceptance kernel: CTAs per logits row.
int accept_blocks_per_row(int V, int k, int num_sms);
cudaError_t launch_accept(const AcceptArgs& a, cudaStream_t s);

}  // namespace vk
