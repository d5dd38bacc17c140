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
constexpr int kQ4CtasPerSm = 2;
constexpr int kMaxExperts = 512;
constexpr int kMaxTopK = 16;

// Dense product: RB row tiles x S K-splits, one cluster of S CTAs per tile.
struct DenseArgs {
  const uint16_t* scales;
  const uint16_t* biases;
  const uint16_t* x;  // [k, K] bf16
  void* y;            // [k, N]
  int* err;
  int N, K, k, dtype;
  int KG, KC, RB;     // groups per row, 256-column chunks per row, 128-row tiles
  int S;              // K-splits per tile (cluster size, 1..8)
};

// Routed experts.  Both kernels recompute the (cheap, deterministic) routing.
struct MoeArgs {
  const float* logits;
  long long logits_ld;
  const float* shared_logit;  // NULL: no shared expert
  const uint16_t* x;          // [k, H]
  const uint16_t* gu_scales;  // [E, 2I, H/64]
  const uint16_t* gu_biases;
  const uint16_t* dn_scales;  // [E, H, I/64]
  const uint16_t* dn_biases;
  const uint16_t* sgu_scales; // shared [2I, H/64]
  const uint16_t* sgu_biases;
  const uint16_t* sdn_scales; // shared [H, I/64]
  const uint16_t* sdn_biases;
  uint16_t* hbuf;             // scratch [k, TS, I] bf16 (TS = T + has_shared)
  float* part;                // scratch [k, TS, H] fp32
  int32_t* idx_out;
  float* w_out;
  void* y;
  int* err;
  int E, T, H, I, k, dtype;
  int has_shared;
  int G;
};

struct GdnArgs {
  const float* S_in;          // [Hv, dv, dk]
  const uint16_t* tail_in;    // [W-1, C]
  float* S_out[17];           // slot receiving the state after row r (r < k)
  uint16_t* tail_out[17];
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
// pdl: launch with programmatic stream serialization (the kernel may start
// while the previous kernel on the stream runs; see griddep_wait).
cudaError_t launch_q4_dense(const CUtensorMap& wmap, const DenseArgs& a, int nt, bool pdl, cudaStream_t s);
cudaError_t launch_moe(const CUtensorMap& gu_map, const CUtensorMap& dn_map, const CUtensorMap& sgu_map,
                       const CUtensorMap& sdn_map, const MoeArgs& a, int nt, bool pdl, cudaStream_t s,
                       int* launches);
cudaError_t gdn_setup_kernels();
cudaError_t launch_gdn(const GdnArgs& a, bool pdl, cudaStream_t s);
cudaError_t launch_rmsnorm(const float* x, const float* w, float eps, int zc, int n, int k, void* out,
                           int dtype, bool pdl, cudaStream_t s);

}  // namespace vk
