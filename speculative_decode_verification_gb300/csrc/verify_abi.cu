// verify_abi.cu - the C ABI declared in include/verify.h: context and scratch,
// argument validation (all done before anything is launched), TMA
// descriptors, launches on the caller's stream, GDN slot bookkeeping.
#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <vector>

#include "internal.h"
#include "verify.h"

struct verify_ctx {
  int device = 0;
  int num_sms = 0;
  int dense_ctas_per_sm = 0;
  int dense_max_clusters[vk::kMaxSplits + 1] = {};  // clusters of S dense CTAs resident at once
  int moe_ctas_per_sm = 0;
  uint16_t* moe_hbuf = nullptr;
  float* moe_part = nullptr;
  int* err = nullptr;
  int* moe_sched = nullptr;  // routed-expert scheduling words (vk::kMoeSchedWords), zero between calls
  uint16_t* st_xn = nullptr;   // layer scratch: bf16 [16, 8192]
  uint16_t* st_proj = nullptr; // bf16 [16, 32768]
  uint16_t* st_o = nullptr;    // bf16 [16, 32768]
  float* st_logits = nullptr;  // fp32 [16, 1024]
  int32_t* st_idx = nullptr;   // [16, 16]
  float* st_w = nullptr;       // [16, 16]
  unsigned long long* acc_best = nullptr;  // greedy acceptance: per-row argmax keys, then the ticket
  unsigned int* acc_ticket = nullptr;
  int64_t launches = 0;
  cudaEvent_t layer_events[8] = {};
  int n_layer_events = 0;
  // Set only inside verify_layer_k: the next launch may start while the
  // kernel before it on the stream still runs (programmatic dependent launch).
  bool pdl = false;
  // Set by verify_stack_k for layers after the first: the layer's first kernel
  // may overlap the previous layer's last one (it reads only static data
  // before its dependency wait).
  bool chain_layer = false;
  char msg[512] = {0};
};

namespace {

constexpr int kMaxN = 1 << 20;
constexpr int kMaxKin = 1 << 17;
constexpr int kMaxH = 8192;
constexpr int kMaxI = 4096;
constexpr int kMaxProj = 32768;
constexpr size_t kHbufElems = (size_t)VERIFY_MAX_K * (vk::kMaxTopK + 1) * kMaxI;
constexpr size_t kMoePartElems = (size_t)VERIFY_MAX_K * (vk::kMaxTopK + 1) * kMaxH;

verify_status fail(verify_ctx* ctx, verify_status st, const char* fmt, const char* what = "") {
  if (ctx) snprintf(ctx->msg, sizeof ctx->msg, fmt, what);
  return st;
}

verify_status cuda_fail(verify_ctx* ctx, cudaError_t e, const char* where) {
  if (ctx) snprintf(ctx->msg, sizeof ctx->msg, "%s: %s", where, cudaGetErrorString(e));
  return VERIFY_ECUDA;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// true if p is device (or managed) memory that this GPU can use
bool is_device_ptr(const void* p) {
  if (!p) return false;
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged;
}

verify_status check_dev(verify_ctx* ctx, const void* p, size_t align, const char* name) {
  if (!p) return fail(ctx, VERIFY_EINVAL, "%s is NULL", name);
  if (!aligned(p, align)) return fail(ctx, VERIFY_EINVAL, "%s is misaligned", name);
  if (!is_device_ptr(p)) return fail(ctx, VERIFY_EINVAL, "%s is not device memory", name);
  return VERIFY_OK;
}

verify_status use_device(verify_ctx* ctx) {
  int cur = -1;
  cudaError_t e = cudaGetDevice(&cur);
  if (e) return cuda_fail(ctx, e, "cudaGetDevice");
  if (cur != ctx->device && (e = cudaSetDevice(ctx->device))) return cuda_fail(ctx, e, "cudaSetDevice");
  return VERIFY_OK;
}

bool valid_shape(int32_t n_out, int32_t k_in) {
  return n_out >= 1 && n_out <= kMaxN && k_in >= 64 && k_in % 64 == 0 && k_in <= kMaxKin;
}

// A compute operand: tiled layout (`layout`), in device memory.
verify_status check_q4(verify_ctx* ctx, const verify_q4_weight* W, const char* name, int layout = VERIFY_Q4_TILED) {
  if (!W) return fail(ctx, VERIFY_EINVAL, "%s is NULL", name);
  if (W->group_size != 64 || W->bits != 4) return fail(ctx, VERIFY_EUNSUPPORTED, "%s: only 4-bit, group 64", name);
  if (W->layout != layout)
    return fail(ctx, VERIFY_EINVAL,
                layout == VERIFY_Q4_TILED_GATE_UP ? "%s: expected the gate/up tiled layout (q4_tile, VERIFY_TILE_GATE_UP)"
                : layout == VERIFY_Q4_TILED_DOWN  ? "%s: expected the expert down layout (q4_tile, VERIFY_TILE_DOWN)"
                                                  : "%s: expected the dense tiled layout (q4_tile, VERIFY_TILE_DENSE)",
                name);
  if (!valid_shape(W->n_out, W->k_in))
    return fail(ctx, VERIFY_EUNSUPPORTED, "%s: n_out in 1..2^20, k_in a multiple of 64 in [64, 131072]", name);
  if (layout == VERIFY_Q4_TILED_GATE_UP && W->n_out % 128 != 0)
    return fail(ctx, VERIFY_EUNSUPPORTED, "%s: gate/up rows must be 2I with I a multiple of 64", name);
  return check_dev(ctx, W->packed, 16, name);
}

// bytes of one 128-row tile of a matrix with k_in columns in the dense layout
long long rt_bytes(int k_in) { return vk::tile_row_bytes(k_in, vk::kGroupsPerUnit); }

// K-splits per row tile: the largest S (at most 16, the largest cluster,
// and at most one split per 256-column chunk) whose RB clusters of S CTAs all
// run at once on this GPU (one wave), by the occupancy of clusters of that
// size.  Depends only on the matrix shape and the GPU.
int dense_splits(const verify_ctx* ctx, int RB, int KC) {
  int S = 1;
  for (int s = 2; s <= vk::kMaxSplits && s <= KC; ++s)
    if (RB <= ctx->dense_max_clusters[s]) S = s;
  return S;
}

verify_status check_dtype(verify_ctx* ctx, int dtype, bool allow_add) {
  if (dtype == VERIFY_F32 || dtype == VERIFY_BF16 || (allow_add && dtype == VERIFY_F32_ADD)) return VERIFY_OK;
  return fail(ctx, VERIFY_EINVAL, "unsupported dtype_out%s", "");
}

}  // namespace

namespace vk {

int moe_shape_status(int k, int max_k, int E_gate_up, int E_down, int top_k, int gu_n_out, int gu_k_in,
                     int dn_n_out, int dn_k_in, const char** msg) {
  if (k < 1 || k > max_k) {
    *msg = max_k == VERIFY_PASS_K ? "k must be in 1..16%s" : "k must be in 1..32%s";
    return VERIFY_EUNSUPPORTED;
  }
  if (E_gate_up < 1 || E_gate_up > kMaxExperts || E_down != E_gate_up) {
    *msg = "n_experts must match and be in 1..512%s";
    return VERIFY_EUNSUPPORTED;
  }
  if (top_k < 1 || top_k > kMaxTopK || top_k > E_gate_up) {
    *msg = "top_k out of range%s";
    return VERIFY_EUNSUPPORTED;
  }
  const int H = gu_k_in, I = gu_n_out / 2;
  if (gu_n_out != 2 * I || dn_n_out != H || dn_k_in != I) {
    *msg = "expert shapes must be gate_up [2I, H], down [H, I]%s";
    return VERIFY_EINVAL;
  }
  if (H > kMaxH || I > kMaxI || I % 64 != 0) {
    *msg = "H <= 8192, I <= 4096, multiples of 64%s";
    return VERIFY_EUNSUPPORTED;
  }
  return VERIFY_OK;
}

}  // namespace vk

extern "C" {

verify_status verify_init(int device, verify_ctx** out) {
  if (!out) return VERIFY_EINVAL;
  *out = nullptr;
  cudaError_t e = cudaSetDevice(device);
  if (e) return VERIFY_ECUDA;
  verify_ctx* ctx = new verify_ctx();
  ctx->device = device;
  auto bail = [&](cudaError_t err) {
    verify_destroy(ctx);
    (void)err;
    return VERIFY_ECUDA;
  };
  if ((e = cudaDeviceGetAttribute(&ctx->num_sms, cudaDevAttrMultiProcessorCount, device))) return bail(e);
  if ((e = cudaMalloc(&ctx->moe_hbuf, kHbufElems * sizeof(uint16_t)))) return bail(e);
  if ((e = cudaMalloc(&ctx->moe_part, kMoePartElems * sizeof(float)))) return bail(e);
  if ((e = cudaMalloc(&ctx->err, sizeof(int)))) return bail(e);
  if ((e = cudaMalloc(&ctx->moe_sched, vk::kMoeSchedWords * sizeof(int)))) return bail(e);
  if ((e = cudaMemset(ctx->moe_sched, 0, vk::kMoeSchedWords * sizeof(int)))) return bail(e);
  if ((e = cudaMalloc(&ctx->st_xn, sizeof(uint16_t) * VERIFY_MAX_K * kMaxH))) return bail(e);
  if ((e = cudaMalloc(&ctx->st_proj, sizeof(uint16_t) * VERIFY_MAX_K * kMaxProj))) return bail(e);
  if ((e = cudaMalloc(&ctx->st_o, sizeof(uint16_t) * VERIFY_MAX_K * kMaxProj))) return bail(e);
  if ((e = cudaMalloc(&ctx->st_logits, sizeof(float) * VERIFY_MAX_K * 1024))) return bail(e);
  if ((e = cudaMalloc(&ctx->st_idx, sizeof(int32_t) * VERIFY_MAX_K * vk::kMaxTopK))) return bail(e);
  if ((e = cudaMalloc(&ctx->st_w, sizeof(float) * VERIFY_MAX_K * vk::kMaxTopK))) return bail(e);
  if ((e = cudaMemset(ctx->err, 0, sizeof(int)))) return bail(e);
  if ((e = cudaMalloc(&ctx->acc_best, sizeof(unsigned long long) * (vk::kMaxAcceptK + 1)))) return bail(e);
  if ((e = cudaMemset(ctx->acc_best, 0, sizeof(unsigned long long) * (vk::kMaxAcceptK + 1)))) return bail(e);
  ctx->acc_ticket = reinterpret_cast<unsigned int*>(ctx->acc_best + vk::kMaxAcceptK);
  if ((e = vk::q4_setup_kernels(&ctx->dense_ctas_per_sm, &ctx->moe_ctas_per_sm))) return bail(e);
  if ((e = vk::q4_dense_cluster_limits(ctx->dense_max_clusters))) return bail(e);
  if ((e = vk::gdn_setup_kernels())) return bail(e);
  if ((e = vk::attn_setup_kernels())) return bail(e);
  if ((e = cudaDeviceSynchronize())) return bail(e);
  *out = ctx;
  return VERIFY_OK;
}

verify_status verify_destroy(verify_ctx* ctx) {
  if (!ctx) return VERIFY_EINVAL;
  cudaSetDevice(ctx->device);
  cudaDeviceSynchronize();
  cudaFree(ctx->moe_hbuf);
  cudaFree(ctx->moe_part);
  cudaFree(ctx->err);
  cudaFree(ctx->moe_sched);
  cudaFree(ctx->st_xn);
  cudaFree(ctx->st_proj);
  cudaFree(ctx->st_o);
  cudaFree(ctx->st_logits);
  cudaFree(ctx->st_idx);
  cudaFree(ctx->st_w);
  cudaFree(ctx->acc_best);
  delete ctx;
  return VERIFY_OK;
}

const char* verify_last_error(const verify_ctx* ctx) { return ctx ? ctx->msg : "null context"; }

int64_t verify_launch_count(const verify_ctx* ctx) { return ctx ? ctx->launches : -1; }

verify_status verify_device_status(verify_ctx* ctx, struct CUstream_st* stream, int32_t* code) {
  if (!ctx) return VERIFY_EINVAL;
  verify_status s = use_device(ctx);
  if (s) return s;
  cudaError_t e = cudaStreamSynchronize(stream);
  if (e) return cuda_fail(ctx, e, "cudaStreamSynchronize");
  int h = 0;
  if ((e = cudaMemcpy(&h, ctx->err, sizeof(int), cudaMemcpyDeviceToHost))) return cuda_fail(ctx, e, "cudaMemcpy");
  if (code) *code = h;
  if (h == 0) return VERIFY_OK;
  cudaMemset(ctx->err, 0, sizeof(int));
  cudaMemset(ctx->moe_sched, 0, vk::kMoeSchedWords * sizeof(int));  // an aborted call may leave counts behind
  cudaMemset(ctx->acc_best, 0, sizeof(unsigned long long) * (vk::kMaxAcceptK + 1));
  cudaDeviceSynchronize();
  snprintf(ctx->msg, sizeof ctx->msg, "device error code %d", h);
  return VERIFY_EDEVICE;
}

verify_status verify_selftest_stuck_wait(verify_ctx* ctx, struct CUstream_st* stream) {
  if (!ctx) return VERIFY_EINVAL;
  verify_status s = use_device(ctx);
  if (s) return s;
  cudaError_t e = vk::launch_stuck_wait_probe(ctx->err, stream);
  if (e) return cuda_fail(ctx, e, "stuck-wait probe launch");
  ctx->launches += 1;
  return VERIFY_OK;
}

int64_t q4_tiled_bytes(int32_t n_out, int32_t k_in, int32_t n_experts, int32_t kind) {
  if (kind != VERIFY_TILE_DENSE && kind != VERIFY_TILE_GATE_UP && kind != VERIFY_TILE_DOWN) return -1;
  if (!valid_shape(n_out, k_in) || n_experts < 1 || (kind == VERIFY_TILE_GATE_UP && n_out % 128 != 0)) return -1;
  return vk::tiled_bytes(n_out, k_in, n_experts, kind);
}

verify_status q4_tile(verify_ctx* ctx, const verify_q4_weight* src, int32_t n_experts, int32_t kind, void* dst,
                      int64_t dst_bytes, verify_q4_weight* out, struct CUstream_st* stream) {
  if (!ctx) return VERIFY_EINVAL;
  verify_status s;
  if ((s = use_device(ctx))) return s;
  if (!src || !out) return fail(ctx, VERIFY_EINVAL, "src or out is NULL%s");
  if (src->layout != VERIFY_Q4_ROWS) return fail(ctx, VERIFY_EINVAL, "src must have the row layout%s");
  if (src->group_size != 64 || src->bits != 4) return fail(ctx, VERIFY_EUNSUPPORTED, "only 4-bit, group 64%s");
  if (kind != VERIFY_TILE_DENSE && kind != VERIFY_TILE_GATE_UP && kind != VERIFY_TILE_DOWN)
    return fail(ctx, VERIFY_EUNSUPPORTED, "unknown tile kind%s");
  const int64_t need = q4_tiled_bytes(src->n_out, src->k_in, n_experts, kind);
  if (need < 0) return fail(ctx, VERIFY_EUNSUPPORTED, "shape or n_experts out of range%s");
  if (dst_bytes < need) return fail(ctx, VERIFY_EINVAL, "dst_bytes is smaller than q4_tiled_bytes%s");
  if ((s = check_dev(ctx, src->packed, 4, "packed"))) return s;
  if ((s = check_dev(ctx, src->scales, 2, "scales"))) return s;
  if ((s = check_dev(ctx, src->biases, 2, "biases"))) return s;
  if ((s = check_dev(ctx, dst, 16, "dst"))) return s;
  cudaError_t e = vk::launch_tile(src->packed, src->scales, src->biases, static_cast<uint8_t*>(dst), src->n_out,
                                  src->k_in, n_experts, kind, stream);
  if (e) return cuda_fail(ctx, e, "q4_tile launch");
  ctx->launches += 1;
  *out = *src;
  out->packed = static_cast<const uint32_t*>(dst);
  out->scales = nullptr;
  out->biases = nullptr;
  out->layout = kind == VERIFY_TILE_GATE_UP ? VERIFY_Q4_TILED_GATE_UP
                : kind == VERIFY_TILE_DOWN  ? VERIFY_Q4_TILED_DOWN
                                            : VERIFY_Q4_TILED;
  return VERIFY_OK;
}

verify_status q4_qmv_k(verify_ctx* ctx, const verify_q4_weight* W, const uint16_t* x, int k, void* y,
                       int dtype_out, struct CUstream_st* stream) {
  if (!ctx) return VERIFY_EINVAL;
  verify_status s;
  if ((s = use_device(ctx))) return s;
  if (k < 1 || k > VERIFY_MAX_K) return fail(ctx, VERIFY_EUNSUPPORTED, "k must be in 1..32%s");
  if ((s = check_q4(ctx, W, "W"))) return s;
  if ((s = check_dtype(ctx, dtype_out, true))) return s;
  if ((s = check_dev(ctx, x, 16, "x"))) return s;
  if ((s = check_dev(ctx, y, dtype_out == VERIFY_BF16 ? 2 : 4, "y"))) return s;

  vk::DenseArgs a{};
  a.tiles = reinterpret_cast<const uint8_t*>(W->packed); a.rt_bytes = rt_bytes(W->k_in);
  a.err = ctx->err;
  a.N = W->n_out; a.K = W->k_in; a.dtype = dtype_out;
  a.KG = a.K / 64; a.KC = (a.KG + vk::kGroupsPerUnit - 1) / vk::kGroupsPerUnit;
  a.RB = (a.N + vk::kBM - 1) / vk::kBM;
  a.S = dense_splits(ctx, a.RB, a.KC);
  const size_t y_elem = dtype_out == VERIFY_BF16 ? 2 : 4;
  // passes of up to VERIFY_PASS_K rows; rows are independent, so each is
  // computed exactly as in a width-1 call
  for (int r0 = 0; r0 < k; r0 += VERIFY_PASS_K) {
    a.k = k - r0 < VERIFY_PASS_K ? k - r0 : VERIFY_PASS_K;
    a.x = x + (size_t)r0 * a.K;
    a.y = static_cast<char*>(y) + (size_t)r0 * a.N * y_elem;
    cudaError_t e = vk::launch_q4_dense(a, a.k <= 8 ? 1 : 2, ctx->pdl, stream);
    if (e) return cuda_fail(ctx, e, "q4_qmv_k launch");
    ctx->launches += 1;
  }
  return VERIFY_OK;
}

verify_status q4_gather_experts_k(verify_ctx* ctx, const verify_q4_experts* gate_up, const verify_q4_experts* down,
                                  const float* logits, int64_t logits_ld, int top_k, const uint16_t* x, int k,
                                  int32_t* idx_out, float* w_out, void* y, int dtype_out,
                                  const verify_q4_weight* shared_gate_up, const verify_q4_weight* shared_down,
                                  const float* shared_gate_logit, struct CUstream_st* stream) {
  if (!ctx) return VERIFY_EINVAL;
  verify_status s;
  if ((s = use_device(ctx))) return s;
  if (!gate_up || !down) return fail(ctx, VERIFY_EINVAL, "expert stacks are NULL%s");
  const int E = gate_up->n_experts;
  const char* why = "";
  if (int rule = vk::moe_shape_status(k, VERIFY_MAX_K, E, down->n_experts, top_k, gate_up->w.n_out, gate_up->w.k_in,
                                      down->w.n_out, down->w.k_in, &why))
    return fail(ctx, (verify_status)rule, why);
  if ((s = check_q4(ctx, &gate_up->w, "gate_up", VERIFY_Q4_TILED_GATE_UP))) return s;
  if ((s = check_q4(ctx, &down->w, "down", VERIFY_Q4_TILED_DOWN))) return s;
  const int H = gate_up->w.k_in, I = gate_up->w.n_out / 2;
  if (logits_ld < E) return fail(ctx, VERIFY_EINVAL, "logits_ld < n_experts%s");
  if ((s = check_dtype(ctx, dtype_out, true))) return s;
  if ((s = check_dev(ctx, logits, 4, "logits"))) return s;
  if ((s = check_dev(ctx, x, 16, "x"))) return s;
  if ((s = check_dev(ctx, idx_out, 4, "idx_out"))) return s;
  if ((s = check_dev(ctx, w_out, 4, "w_out"))) return s;
  if ((s = check_dev(ctx, y, dtype_out == VERIFY_BF16 ? 2 : 4, "y"))) return s;
  const int n_shared = (shared_gate_up != nullptr) + (shared_down != nullptr) + (shared_gate_logit != nullptr);
  if (n_shared != 0 && n_shared != 3)
    return fail(ctx, VERIFY_EINVAL, "shared expert: give all of gate_up, down and gate logit, or none%s");
  if (n_shared == 3) {
    if ((s = check_q4(ctx, shared_gate_up, "shared_gate_up", VERIFY_Q4_TILED_GATE_UP))) return s;
    if ((s = check_q4(ctx, shared_down, "shared_down", VERIFY_Q4_TILED_DOWN))) return s;
    if (shared_gate_up->n_out != 2 * I || shared_gate_up->k_in != H || shared_down->n_out != H ||
        shared_down->k_in != I)
      return fail(ctx, VERIFY_EINVAL, "shared expert shape differs from the routed experts%s");
    if ((s = check_dev(ctx, shared_gate_logit, 4, "shared_gate_logit"))) return s;
  }

  vk::MoeArgs a{};
  a.logits = logits; a.logits_ld = logits_ld; a.shared_logit = n_shared ? shared_gate_logit : nullptr;
  a.x = x;
  a.gu_tiles = reinterpret_cast<const uint8_t*>(gate_up->w.packed);
  a.dn_tiles = reinterpret_cast<const uint8_t*>(down->w.packed);
  if (n_shared) {
    a.sgu_tiles = reinterpret_cast<const uint8_t*>(shared_gate_up->packed);
    a.sdn_tiles = reinterpret_cast<const uint8_t*>(shared_down->packed);
  }
  a.gu_rt_bytes = vk::tile_row_bytes(H, vk::kExpertGroups);
  a.dn_rt_bytes = vk::tile_row_bytes(I, vk::kExpertGroups);
  a.hbuf = ctx->moe_hbuf; a.part = ctx->moe_part;
  a.work = ctx->moe_sched; a.done = ctx->moe_sched + 2 + vk::kMoeSmSlots;
  a.idx_out = idx_out; a.w_out = w_out; a.y = y; a.err = ctx->err;
  a.E = E; a.T = top_k; a.H = H; a.I = I; a.dtype = dtype_out;
  a.has_shared = n_shared ? 1 : 0;
  a.G = vk::moe_ctas_per_sm_for(k, top_k, E, a.has_shared, I, ctx->num_sms, ctx->moe_ctas_per_sm) * ctx->num_sms;
  a.n_sm = ctx->num_sms;
  const size_t y_elem = dtype_out == VERIFY_BF16 ? 2 : 4;
  // passes of up to VERIFY_PASS_K rows (each row's routing, experts and
  // combine depend on that row alone); a later pass's kernels write the
  // shared scratch only after their dependency wait
  for (int r0 = 0; r0 < k; r0 += VERIFY_PASS_K) {
    a.k = k - r0 < VERIFY_PASS_K ? k - r0 : VERIFY_PASS_K;
    a.logits = logits + (size_t)r0 * logits_ld;
    a.shared_logit = n_shared ? shared_gate_logit + (size_t)r0 * logits_ld : nullptr;
    a.x = x + (size_t)r0 * H;
    a.idx_out = idx_out + (size_t)r0 * top_k;
    a.w_out = w_out + (size_t)r0 * top_k;
    a.y = static_cast<char*>(y) + (size_t)r0 * H * y_elem;
    int launched = 0;
    cudaError_t e = vk::launch_moe(a, ctx->pdl, stream, &launched);
    ctx->launches += launched;
    if (e) return cuda_fail(ctx, e, "q4_gather_experts_k launch");
  }
  return VERIFY_OK;
}

verify_status gdn_verify_k(verify_ctx* ctx, const verify_gdn_params* p, verify_gdn_state* st,
                           const verify_gdn_inputs* in, int k, void* o, int dtype_out, struct CUstream_st* stream) {
  if (!ctx) return VERIFY_EINVAL;
  verify_status s;
  if ((s = use_device(ctx))) return s;
  if (!p || !st || !in) return fail(ctx, VERIFY_EINVAL, "params, state or inputs is NULL%s");
  if (k < 1 || k > VERIFY_MAX_K) return fail(ctx, VERIFY_EUNSUPPORTED, "k must be in 1..32%s");
  if (p->n_qk_heads < 1 || p->n_v_heads < 1 || p->n_v_heads % p->n_qk_heads != 0)
    return fail(ctx, VERIFY_EUNSUPPORTED, "n_v_heads must be a positive multiple of n_qk_heads%s");
  if (p->head_dim_k != p->head_dim_v ||
      (p->head_dim_k != 32 && p->head_dim_k != 64 && p->head_dim_k != 128))
    return fail(ctx, VERIFY_EUNSUPPORTED, "head_dim_k == head_dim_v in {32, 64, 128}%s");
  if (p->conv_kernel != 4) return fail(ctx, VERIFY_EUNSUPPORTED, "conv_kernel must be 4%s");
  if (p->gate_act != 0 && p->gate_act != 1) return fail(ctx, VERIFY_EINVAL, "gate_act must be 0 or 1%s");
  if (dtype_out != VERIFY_F32 && dtype_out != VERIFY_BF16) return fail(ctx, VERIFY_EINVAL, "dtype_out F32 or BF16%s");
  if (st->n_slots < k + 1 || st->n_slots > VERIFY_GDN_MAX_SLOTS)
    return fail(ctx, VERIFY_EINVAL, "n_slots must be in k+1..33%s");
  if (!st->dev && (st->cur < 0 || st->cur >= st->n_slots)) return fail(ctx, VERIFY_EINVAL, "cur is not a slot%s");
  if (st->dev && (s = check_dev(ctx, st->dev, 8, "state dev words"))) return s;
  const int d = p->head_dim_k, Hk = p->n_qk_heads, Hv = p->n_v_heads;
  const int C = 2 * Hk * d + Hv * d;
  if (in->ld_qkv < C || in->ld_z < (int64_t)Hv * d || in->ld_a < Hv || in->ld_b < Hv)
    return fail(ctx, VERIFY_EINVAL, "an input row stride is smaller than its row%s");
  if ((s = check_dev(ctx, p->conv_w, 4, "conv_w")) || (s = check_dev(ctx, p->A_log, 4, "A_log")) ||
      (s = check_dev(ctx, p->dt_bias, 4, "dt_bias")) || (s = check_dev(ctx, p->norm_w, 4, "norm_w")) ||
      (s = check_dev(ctx, in->qkv, 2, "qkv")) || (s = check_dev(ctx, in->z, 2, "z")) ||
      (s = check_dev(ctx, in->a, 2, "a")) || (s = check_dev(ctx, in->b, 2, "b")) ||
      (s = check_dev(ctx, o, dtype_out == VERIFY_BF16 ? 2 : 4, "o")))
    return s;

  // Slots in use: cur, then the state after row r in slot r + (r >= cur), the
  // free slots in ascending order.  With a device-held commit cur is known only
  // on the device, so every slot must be valid.
  int pending[VERIFY_GDN_MAX_SLOTS];
  const int n_used = st->dev ? st->n_slots : k + 1;
  if (st->dev) {
    for (int sl = 0; sl < n_used; ++sl) pending[sl] = sl;
  } else {
    pending[0] = st->cur;
    for (int r = 0; r < k; ++r) pending[r + 1] = r + (r >= st->cur ? 1 : 0);
  }
  for (int u = 0; u < n_used; ++u) {
    if ((s = check_dev(ctx, st->S_slots[pending[u]], 16, "S slot"))) return s;
    if ((s = check_dev(ctx, st->conv_slots[pending[u]], 2, "conv slot"))) return s;
  }

  vk::GdnArgs a{};
  for (int sl = 0; sl < st->n_slots; ++sl) {
    a.S_slots[sl] = st->S_slots[sl];
    a.tail_slots[sl] = st->conv_slots[sl];
  }
  a.n_slots = st->n_slots;
  a.cur = st->dev ? 0 : st->cur;
  a.dev_state = st->dev;
  a.r0 = 0;
  a.qkv = in->qkv; a.ld_qkv = in->ld_qkv; a.z = in->z; a.ld_z = in->ld_z;
  a.a = in->a; a.ld_a = in->ld_a; a.b = in->b; a.ld_b = in->ld_b;
  a.conv_w = p->conv_w; a.A_log = p->A_log; a.dt_bias = p->dt_bias; a.norm_w = p->norm_w;
  a.o = o; a.err = ctx->err;
  a.Hk = Hk; a.Hv = Hv; a.d = d; a.W = p->conv_kernel; a.k = k; a.dtype = dtype_out; a.gate_act = p->gate_act;
  a.q_scale = p->q_scale; a.l2_eps = p->l2_eps; a.norm_eps = p->norm_eps;
  // rows 0..15, then (k > 16) a continuation from the snapshot after row 15;
  // it reads that snapshot before its dependency wait, so it is launched
  // after the first pass has finished (no dependent launch)
  const size_t o_elem = dtype_out == VERIFY_BF16 ? 2 : 4;
  for (int r0 = 0; r0 < k; r0 += VERIFY_PASS_K) {
    a.r0 = r0;
    a.k = k - r0 < VERIFY_PASS_K ? k - r0 : VERIFY_PASS_K;
    a.qkv = in->qkv + (size_t)r0 * in->ld_qkv;
    a.z = in->z + (size_t)r0 * in->ld_z;
    a.a = in->a + (size_t)r0 * in->ld_a;
    a.b = in->b + (size_t)r0 * in->ld_b;
    a.o = static_cast<char*>(o) + (size_t)r0 * Hv * d * o_elem;
    cudaError_t e = vk::launch_gdn(a, r0 == 0 && ctx->pdl, stream);
    if (e) return cuda_fail(ctx, e, "gdn_verify_k launch");
    ctx->launches += 1;
  }
  if (!st->dev) {
    for (int r = 0; r <= k; ++r) st->pending[r] = pending[r];
    st->pending_k = k;
  }
  return VERIFY_OK;
}

verify_status gdn_commit(verify_gdn_state* st, int accepted) {
  if (!st || st->dev) return VERIFY_EINVAL;
  if (st->pending_k <= 0) return VERIFY_EINVAL;
  if (accepted < 0 || accepted > st->pending_k) return VERIFY_EINVAL;
  st->cur = st->pending[accepted];
  st->pending_k = 0;
  return VERIFY_OK;
}

verify_status gdn_commit_all(verify_gdn_state* states, int n_states, int accepted) {
  if (!states || n_states < 1) return VERIFY_EINVAL;
  for (int l = 0; l < n_states; ++l)
    if (states[l].dev || states[l].pending_k <= 0 || accepted < 0 || accepted > states[l].pending_k)
      return VERIFY_EINVAL;
  for (int l = 0; l < n_states; ++l) {
    states[l].cur = states[l].pending[accepted];
    states[l].pending_k = 0;
  }
  return VERIFY_OK;
}

// The dev words of states[0 .. n-1] are consecutive int32 pairs in device memory.
static verify_status check_dev_states(verify_ctx* ctx, const verify_gdn_state* states, int n_states) {
  if (!states || n_states < 1) return fail(ctx, VERIFY_EINVAL, "states is NULL or n_states < 1%s");
  verify_status s;
  if ((s = check_dev(ctx, states[0].dev, 8, "state dev words"))) return s;
  for (int l = 1; l < n_states; ++l)
    if (states[l].dev != states[0].dev + 2 * l)
      return fail(ctx, VERIFY_EINVAL, "the states' dev words must be consecutive pairs%s");
  return VERIFY_OK;
}

verify_status gdn_state_to_device(verify_ctx* ctx, verify_gdn_state* states, int n_states, int32_t* dev,
                                  struct CUstream_st* stream) {
  if (!ctx) return VERIFY_EINVAL;
  verify_status s;
  if ((s = use_device(ctx))) return s;
  if (!states || n_states < 1 || n_states > (1 << 20)) return fail(ctx, VERIFY_EINVAL, "states or n_states invalid%s");
  if ((s = check_dev(ctx, dev, 8, "dev"))) return s;
  std::vector<int32_t> words(2 * (size_t)n_states);
  for (int l = 0; l < n_states; ++l) {
    if (states[l].dev) return fail(ctx, VERIFY_EINVAL, "a state is already on the device%s");
    if (states[l].n_slots < 2 || states[l].n_slots > VERIFY_GDN_MAX_SLOTS || states[l].cur < 0 ||
        states[l].cur >= states[l].n_slots)
      return fail(ctx, VERIFY_EINVAL, "a state's cur or n_slots is invalid%s");
    words[2 * l] = states[l].cur;
    words[2 * l + 1] = 0;
  }
  cudaError_t e = cudaMemcpyAsync(dev, words.data(), words.size() * sizeof(int32_t), cudaMemcpyHostToDevice, stream);
  if (!e) e = cudaStreamSynchronize(stream);
  if (e) return cuda_fail(ctx, e, "gdn_state_to_device copy");
  for (int l = 0; l < n_states; ++l) {
    states[l].dev = dev + 2 * l;
    states[l].pending_k = 0;
  }
  return VERIFY_OK;
}

verify_status gdn_state_to_host(verify_ctx* ctx, verify_gdn_state* states, int n_states, struct CUstream_st* stream) {
  if (!ctx) return VERIFY_EINVAL;
  verify_status s;
  if ((s = use_device(ctx))) return s;
  if ((s = check_dev_states(ctx, states, n_states))) return s;
  std::vector<int32_t> words(2 * (size_t)n_states);
  cudaError_t e = cudaStreamSynchronize(stream);
  if (!e) e = cudaMemcpy(words.data(), states[0].dev, words.size() * sizeof(int32_t), cudaMemcpyDeviceToHost);
  if (e) return cuda_fail(ctx, e, "gdn_state_to_host copy");
  for (int l = 0; l < n_states; ++l)
    if (words[2 * l] < 0 || words[2 * l] >= states[l].n_slots)
      return fail(ctx, VERIFY_EINVAL, "a device-held committed slot is invalid%s");
  for (int l = 0; l < n_states; ++l) {
    states[l].cur = words[2 * l];
    states[l].pending_k = 0;
    states[l].dev = nullptr;
  }
  return VERIFY_OK;
}

verify_status gdn_commit_dev(verify_ctx* ctx, const verify_gdn_state* states, int n_states, const int32_t* accepted,
                             struct CUstream_st* stream) {
  if (!ctx) return VERIFY_EINVAL;
  verify_status s;
  if ((s = use_device(ctx))) return s;
  if ((s = check_dev_states(ctx, states, n_states))) return s;
  if ((s = check_dev(ctx, accepted, 4, "accepted"))) return s;
  vk::AcceptArgs a{};
  a.V = 0;
  a.k = 1;
  a.accepted = accepted;
  a.dev_state = states[0].dev;
  a.n_states = n_states;
  a.need_k = 0;
  a.err = ctx->err;
  cudaError_t e = vk::launch_accept(a, stream);
  if (e) return cuda_fail(ctx, e, "gdn_commit_dev launch");
  ctx->launches += 1;
  return VERIFY_OK;
}

verify_status verify_accept_greedy(verify_ctx* ctx, const float* logits, int64_t ld, int V, int k,
                                   const int32_t* draft, int32_t* result, const verify_gdn_state* states,
                                   int n_states, struct CUstream_st* stream) {
  if (!ctx) return VERIFY_EINVAL;
  verify_status s;
  if ((s = use_device(ctx))) return s;
  if (k < 1 || k > vk::kMaxAcceptK) return fail(ctx, VERIFY_EUNSUPPORTED, "k must be in 1..32%s");
  if (V < 1 || V > (1 << 30)) return fail(ctx, VERIFY_EUNSUPPORTED, "V must be in 1..2^30%s");
  if (ld < V) return fail(ctx, VERIFY_EINVAL, "ld must be >= V%s");
  if ((s = check_dev(ctx, logits, 4, "logits")) || (s = check_dev(ctx, result, 4, "result"))) return s;
  if (k > 1 && (s = check_dev(ctx, draft, 4, "draft"))) return s;
  if (n_states < 0) return fail(ctx, VERIFY_EINVAL, "n_states < 0%s");
  if (n_states > 0 && (s = check_dev_states(ctx, states, n_states))) return s;
  vk::AcceptArgs a{};
  a.logits = logits;
  a.ld = ld;
  a.V = V;
  a.k = k;
  a.vec = aligned(logits, 16) && ld % 4 == 0;
  a.blocks_per_row = vk::accept_blocks_per_row(V, k, ctx->num_sms);
  a.draft = draft;
  a.result = result;
  a.dev_state = n_states > 0 ? states[0].dev : nullptr;
  a.n_states = n_states;
  a.need_k = k;
  a.best = ctx->acc_best;
  a.ticket = ctx->acc_ticket;
  a.err = ctx->err;
  cudaError_t e = vk::launch_accept(a, stream);
  if (e) return cuda_fail(ctx, e, "verify_accept_greedy launch");
  ctx->launches += 1;
  return VERIFY_OK;
}

verify_status verify_lm_head_accept(verify_ctx* ctx, const verify_q4_weight* W, const uint16_t* x, int k,
                                    const int32_t* draft, int32_t* result, const verify_gdn_state* states,
                                    int n_states, struct CUstream_st* stream) {
  if (!ctx) return VERIFY_EINVAL;
  verify_status s;
  if ((s = use_device(ctx))) return s;
  if (k < 1 || k > VERIFY_MAX_K) return fail(ctx, VERIFY_EUNSUPPORTED, "k must be in 1..32%s");
  if ((s = check_q4(ctx, W, "W"))) return s;
  if ((s = check_dev(ctx, x, 16, "x")) || (s = check_dev(ctx, result, 4, "result"))) return s;
  if (k > 1 && (s = check_dev(ctx, draft, 4, "draft"))) return s;
  if (n_states < 0) return fail(ctx, VERIFY_EINVAL, "n_states < 0%s");
  if (n_states > 0 && (s = check_dev_states(ctx, states, n_states))) return s;
  vk::DenseArgs a{};
  a.tiles = reinterpret_cast<const uint8_t*>(W->packed); a.rt_bytes = rt_bytes(W->k_in);
  a.err = ctx->err;
  a.N = W->n_out; a.K = W->k_in; a.dtype = VERIFY_F32;
  a.KG = a.K / 64; a.KC = (a.KG + vk::kGroupsPerUnit - 1) / vk::kGroupsPerUnit;
  a.RB = (a.N + vk::kBM - 1) / vk::kBM;
  a.S = dense_splits(ctx, a.RB, a.KC);  // as q4_qmv_k: the same fp32 outputs
  a.best = ctx->acc_best;
  for (int r0 = 0; r0 < k; r0 += VERIFY_PASS_K) {
    a.k = k - r0 < VERIFY_PASS_K ? k - r0 : VERIFY_PASS_K;
    a.r0 = r0;
    a.x = x + (size_t)r0 * a.K;
    cudaError_t e = vk::launch_q4_dense_argmax(a, a.k <= 8 ? 1 : 2, stream);
    if (e) return cuda_fail(ctx, e, "verify_lm_head_accept launch");
    ctx->launches += 1;
  }
  // then one CTA: the accepted prefix from the merged keys, the result, the commit
  vk::AcceptArgs f{};
  f.V = -1;
  f.k = k;
  f.draft = draft;
  f.result = result;
  f.dev_state = n_states > 0 ? states[0].dev : nullptr;
  f.n_states = n_states;
  f.need_k = k;
  f.best = ctx->acc_best;
  f.ticket = ctx->acc_ticket;
  f.err = ctx->err;
  cudaError_t e = vk::launch_accept(f, stream);
  if (e) return cuda_fail(ctx, e, "verify_lm_head_accept finish launch");
  ctx->launches += 1;
  return VERIFY_OK;
}

// ------------------------------------------------------------ attention

// Workspace of one attention call: the rotated queries (hi and lo binary16
// parts, per KV head its pairs in rows padded to a multiple of 128), then
// (max, sum) and the unnormalised outputs of every (KV head, split, pair),
// each 256-byte aligned.
struct AttnWork {
  long long qh, ql, ml, po, total;
};
static AttnWork attn_work(const verify_attn_params* p, long long nsplit, int k) {
  auto up = [](long long b) { return (b + 255) / 256 * 256; };
  const long long G = p->n_q_heads / p->n_kv_heads;
  const long long Mpad = (k * G + 15) / 16 * 16;
  const long long qbytes = p->n_kv_heads * ((k * G + 127) / 128 * 128) * p->head_dim * 2;
  AttnWork w;
  w.qh = 0;
  w.ql = up(qbytes);
  w.ml = w.ql + up(qbytes);
  w.po = w.ml + up(p->n_kv_heads * nsplit * Mpad * 8);
  w.total = w.po + up(p->n_kv_heads * nsplit * Mpad * (long long)p->head_dim * 4);
  return w;
}

static bool attn_params_ok(const verify_attn_params* p) {
  return p && p->n_q_heads >= 1 && p->n_kv_heads >= 1 && p->n_q_heads % p->n_kv_heads == 0 &&
         p->n_q_heads <= 1024 && (p->head_dim == 128 || p->head_dim == 256) && p->rope_dim >= 0 &&
         p->rope_dim <= p->head_dim && p->rope_dim % 2 == 0 && p->rope_theta > 0.f;
}

// About 128 key splits per KV head at full length, and at least 128
// positions per split (a sweep at 4,096 and 65,536 positions, k = 1 and 9).
int32_t attn_default_split(int64_t capacity) {
  // about 74 splits per KV head: with two KV heads, one wave of one
  // partial-kernel CTA per SM on a 148- to 152-SM GPU; a multiple of the
  // kernel's 64-position sub-tile, at least 128
  if (capacity < 1) return 128;
  const int64_t per = (capacity + 73) / 74;
  const int64_t s = (per + 63) / 64 * 64;
  return (int32_t)(s < 128 ? 128 : (s > (1 << 20) ? (1 << 20) : s));
}

int64_t attn_workspace_bytes(const verify_attn_params* p, int64_t capacity, int32_t split, int32_t max_k) {
  if (!attn_params_ok(p) || capacity < 1 || split < 32 || split % 32 || max_k < 1 || max_k > VERIFY_MAX_K)
    return 0;
  return attn_work(p, (capacity + split - 1) / split, max_k).total;
}

verify_status attn_verify_k(verify_ctx* ctx, const verify_attn_params* p, verify_kv_cache* cache,
                            const verify_attn_inputs* in, int k, void* o, int dtype_out, struct CUstream_st* stream) {
  if (!ctx) return VERIFY_EINVAL;
  verify_status s;
  if ((s = use_device(ctx))) return s;
  if (!p || !cache || !in) return fail(ctx, VERIFY_EINVAL, "params, cache or inputs is NULL%s");
  if (!attn_params_ok(p))
    return fail(ctx, VERIFY_EUNSUPPORTED, "attention: head_dim 128 or 256, n_q_heads a multiple of n_kv_heads, "
                                          "even rope_dim <= head_dim%s");
  if (k < 1 || k > VERIFY_MAX_K) return fail(ctx, VERIFY_EUNSUPPORTED, "k must be in 1..32%s");
  const int G = p->n_q_heads / p->n_kv_heads, D = p->head_dim;
  if (k * G > vk::kAttnMaxM) return fail(ctx, VERIFY_EUNSUPPORTED, "k * n_q_heads / n_kv_heads must be <= 512%s");
  if (cache->split < 32 || cache->split % 32) return fail(ctx, VERIFY_EINVAL, "split must be a multiple of 32%s");
  if (cache->len < 0 || cache->capacity < 1 || (int64_t)cache->len + k > cache->capacity)
    return fail(ctx, VERIFY_EINVAL, "len + k must be <= capacity%s");
  const long long nsplit = ((long long)cache->len + k + cache->split - 1) / cache->split;
  if (nsplit > 65535) return fail(ctx, VERIFY_EUNSUPPORTED, "more than 65535 key splits: use a larger split%s");
  if (dtype_out != VERIFY_F32 && dtype_out != VERIFY_BF16) return fail(ctx, VERIFY_EINVAL, "dtype_out F32 or BF16%s");
  if (in->ld_q < (int64_t)p->n_q_heads * D || in->ld_gate < (int64_t)p->n_q_heads * D ||
      in->ld_k < (int64_t)p->n_kv_heads * D || in->ld_v < (int64_t)p->n_kv_heads * D)
    return fail(ctx, VERIFY_EINVAL, "an input row stride is smaller than its row%s");
  const AttnWork w = attn_work(p, nsplit, k);
  if (cache->work_bytes < w.total) return fail(ctx, VERIFY_EINVAL, "cache workspace too small%s");
  if ((s = check_dev(ctx, cache->K, 16, "K cache")) || (s = check_dev(ctx, cache->V, 16, "V cache")) ||
      (s = check_dev(ctx, cache->work, 256, "workspace")) || (s = check_dev(ctx, in->q, 2, "q")) ||
      (s = check_dev(ctx, in->gate, 2, "gate")) || (s = check_dev(ctx, in->k, 2, "k")) ||
      (s = check_dev(ctx, in->v, 2, "v")) || (s = check_dev(ctx, o, dtype_out == VERIFY_BF16 ? 2 : 4, "o")))
    return s;
  vk::AttnArgs a{};
  a.q = in->q; a.ld_q = in->ld_q; a.gate = in->gate; a.ld_gate = in->ld_gate;
  a.kin = in->k; a.ld_k = in->ld_k; a.vin = in->v; a.ld_v = in->ld_v;
  a.K = cache->K; a.V = cache->V; a.cap = cache->capacity;
  a.Hq = p->n_q_heads; a.Hkv = p->n_kv_heads; a.D = D; a.rope_dim = p->rope_dim;
  for (int j = 0; j < p->rope_dim / 2; ++j) a.inv_freq[j] = pow((double)p->rope_theta, -2.0 * j / p->rope_dim);
  a.qscale = 1.4426950408889634 / sqrt((double)D);
  a.P = cache->len; a.k = k; a.split = cache->split; a.nsplit = (int)nsplit;
  a.err = ctx->err;
  a.n_mtiles = (k * G + 15) / 16;
  a.q_rows = (k * G + 127) / 128 * 128;
  char* base = static_cast<char*>(cache->work);
  a.qh = reinterpret_cast<uint16_t*>(base + w.qh);
  a.ql = reinterpret_cast<uint16_t*>(base + w.ql);
  a.part_ml = reinterpret_cast<float2*>(base + w.ml);
  a.part_o = reinterpret_cast<float*>(base + w.po);
  a.o = o; a.dtype = dtype_out == VERIFY_BF16 ? 1 : 0;
  int launched = 0;
  cudaError_t e = vk::launch_attn(a, stream, &launched);
  ctx->launches += launched;
  if (e) return cuda_fail(ctx, e, "attn_verify_k launch");
  cache->pending_k = k;
  return VERIFY_OK;
}

verify_status attn_commit(verify_kv_cache* cache, int accepted) {
  if (!cache || cache->pending_k <= 0 || accepted < 0 || accepted > cache->pending_k) return VERIFY_EINVAL;
  cache->len += accepted;
  cache->pending_k = 0;
  return VERIFY_OK;
}

verify_status verify_rmsnorm_k(verify_ctx* ctx, const float* x, const float* w, float eps, int zero_centered, int n,
                               int k, void* out, int dtype_out, struct CUstream_st* stream) {
  if (!ctx) return VERIFY_EINVAL;
  verify_status s;
  if ((s = use_device(ctx))) return s;
  if (n < 4 || n > 16384 || n % 4 != 0) return fail(ctx, VERIFY_EUNSUPPORTED, "n must be a multiple of 4 in [4, 16384]%s");
  if (k < 1 || k > 65535) return fail(ctx, VERIFY_EINVAL, "k out of range%s");
  if (dtype_out != VERIFY_F32 && dtype_out != VERIFY_BF16) return fail(ctx, VERIFY_EINVAL, "dtype_out F32 or BF16%s");
  if ((s = check_dev(ctx, x, 4, "x")) || (s = check_dev(ctx, w, 4, "w")) ||
      (s = check_dev(ctx, out, dtype_out == VERIFY_BF16 ? 2 : 4, "out")))
    return s;
  cudaError_t e = vk::launch_rmsnorm(x, w, eps, zero_centered, n, k, out, dtype_out, ctx->pdl, stream);
  if (e) return cuda_fail(ctx, e, "verify_rmsnorm_k launch");
  ctx->launches += 1;
  return VERIFY_OK;
}

verify_status verify_layer_k(verify_ctx* ctx, const verify_layer* L, verify_gdn_state* st, float* h, int k,
                             int32_t* idx_out, struct CUstream_st* stream) {
  if (!ctx) return VERIFY_EINVAL;
  if (!L || !st) return fail(ctx, VERIFY_EINVAL, "layer or state is NULL%s");
  if (k < 1 || k > VERIFY_MAX_K) return fail(ctx, VERIFY_EUNSUPPORTED, "k must be in 1..32%s");
  const verify_gdn_params& g = L->gdn;
  const int H = L->in_proj.k_in;
  const int C = 2 * g.n_qk_heads * g.head_dim_k + g.n_v_heads * g.head_dim_v;
  const int Z = g.n_v_heads * g.head_dim_v;
  const int NP = C + Z + 2 * g.n_v_heads;
  const int E = L->gate_up.n_experts;
  if (H > kMaxH || H % 4 != 0) return fail(ctx, VERIFY_EUNSUPPORTED, "hidden size must be a multiple of 4, <= 8192%s");
  if (L->in_proj.n_out != NP || NP > kMaxProj) return fail(ctx, VERIFY_EINVAL, "in_proj must have C + Hv*dv + 2*Hv rows%s");
  if (L->out_proj.n_out != H || L->out_proj.k_in != Z) return fail(ctx, VERIFY_EINVAL, "out_proj must be [H, Hv*dv]%s");
  if (L->router.n_out != E + 1 || L->router.k_in != H || E + 1 > 1024)
    return fail(ctx, VERIFY_EINVAL, "router must be [E+1, H] (routing rows, then the shared gate row)%s");
  verify_status s;
  cudaStream_t sm = stream;
  auto mark = [&](int i) {
    // external record: inside stream capture this becomes an event-record node of the graph
    if (ctx->n_layer_events == 8 && ctx->layer_events[i])
      cudaEventRecordWithFlags(ctx->layer_events[i], sm, cudaEventRecordExternal);
  };
  // The layer's first kernel waits for everything enqueued before the call
  // (inside verify_stack_k, layers after the first chain to the previous
  // layer instead); each later one may start during its predecessor's tail,
  // unless an event is recorded between the two.
  struct PdlOff {
    verify_ctx* c;
    ~PdlOff() { c->pdl = false; }
  } pdl_off{ctx};
  auto overlap_after = [&](int i) { ctx->pdl = !(ctx->n_layer_events == 8 && ctx->layer_events[i]); };
  mark(0);
  ctx->pdl = ctx->chain_layer && !(ctx->n_layer_events == 8 && ctx->layer_events[0]);
  // 1. pre-mixer norm
  if ((s = verify_rmsnorm_k(ctx, h, L->norm1_w, L->norm_eps, 1, H, k, ctx->st_xn, VERIFY_BF16, sm))) return s;
  mark(1);
  overlap_after(1);
  // 2. in_proj -> q|k|v, z, a, b
  if ((s = q4_qmv_k(ctx, &L->in_proj, ctx->st_xn, k, ctx->st_proj, VERIFY_BF16, sm))) return s;
  mark(2);
  overlap_after(2);
  // 3. Gated DeltaNet verify
  verify_gdn_inputs in;
  in.qkv = ctx->st_proj; in.ld_qkv = NP;
  in.z = ctx->st_proj + C; in.ld_z = NP;
  in.a = ctx->st_proj + C + Z; in.ld_a = NP;
  in.b = ctx->st_proj + C + Z + g.n_v_heads; in.ld_b = NP;
  if ((s = gdn_verify_k(ctx, &L->gdn, st, &in, k, ctx->st_o, VERIFY_BF16, sm))) return s;
  mark(3);
  overlap_after(3);
  // 4. out_proj into the residual
  if ((s = q4_qmv_k(ctx, &L->out_proj, ctx->st_o, k, h, VERIFY_F32_ADD, sm))) return s;
  mark(4);
  overlap_after(4);
  // 5. pre-FFN norm
  if ((s = verify_rmsnorm_k(ctx, h, L->norm2_w, L->norm_eps, 1, H, k, ctx->st_xn, VERIFY_BF16, sm))) return s;
  mark(5);
  overlap_after(5);
  // 6. router + shared-expert gate logits
  if ((s = q4_qmv_k(ctx, &L->router, ctx->st_xn, k, ctx->st_logits, VERIFY_F32, sm))) return s;
  mark(6);
  overlap_after(6);
  // 7. routed + shared experts into the residual
  if ((s = q4_gather_experts_k(ctx, &L->gate_up, &L->down, ctx->st_logits, E + 1, L->top_k, ctx->st_xn, k,
                               idx_out ? idx_out : ctx->st_idx, ctx->st_w, h, VERIFY_F32_ADD, &L->shared_gate_up,
                               &L->shared_down, ctx->st_logits + E, sm)))
    return s;
  mark(7);
  return VERIFY_OK;
}

verify_status verify_stack_k(verify_ctx* ctx, const verify_layer* layers, verify_gdn_state* states, int n_layers,
                             float* h, int k, int32_t* idx_out, struct CUstream_st* stream) {
  if (!ctx) return VERIFY_EINVAL;
  if (!layers || !states || n_layers < 1) return fail(ctx, VERIFY_EINVAL, "layers, states or n_layers invalid%s");
  int32_t* idx = idx_out;
  for (int l = 0; l < n_layers; ++l) {
    ctx->chain_layer = l > 0;
    verify_status s = verify_layer_k(ctx, &layers[l], &states[l], h, k, idx, stream);
    ctx->chain_layer = false;
    if (s) return s;
    if (idx) idx += (long long)k * layers[l].top_k;
  }
  return VERIFY_OK;
}

verify_status verify_set_layer_events(verify_ctx* ctx, void* const* events, int n) {
  if (!ctx) return VERIFY_EINVAL;
  if (!events || n == 0) {
    ctx->n_layer_events = 0;
    return VERIFY_OK;
  }
  if (n != 8) return fail(ctx, VERIFY_EINVAL, "verify_set_layer_events needs 8 events%s");
  for (int i = 0; i < 8; ++i) ctx->layer_events[i] = reinterpret_cast<cudaEvent_t>(events[i]);
  ctx->n_layer_events = 8;
  return VERIFY_OK;
}

}  // extern "C"
