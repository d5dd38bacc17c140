// gdn_kernel.cu - k-row Gated DeltaNet verify step with in-kernel snapshots.
//
// What is computed (pages, by title): "QWEN38FLASH.md - Plan for supporting
// Qwen/Qwen3.8-Flash-Next" section 2.1 (causal depthwise conv over q|k|v, L2
// norm of q and k per head, softplus/exp decay from A_log/dt_bias, the
// delta rule S <- gS; m = S k; delta = (v - m) beta; S += delta k^T;
// y = S q, gated RMSNorm) and 3.1 (scalar per-head decay, sigmoid beta, each
// k head shared by Hv/Hk v heads); "Red Lite dev45 - speculative decoding
// with the Qwen3-Next MTP block", "What it is" (row r runs from row r-1's
// state; the state after each row is written to snapshot buffers from inside
// the kernel).
//
// Design (GB300): one thread-block cluster per V head, one CTA per 16 value
// rows of that head (8 CTAs for head dim 128, 384 CTAs for 48 heads).  The
// value rows of the delta rule are independent, so each CTA keeps its
// 16 x 128 slice of the fp32 state in registers (16 floats per thread, 8
// threads per value row) for all k rows: the state is read from HBM once and
// each snapshot is written once with coalesced 16-byte stores.  The conv, the
// L2 norms and the gates are cheap and recomputed by every CTA of the head.
// The only cross-CTA step, the RMSNorm's sum of squares over the head's value
// rows, goes through distributed shared memory in fixed rank order.  There is
// no atomic and no order that depends on k: row r of a width-k call is
// bit-identical to a width-1 call from the snapshot after r rows.
#include "common.cuh"
#include "internal.h"

namespace vk {

constexpr int kGdnRows = 16;  // value rows per CTA
constexpr int kGdnMaxK = 16;

// Threads per value row: each holds D / TPR state columns (a multiple of 4).
template <int D>
struct GdnShape {
  static constexpr int TPR = D >= 64 ? 16 : 8;
  static constexpr int THREADS = kGdnRows * TPR;  // 256 for D >= 64
  static constexpr int NV4 = D / TPR / 4;         // float4 groups of state columns per thread
  static constexpr int P = D / kGdnRows;          // CTAs per head (cluster size)
};

__device__ __forceinline__ float sigmoidf_(float t) { return 1.f / (1.f + expf(-t)); }
// The conv's SiLU, evaluated k x (2 d + 16) times per CTA, uses the fast
// exponential and divide (a few ulp; the state and the outputs are held to
// 1e-3 of their rms against the float64 oracle).
__device__ __forceinline__ float siluf_(float t) { return __fdividef(t, 1.f + __expf(-t)); }
__device__ __forceinline__ float softplusf_(float t) { return fmaxf(t, 0.f) + log1pf(expf(-fabsf(t))); }

template <int D>
__global__ void __launch_bounds__(GdnShape<D>::THREADS) gdn_verify_kernel(const GdnArgs a) {
  using SH = GdnShape<D>;
  constexpr int TPR = SH::TPR, NT = SH::THREADS, NV4 = SH::NV4, P = SH::P;
  // rows padded by 16 floats: the two half-warps of the L2 norms read
  // adjacent rows in different banks
  __shared__ __align__(16) float qn[kGdnMaxK][D + 16];
  __shared__ __align__(16) float kn[kGdnMaxK][D + 16];
  __shared__ float vs[kGdnMaxK][kGdnRows];
  __shared__ float ys[kGdnMaxK][kGdnRows];
  __shared__ float gs[kGdnMaxK], bs[kGdnMaxK], kq[kGdnMaxK];
  __shared__ float ss_part[kGdnMaxK];
  __shared__ float ss_all[kGdnMaxK][P];
  __shared__ float inv_s[kGdnMaxK];

  const int p = (int)cluster_rank();
  const int h = blockIdx.x / P;
  const int hq = h / (a.Hv / a.Hk);
  const int tid = threadIdx.x;
  const int k = a.k;
  const int C = 2 * a.Hk * D + a.Hv * D;
  const bool owns_qk_tail = (h % (a.Hv / a.Hk)) == 0;

  // thread (il, l): value row il of this CTA, state columns 4 l + 4 TPR m + e
  const int il = tid / TPR, l = tid % TPR;
  const int i = p * kGdnRows + il;  // value row within the head

  // Committed slot.  A device-held one was written by a commit at least two
  // launches before this one (the layer's first launch waits for all earlier
  // work), so it may be read before the dependency wait.  Every CTA reads the
  // same word; an invalid slot makes all of them leave before writing anything.
  int cur = a.cur;
  if (a.dev_state) {
    cur = __ldcg(a.dev_state);
    if (cur < 0 || cur >= a.n_slots) {
      if (blockIdx.x == 0 && tid == 0) record_error(a.err, VERIFY_DEV_ESLOT);
      return;
    }
  }
  // this launch starts from the state after the block's first r0 rows
  const int in_slot = a.r0 == 0 ? cur : (a.r0 - 1) + (a.r0 - 1 >= cur ? 1 : 0);
  const float* S_in = a.S_slots[in_slot];
  const uint16_t* tail_in = a.tail_slots[in_slot];

  // ---- before the grid dependency wait: the state slice and the conv
  //      weights and tail (parameters, or written by an earlier verify call)
  float s[4 * NV4];
  {
    const float* src = S_in + ((long long)h * D + i) * D;
#pragma unroll
    for (int m = 0; m < NV4; ++m) {
      const float4 v = __ldcg(reinterpret_cast<const float4*>(src + 4 * l + 4 * TPR * m));
      s[4 * m] = v.x; s[4 * m + 1] = v.y; s[4 * m + 2] = v.z; s[4 * m + 3] = v.w;
    }
  }
  // Conv channels of this CTA: the q and k channels of QK head hq, then the v
  // channels of its value rows; thread tid takes channels tid, tid + NT, ...
  constexpr int NCH = 2 * D + kGdnRows;
  constexpr int NIT = (NCH + NT - 1) / NT;
  int chn[NIT];
  float cw[NIT][4];
  uint16_t tl[NIT][3];
#pragma unroll
  for (int it = 0; it < NIT; ++it) {
    const int cl = tid + it * NT;
    int ch = 0;
    if (cl < D) ch = hq * D + cl;
    else if (cl < 2 * D) ch = a.Hk * D + hq * D + (cl - D);
    else if (cl < NCH) ch = 2 * a.Hk * D + h * D + p * kGdnRows + (cl - 2 * D);
    chn[it] = ch;
#pragma unroll
    for (int t = 0; t < 4; ++t) cw[it][t] = cl < NCH ? a.conv_w[ch * 4 + t] : 0.f;
#pragma unroll
    for (int t = 0; t < 3; ++t) tl[it][t] = cl < NCH ? __ldcg(tail_in + t * C + ch) : (uint16_t)0;
  }
  // gated RMSNorm: output e = tid + NT h2 is (row e / 16, value row e % 16)
  constexpr int EPT = (kGdnMaxK * kGdnRows + NT - 1) / NT;  // outputs per thread
  float nw[EPT];
#pragma unroll
  for (int h2 = 0; h2 < EPT; ++h2) nw[h2] = a.norm_w[p * kGdnRows + (tid + h2 * NT) % kGdnRows];
  griddep_wait();
  griddep_launch();
  if (a.dev_state && blockIdx.x == 0 && tid == 0) a.dev_state[1] = a.r0 + k;

  // ---- 1. causal depthwise conv + SiLU; slide the window
  uint16_t xin[NIT][kGdnMaxK];
#pragma unroll
  for (int it = 0; it < NIT; ++it)
#pragma unroll
    for (int r = 0; r < kGdnMaxK; ++r)
      xin[it][r] = (r < k && tid + it * NT < NCH) ? a.qkv[r * a.ld_qkv + chn[it]] : (uint16_t)0;
  uint16_t zin[EPT];
#pragma unroll
  for (int h2 = 0; h2 < EPT; ++h2) {
    const int e = tid + h2 * NT;
    zin[h2] = e < k * kGdnRows ? a.z[(e / kGdnRows) * a.ld_z + h * D + p * kGdnRows + e % kGdnRows] : (uint16_t)0;
  }
  // gate inputs, loaded with the conv inputs
  float av = 0.f, bv = 0.f;
  if (tid < k) {
    av = bf16f(a.a[tid * a.ld_a + h]);
    bv = bf16f(a.b[tid * a.ld_b + h]);
  }
#pragma unroll
  for (int it = 0; it < NIT; ++it) {
    const int cl = tid + it * NT;
    if (cl >= NCH) break;
    const int ch = chn[it];
    bool write_tail;
    if (cl < D) write_tail = owns_qk_tail && (cl / (D / P) == p);
    else if (cl < 2 * D) write_tail = owns_qk_tail && ((cl - D) / (D / P) == p);
    else write_tail = true;
    uint16_t w0 = tl[it][0], w1 = tl[it][1], w2 = tl[it][2];
#pragma unroll
    for (int r = 0; r < kGdnMaxK; ++r) {
      if (r >= k) break;
      const uint16_t xr = xin[it][r];
      float acc = cw[it][0] * bf16f(w0);
      acc = fmaf(cw[it][1], bf16f(w1), acc);
      acc = fmaf(cw[it][2], bf16f(w2), acc);
      acc = fmaf(cw[it][3], bf16f(xr), acc);
      const float cv = siluf_(acc);
      if (cl < D) qn[r][cl] = cv;
      else if (cl < 2 * D) kn[r][cl - D] = cv;
      else vs[r][cl - 2 * D] = cv;
      w0 = w1; w1 = w2; w2 = xr;
      if (write_tail) {
        const int rr = a.r0 + r;
        uint16_t* to = a.tail_slots[rr + (rr >= cur)];
        to[ch] = w0;
        to[C + ch] = w1;
        to[2 * C + ch] = w2;
      }
    }
  }
  // ---- gates
  if (tid < k) {
    bs[tid] = sigmoidf_(bv);
    gs[tid] = expf(-expf(a.A_log[h]) * softplusf_(av + a.dt_bias[h]));
  }
  __syncthreads();

  // ---- 2. L2 norms of q and k per row, k.q: half-warp h takes rows h,
  //      h + NT/16, ... (all of a 16-row block at once for D >= 64)
  {
    constexpr int HW = NT / 16;
    const int hw = tid >> 4, hl = tid & 15;
    const unsigned half = 0xFFFFu << (16 * (hw & 1));
    for (int r = hw; r < k; r += HW) {
      float sq = 0.f, sk = 0.f;
#pragma unroll
      for (int j = hl; j < D; j += 16) {
        sq = fmaf(qn[r][j], qn[r][j], sq);
        sk = fmaf(kn[r][j], kn[r][j], sk);
      }
#pragma unroll
      for (int off = 8; off > 0; off >>= 1) {
        sq += __shfl_xor_sync(half, sq, off);
        sk += __shfl_xor_sync(half, sk, off);
      }
      const float iq = a.q_scale / sqrtf(sq + a.l2_eps), ik = 1.f / sqrtf(sk + a.l2_eps);
      float dot = 0.f;
#pragma unroll
      for (int j = hl; j < D; j += 16) {
        const float qv = qn[r][j] * iq;
        const float kv = kn[r][j] * ik;
        qn[r][j] = qv;
        kn[r][j] = kv;
        dot = fmaf(kv, qv, dot);
      }
#pragma unroll
      for (int off = 8; off > 0; off >>= 1) dot += __shfl_xor_sync(half, dot, off);
      if (hl == 0) kq[r] = dot;
    }
  }
  __syncthreads();

  // ---- 3. delta rule over the k rows, state slice in registers
  for (int r = 0; r < k; ++r) {
    const float g = gs[r], beta = bs[r];
    float mk = 0.f, mq = 0.f;
#pragma unroll
    for (int m = 0; m < NV4; ++m) {
      const float4 kv = *reinterpret_cast<const float4*>(&kn[r][4 * l + 4 * TPR * m]);
      const float4 qv = *reinterpret_cast<const float4*>(&qn[r][4 * l + 4 * TPR * m]);
      const float kk[4] = {kv.x, kv.y, kv.z, kv.w};
      const float qq[4] = {qv.x, qv.y, qv.z, qv.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float sv = g * s[4 * m + e];
        s[4 * m + e] = sv;
        mk = fmaf(sv, kk[e], mk);
        mq = fmaf(sv, qq[e], mq);
      }
    }
#pragma unroll
    for (int off = TPR / 2; off > 0; off >>= 1) {  // the TPR threads of this value row
      mk += __shfl_xor_sync(0xffffffffu, mk, off);
      mq += __shfl_xor_sync(0xffffffffu, mq, off);
    }
    const float delta = (vs[r][il] - mk) * beta;
    const float y = fmaf(delta, kq[r], mq);  // (S + delta k^T) q = S q + delta (k.q)
    const int rr = a.r0 + r;
    float* dst = a.S_slots[rr + (rr >= cur)] + ((long long)h * D + i) * D;
#pragma unroll
    for (int m = 0; m < NV4; ++m) {
      const float4 kv = *reinterpret_cast<const float4*>(&kn[r][4 * l + 4 * TPR * m]);
      s[4 * m] = fmaf(delta, kv.x, s[4 * m]);
      s[4 * m + 1] = fmaf(delta, kv.y, s[4 * m + 1]);
      s[4 * m + 2] = fmaf(delta, kv.z, s[4 * m + 2]);
      s[4 * m + 3] = fmaf(delta, kv.w, s[4 * m + 3]);
      *reinterpret_cast<float4*>(dst + 4 * l + 4 * TPR * m) =
          make_float4(s[4 * m], s[4 * m + 1], s[4 * m + 2], s[4 * m + 3]);
    }
    if (l == 0) ys[r][il] = y;
  }
  __syncthreads();

  // ---- 4. gated RMSNorm over the head's D value rows (cluster-wide sum)
  // The output gates do not depend on the sum: compute them first.
  float act[EPT];
#pragma unroll
  for (int h2 = 0; h2 < EPT; ++h2) {
    const float zz = bf16f(zin[h2]);
    act[h2] = a.gate_act == 1 ? siluf_(zz) : sigmoidf_(zz);
  }
  if (tid < k) {
    float ss = 0.f;
    for (int t = 0; t < kGdnRows; ++t) ss = fmaf(ys[tid][t], ys[tid][t], ss);
    ss_part[tid] = ss;
  }
  cluster_sync();
  // one remote load per (row, rank), all in flight together; then the sum in rank order
  if (tid < k * P) ss_all[tid / P][tid % P] = ld_dsmem_f32(&ss_part[tid / P], (uint32_t)(tid % P));
  cluster_arrive();  // this CTA has read its peers' sums
  __syncthreads();
  if (tid < k) {
    float tot = 0.f;
    for (int q = 0; q < P; ++q) tot += ss_all[tid][q];
    inv_s[tid] = 1.f / sqrtf(tot / (float)D + a.norm_eps);
  }
  __syncthreads();
#pragma unroll
  for (int h2 = 0; h2 < EPT; ++h2) {
    const int e = tid + h2 * NT;
    if (e >= k * kGdnRows) break;
    const int r = e / kGdnRows, ii = e % kGdnRows;
    const int iv = p * kGdnRows + ii;
    const float ov = ys[r][ii] * inv_s[r] * nw[h2] * act[h2];
    const long long oi = (long long)r * a.Hv * D + h * D + iv;
    if (a.dtype == 1) reinterpret_cast<uint16_t*>(a.o)[oi] = f2bf16(ov);
    else reinterpret_cast<float*>(a.o)[oi] = ov;
  }
  cluster_wait();  // keep this CTA's shared memory alive until every peer has read it
}

template <int D>
static cudaError_t launch_gdn_d(const GdnArgs& a, bool pdl, cudaStream_t s) {
  constexpr int P = GdnShape<D>::P;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.Hv * P);
  cfg.blockDim = dim3(GdnShape<D>::THREADS);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = P;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, gdn_verify_kernel<D>, a);
}

cudaError_t gdn_setup_kernels() { return cudaSuccess; }

cudaError_t launch_gdn(const GdnArgs& a, bool pdl, cudaStream_t s) {
  switch (a.d) {
    case 32: return launch_gdn_d<32>(a, pdl, s);
    case 64: return launch_gdn_d<64>(a, pdl, s);
    case 128: return launch_gdn_d<128>(a, pdl, s);
    default: return cudaErrorInvalidValue;
  }
}

// ------------------------------------------------------------------ glue

// out = x / sqrt(mean(x^2) + eps) * (zc ? 1 + w : w), one CTA of 256 threads
// per row.  Thread t holds elements t, t + 256, ... (VPT of them, n <= 256 VPT)
// in registers; the weights are static and are loaded before the dependency wait.
template <int VPT>
__global__ void __launch_bounds__(256) rmsnorm_kernel(const float* x, const float* w, float eps, int zc, int n,
                                                      void* out, int dtype) {
  const int nt = blockDim.x, tid = threadIdx.x;
  float wt[VPT];
#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    const int c = i * nt + tid;
    wt[i] = c < n ? (zc ? 1.f + w[c] : w[c]) : 0.f;
  }
  // the kernel after a norm (a product) reads only its weights before its
  // own wait: it may start now and fetch them while this kernel's
  // predecessor finishes
  griddep_launch();
  griddep_wait();
  const int r = blockIdx.x;
  const float* xr = x + (long long)r * n;
  __shared__ float red[8];
  float v[VPT];
#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    const int c = i * nt + tid;
    v[i] = c < n ? xr[c] : 0.f;
  }
  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < VPT; ++i) ss = fmaf(v[i], v[i], ss);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
  if ((tid & 31) == 0) red[tid >> 5] = ss;
  __syncthreads();
  float tot = 0.f;
  for (int q = 0; q < (int)(blockDim.x >> 5); ++q) tot += red[q];
  const float inv = 1.f / sqrtf(tot / (float)n + eps);
#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    const int c = i * nt + tid;
    if (c >= n) break;
    const float o = v[i] * inv * wt[i];
    if (dtype == 1) reinterpret_cast<uint16_t*>(out)[(long long)r * n + c] = f2bf16(o);
    else reinterpret_cast<float*>(out)[(long long)r * n + c] = o;
  }
}

cudaError_t launch_rmsnorm(const float* x, const float* w, float eps, int zc, int n, int k, void* out, int dtype,
                           bool pdl, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(k);
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  if (n <= 256 * 4) return cudaLaunchKernelEx(&cfg, rmsnorm_kernel<4>, x, w, eps, zc, n, out, dtype);
  if (n <= 256 * 8) return cudaLaunchKernelEx(&cfg, rmsnorm_kernel<8>, x, w, eps, zc, n, out, dtype);
  if (n <= 256 * 16) return cudaLaunchKernelEx(&cfg, rmsnorm_kernel<16>, x, w, eps, zc, n, out, dtype);
  if (n <= 256 * 32) return cudaLaunchKernelEx(&cfg, rmsnorm_kernel<32>, x, w, eps, zc, n, out, dtype);
  return cudaLaunchKernelEx(&cfg, rmsnorm_kernel<64>, x, w, eps, zc, n, out, dtype);  // n <= 16384
}

}  // namespace vk
