// synth.cu - device twin of the host SplitMix64 input generator (bench inputs).
#include <cuda_bf16.h>

#include "verify_synth.h"

namespace {

__device__ __forceinline__ uint64_t draw(uint64_t seed, uint64_t i) {
  uint64_t z = seed + (i + 1) * 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

__device__ __forceinline__ float uniform_f32(uint64_t seed, uint64_t i, float lo, float span) {
  const float u = __fmul_rn((float)(draw(seed, i) >> 40), 5.9604644775390625e-8f);  // 2^-24
  return __fadd_rn(__fmul_rn(span, u), lo);
}

__device__ __forceinline__ uint16_t to_bf16(float v) { return __bfloat16_as_ushort(__float2bfloat16_rn(v)); }

__global__ void synth_q4_kernel(uint32_t* packed, uint16_t* scales, uint16_t* biases, int64_t n_words,
                                int64_t n_groups, uint64_t sp, uint64_t ss, uint64_t sb, float lo_s, float span_s,
                                float lo_b, float span_b, int centered) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n_words; i += stride)
    packed[i] = (uint32_t)draw(sp, (uint64_t)i);
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n_groups; i += stride) {
    const uint16_t sc = to_bf16(uniform_f32(ss, (uint64_t)i, lo_s, span_s));
    const float u = uniform_f32(sb, (uint64_t)i, lo_b, span_b);
    scales[i] = sc;
    biases[i] = centered ? to_bf16(-__fmul_rn(__uint_as_float((uint32_t)sc << 16), u)) : to_bf16(u);
  }
}

}  // namespace

extern "C" verify_status verify_synth_q4(verify_ctx* ctx, uint32_t* packed, uint16_t* scales, uint16_t* biases,
                                         int64_t n_words, int64_t n_groups, uint64_t seed_packed,
                                         uint64_t seed_scales, uint64_t seed_biases, float lo_s, float hi_s,
                                         float lo_b, float hi_b, int centered, struct CUstream_st* stream) {
  if (!ctx || !packed || !scales || !biases || n_words < 0 || n_groups < 0) return VERIFY_EINVAL;
  int sms = 0, dev = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  synth_q4_kernel<<<sms * 8, 256, 0, stream>>>(packed, scales, biases, n_words, n_groups, seed_packed, seed_scales,
                                               seed_biases, lo_s, hi_s - lo_s, lo_b, hi_b - lo_b, centered);
  return cudaGetLastError() == cudaSuccess ? VERIFY_OK : VERIFY_ECUDA;
}
