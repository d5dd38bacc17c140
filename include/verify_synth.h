/*
 * verify_synth.h - device-side twin of the seeded input generator.
 *
 * Not part of the verification method: it fills multi-GB synthetic weight
 * tensors directly on the GPU for benchmarks, with exactly the bits the host
 * generator (speculative_decode_verification_gb300/synth.py) produces for the
 * same seeds, so the CPU oracle can re-draw any sampled row on the host.
 *
 * Generator: SplitMix64 (Steele, Lea, Flood, OOPSLA 2014) used as a counter:
 * element i of a tensor with seed s is mix64(s + (i + 1) * 0x9E3779B97F4A7C15).
 */
#ifndef VERIFY_SYNTH_H_
#define VERIFY_SYNTH_H_

#include <stdint.h>

#include "verify.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * packed[i] = low 32 bits of draw i of seed_packed        (i < n_words)
 * scales[i] = bf16(lo_s + (hi_s - lo_s) * u_i)              (i < n_groups)
 * biases[i] = bf16(lo_b + (hi_b - lo_b) * u_i)                 (centered == 0)
 *            bf16(-(scales[i] * (lo_b + (hi_b - lo_b) * u_i)))  (centered != 0)
 * with u_i = (draw i >> 40) * 2^-24 and every step an fp32 IEEE operation
 * ((hi - lo) is rounded to fp32 first; scales[i] is the stored bf16 value),
 * bf16 rounding to nearest-even.
 * All pointers are device memory; asynchronous on `stream`.
 */
verify_status verify_synth_q4(verify_ctx* ctx, uint32_t* packed, uint16_t* scales, uint16_t* biases,
                              int64_t n_words, int64_t n_groups, uint64_t seed_packed, uint64_t seed_scales,
                              uint64_t seed_biases, float lo_s, float hi_s, float lo_b, float hi_b,
                              int centered, struct CUstream_st* stream);

#ifdef __cplusplus
}
#endif

#endif /* VERIFY_SYNTH_H_ */
