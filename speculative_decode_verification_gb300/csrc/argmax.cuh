// Greedy-choice helpers shared by the acceptance kernel and the LM-head
// product's argmax epilogue.
#pragma once
#include <stdint.h>

namespace vk {

// Order-preserving 64-bit key of logit f at vocabulary index v: the largest
// key is the largest logit and, among equal logits, the lowest index; -0 is
// keyed as +0 and every NaN as the top key (numpy's argmax).
__device__ __forceinline__ unsigned long long argmax_key(float f, int v) {
  uint32_t u = __float_as_uint(f);
  uint32_t key;
  if (f != f) {
    key = 0xFFFFFFFFu;
  } else {
    if (f == 0.f) u = 0u;
    key = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  }
  return ((unsigned long long)key << 32) | (0xFFFFFFFFu - (uint32_t)v);
}

__device__ __forceinline__ unsigned long long umax64(unsigned long long a, unsigned long long b) {
  return a > b ? a : b;
}

__device__ __forceinline__ int argmax_index(unsigned long long key) {
  return (int)(0xFFFFFFFFu - (uint32_t)(key & 0xFFFFFFFFull));
}

// Slot that becomes committed when `a` rows of the pending verify stand: the
// state after the first a rows was written to slot a-1 + (a-1 >= cur).
__device__ __forceinline__ int committed_slot(int cur, int a) {
  return a == 0 ? cur : (a - 1) + ((a - 1) >= cur ? 1 : 0);
}

}  // namespace vk
