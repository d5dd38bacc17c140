// Greedy acceptance of a verify block on the device, fused with the commit of
// every Gated DeltaNet state ("Red Lite dev45 - speculative decoding with the
// Qwen3-Next MTP block", sections "What it is" and "Acceptance").
//
// Row r's greedy choice t_r is the argmax of its logits.  Each CTA scans a
// contiguous slice of one row and folds it into one 64-bit key,
//   (order-preserving bits of the logit) << 32 | (2^32 - 1 - index),
// so that the largest key is the largest logit and, among equal logits, the
// lowest index.  -0 is keyed as +0 and every NaN as the top key, so the
// result is numpy's argmax.  The key max is exact and order-free: the CTAs
// merge with one 64-bit atomicMax per CTA into a per-row scratch word, and the
// last CTA to finish (a ticket counter) reads the k winners, computes the
// accepted prefix, writes the result, commits the states and zeroes the
// scratch for the next call.  No CTA waits on another.
//
// Bound: HBM, k * V * 4 bytes of logits read once (8.9 MB at k = 9 over a
// 248,320-entry vocabulary); the grid is sized to about four CTAs per SM.
#include <cuda_runtime.h>
#include <stdint.h>

#include "argmax.cuh"
#include "common.cuh"
#include "internal.h"

namespace vk {
namespace {

// Commits `acc` rows on every state, all or nothing (one CTA, all threads).
__device__ void commit_states(const AcceptArgs& p, int acc) {
  __shared__ int bad;
  if (threadIdx.x == 0) bad = 0;
  __syncthreads();
  for (int l = threadIdx.x; l < p.n_states; l += blockDim.x) {
    const int pend = p.dev_state[2 * l + 1];
    if (pend <= 0 || acc < 0 || acc > pend || (p.need_k > 0 && pend != p.need_k)) atomicOr(&bad, 1);
  }
  __syncthreads();
  if (bad) {
    if (threadIdx.x == 0) record_error(p.err, VERIFY_DEV_ESEQUENCE);
    return;
  }
  for (int l = threadIdx.x; l < p.n_states; l += blockDim.x) {
    const int cur = p.dev_state[2 * l];
    p.dev_state[2 * l] = committed_slot(cur, acc);
    p.dev_state[2 * l + 1] = 0;
  }
}

// The k winners (read and reset), the accepted prefix by one warp ballot, the
// result, then the commit; ticket: also reset the ticket.  One CTA, all threads.
__device__ void finish(const AcceptArgs& p, bool ticket) {
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  __shared__ int acc_sh;
  if (w == 0) {  // lane r < k: row r's winner and draft d_{r+1}, then one ballot
    int t = 0;
    bool match = false;
    if (lane < p.k) {
      const int d = lane < p.k - 1 ? __ldcg(p.draft + lane) : 0;
      const unsigned long long b = atomicExch(p.best + lane, 0ull);  // read and reset for the next call
      t = argmax_index(b);
      match = lane < p.k - 1 && d == t;
      p.result[2 + lane] = t;
    }
    const int m = __ffs(~__ballot_sync(0xffffffffu, match)) - 1;  // leading drafts that stand
    const int tm = __shfl_sync(0xffffffffu, t, m);
    if (lane == 0) {
      p.result[0] = m + 1;
      p.result[1] = tm;
      acc_sh = m + 1;
      if (ticket) *p.ticket = 0u;
    }
  }
  __syncthreads();
  if (p.n_states > 0) commit_states(p, acc_sh);
}

__global__ void __launch_bounds__(kAcceptThreads) accept_kernel(const AcceptArgs p) {
  constexpr int NW = kAcceptThreads / 32;
  __shared__ unsigned long long warp_best[NW];
  __shared__ int is_last;
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;

  if (p.V == 0) {  // commit only
    const int acc = __ldcg(p.accepted);
    commit_states(p, acc);
    return;
  }
  if (p.V < 0) {  // the keys were merged by the LM head's argmax epilogue
    finish(p, false);
    return;
  }

  // ---- this CTA's slice of row r
  const int r = blockIdx.x / p.blocks_per_row;
  const int part = blockIdx.x % p.blocks_per_row;
  const int per = ((p.V + p.blocks_per_row - 1) / p.blocks_per_row + 3) & ~3;
  const int lo = part * per;
  const int hi = max(lo, min(p.V, lo + per));  // the last slices may be empty
  const float* row = p.logits + (long long)r * p.ld;
  unsigned long long best = 0ull;
  int v0 = lo;
  if (p.vec) {
    const int n4 = (hi - lo) >> 2;
    const float4* row4 = reinterpret_cast<const float4*>(row + lo);
    constexpr int U = 4;
    int j = tid;
    for (; j + (U - 1) * kAcceptThreads < n4; j += U * kAcceptThreads) {
      float4 q[U];
#pragma unroll
      for (int u = 0; u < U; ++u) q[u] = __ldcs(row4 + j + u * kAcceptThreads);
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int v = lo + 4 * (j + u * kAcceptThreads);
        best = umax64(best, argmax_key(q[u].x, v));
        best = umax64(best, argmax_key(q[u].y, v + 1));
        best = umax64(best, argmax_key(q[u].z, v + 2));
        best = umax64(best, argmax_key(q[u].w, v + 3));
      }
    }
    for (; j < n4; j += kAcceptThreads) {
      const float4 q = __ldcs(row4 + j);
      const int v = lo + 4 * j;
      best = umax64(best, argmax_key(q.x, v));
      best = umax64(best, argmax_key(q.y, v + 1));
      best = umax64(best, argmax_key(q.z, v + 2));
      best = umax64(best, argmax_key(q.w, v + 3));
    }
    v0 = lo + 4 * n4;
  }
  for (int v = v0 + tid; v < hi; v += kAcceptThreads) best = umax64(best, argmax_key(__ldcs(row + v), v));

  // ---- CTA max, one atomic per CTA
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) best = umax64(best, __shfl_xor_sync(0xffffffffu, best, off));
  if (lane == 0) warp_best[w] = best;
  __syncthreads();
  if (tid == 0) {
    unsigned long long b = warp_best[0];
#pragma unroll
    for (int i = 1; i < NW; ++i) b = umax64(b, warp_best[i]);
    if (lo < hi) atomicMax(p.best + r, b);
    __threadfence();
    is_last = atomicAdd(p.ticket, 1u) == gridDim.x - 1;
  }
  __syncthreads();
  if (!is_last) return;

  // ---- last CTA: every other CTA's atomicMax happened before its ticket
  __threadfence();
  finish(p, true);
}

}  // namespace

int accept_blocks_per_row(int V, int k, int num_sms) {
  // about four CTAs per SM over all rows, and at least 1024 logits per CTA
  const int by_size = (V + 1023) / 1024;
  const int by_grid = (4 * num_sms + k - 1) / k;
  int b = by_size < by_grid ? by_size : by_grid;
  return b < 1 ? 1 : b;
}

cudaError_t launch_accept(const AcceptArgs& a, cudaStream_t s) {
  const int grid = a.V <= 0 ? 1 : a.k * a.blocks_per_row;
  accept_kernel<<<grid, kAcceptThreads, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace vk
