// kvq_merge.cuh — split-K merge of decode-attention partials (library-internal).
//
// Every part s (a split, or a cluster of splits) of a (batch row, kv head) leaves, per query head i, its running max
// m_s (log2 units), its denominator l_s and its unnormalised output o_s[c]. The
// exact softmax over all tokens is the log-sum-exp combination
//   M = max_s m_s,  out[c] = sum_s 2^(m_s - M) o_s[c] / sum_s 2^(m_s - M) l_s.
// The last CTA of a (batch row, kv head) to finish performs it: an atomic ticket
// decides who is last, nobody waits. Every load of the partials is independent of
// the others (all query heads at once), so the merge costs two memory latencies.
#pragma once

#include <cuda_runtime.h>

#include "kvq_common.cuh"
#include "kvq_kernels.h"

namespace kvq {

constexpr int kMaxSplits = 256;

constexpr int kMergeScratchFloats = kMaxGqa * kMaxSplits + kMaxGqa;

// Called by all 128 threads of the CTA after it wrote its partials (n_parts: partials of
// this CTA's pair). Returns after
// writing the outputs if this CTA was the last of its (batch row, kv head).
// `scratch`: shared memory of at least kMergeScratchFloats floats, free for reuse.
__device__ __forceinline__ void merge_if_last(const DecodeParams& p, int n_parts, int64_t slice, int64_t qrow0,
                                              float* scratch) {
  __shared__ int last_s;
  float (*w_s)[kMaxSplits] = reinterpret_cast<float (*)[kMaxSplits]>(scratch);
  float* inv_l_s = scratch + kMaxGqa * kMaxSplits;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    const uint32_t ticket = atomicAdd(&p.tickets[slice], 1u);
    last_s = (ticket == (uint32_t)(n_parts - 1));
  }
  __syncthreads();
  if (!last_s) return;
  __threadfence();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // weights 2^(m_s - M) and 1 / sum_s 2^(m_s - M) l_s; warp w handles query heads w, w + 4
  for (int i = warp; i < p.r; i += 4) {
    const float2* ml = p.ws_ml + (qrow0 + i) * p.cap;
    float2 v[kMaxSplits / 32];
    float M = -__int_as_float(0x7f800000);
#pragma unroll
    for (int k = 0; k < kMaxSplits / 32; ++k) {
      const int s = lane + 32 * k;
      v[k] = (s < n_parts) ? __ldcg(&ml[s]) : make_float2(-__int_as_float(0x7f800000), 0.0f);
      M = fmaxf(M, v[k].x);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    float L = 0.0f;
#pragma unroll
    for (int k = 0; k < kMaxSplits / 32; ++k) {
      const int s = lane + 32 * k;
      if (s < n_parts) {
        const float wt = exp2f(v[k].x - M);
        w_s[i][s] = wt;
        L += wt * v[k].y;
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) L += __shfl_xor_sync(0xffffffffu, L, off);
    if (lane == 0) inv_l_s[i] = 1.0f / L;
  }
  __syncthreads();
  // thread = channel; all (query, split) loads in flight together
  const int c = threadIdx.x;
  float acc[kMaxGqa];
#pragma unroll
  for (int i = 0; i < kMaxGqa; ++i) acc[i] = 0.0f;
  for (int s0 = 0; s0 < n_parts; s0 += 4) {
    float ov[kMaxGqa][4];
#pragma unroll
    for (int i = 0; i < kMaxGqa; ++i)
#pragma unroll
      for (int u = 0; u < 4; ++u)
        ov[i][u] = (i < p.r && s0 + u < n_parts)
                       ? __ldcg(p.ws_o + ((qrow0 + i) * p.cap + s0 + u) * kHeadDim + c)
                       : 0.0f;
#pragma unroll
    for (int i = 0; i < kMaxGqa; ++i)
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (i < p.r && s0 + u < n_parts) acc[i] = fmaf(w_s[i][s0 + u], ov[i][u], acc[i]);
  }
#pragma unroll
  for (int i = 0; i < kMaxGqa; ++i)
    if (i < p.r) p.out[(qrow0 + i) * kHeadDim + c] = acc[i] * inv_l_s[i];
  if (threadIdx.x == 0) p.tickets[slice] = 0u;  // ready for the next call
}

}  // namespace kvq
