// Expert-choice routing: ExpertChoiceGating.forward of "Sparse Mixture of
// Experts(MoE) 아키텍처 심층 분석" (youngju.dev).
//
// Each expert scores all tokens with a softmax over its logit column and keeps
// the C best tokens, C = floor(T * capacity_factor / E).  One CTA per expert:
// the column max and sum of exponentials are block reductions; the selection
// sorts 64-bit keys (descending logit as an order-preserving integer, then
// ascending token id) with a shared-memory bitonic sort, so ties go to the
// lower token and the output is in descending score order.  The logits come
// from the router kernel run in logits-only mode.
#pragma once

#include <float.h>

#include "common.cuh"

namespace moe {

constexpr int kEcThreads = 1024;
constexpr int kEcMaxTokens = 16384;

__device__ __forceinline__ float block_reduce_max(float v, float* scratch) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(kFullMask, v, off));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) scratch[warp] = v;
  __syncthreads();
  const int nw = blockDim.x >> 5;
  float r = scratch[0];
  for (int w = 1; w < nw; ++w) r = fmaxf(r, scratch[w]);
  __syncthreads();
  return r;
}

__device__ __forceinline__ float block_reduce_sum(float v, float* scratch) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(kFullMask, v, off);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) scratch[warp] = v;
  __syncthreads();
  const int nw = blockDim.x >> 5;
  float r = 0.f;
  for (int w = 0; w < nw; ++w) r += scratch[w];  // fixed order
  __syncthreads();
  return r;
}

// Order-preserving map of a float to uint32 (ascending float -> ascending key).
__device__ __forceinline__ uint32_t float_order_key(float v) {
  const uint32_t u = __float_as_uint(v + 0.0f);  // -0 -> +0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__global__ void __launch_bounds__(kEcThreads)
    ec_route_kernel(const float* __restrict__ logits, int T, int E, int C, int n_pow2,
                    int32_t* __restrict__ ec_idx, float* __restrict__ ec_score,
                    int32_t* __restrict__ pos) {
  extern __shared__ __align__(16) unsigned long long keys[];
  __shared__ float scratch[32];
  const int e = blockIdx.x;
  float m = -FLT_MAX;
  for (int t = threadIdx.x; t < T; t += blockDim.x) m = fmaxf(m, logits[(size_t)t * E + e]);
  m = block_reduce_max(m, scratch);
  float s = 0.f;
  for (int t = threadIdx.x; t < n_pow2; t += blockDim.x) {
    if (t < T) {
      const float v = logits[(size_t)t * E + e];
      s += expf(v - m);
      keys[t] = ((unsigned long long)(~float_order_key(v)) << 32) | (unsigned)t;
      pos[(size_t)e * T + t] = -1;
    } else {
      keys[t] = ~0ull;
    }
  }
  s = block_reduce_sum(s, scratch);  // contains __syncthreads: keys and pos are visible
  for (int kk = 2; kk <= n_pow2; kk <<= 1) {
    for (int j = kk >> 1; j > 0; j >>= 1) {
      for (int i = threadIdx.x; i < n_pow2; i += blockDim.x) {
        const int ixj = i ^ j;
        if (ixj > i) {
          const unsigned long long a = keys[i], b = keys[ixj];
          const bool up = (i & kk) == 0;
          if ((a > b) == up) {
            keys[i] = b;
            keys[ixj] = a;
          }
        }
      }
      __syncthreads();
    }
  }
  const float inv = 1.0f / s;
  for (int c = threadIdx.x; c < C; c += blockDim.x) {
    const int t = (int)(keys[c] & 0xffffffffu);
    const float v = logits[(size_t)t * E + e];
    ec_idx[(size_t)e * C + c] = t;
    ec_score[(size_t)e * C + c] = expf(v - m) * inv;
    pos[(size_t)e * T + t] = e * C + c;
  }
}

inline int next_pow2(int v) {
  int p = 1;
  while (p < v) p <<= 1;
  return p;
}

}  // namespace moe
