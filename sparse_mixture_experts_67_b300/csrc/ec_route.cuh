// Expert-choice routing: ExpertChoiceGating.forward of "Sparse Mixture of
// Experts(MoE) 아키텍처 심층 분석" (youngju.dev).
//
// Each expert scores all tokens with a softmax over its logit column and keeps
// the C best tokens, C = floor(T * capacity_factor / E).  One CTA per expert,
// each thread owning a contiguous run of tokens:
//   - the column max and the sum of exponentials are block reductions;
//   - a radix select (four 8-bit passes over order-preserving 32-bit keys)
//     finds the C-th best logit;
//   - ordered block scans keep every token above it plus, among the tokens
//     equal to it, the lowest token ids (ties go to the lower token);
//   - only the C picks are sorted (bitonic, in shared memory) by descending
//     logit then ascending token, the output order.
// The logits come from the router kernel run in logits-only mode, which also
// writes them transposed into pos ([E, T], as fp32 bits): CTA e reads its row
// there once, coalesced, keeps the order-preserving keys in shared memory and
// only then overwrites the row with the position map.
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

// Inverse of float_order_key (exact; -0 comes back as +0).
__device__ __forceinline__ float order_key_float(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

inline int next_pow2_host(int v) {
  int p = 1;
  while (p < v) p <<= 1;
  return p;
}

// Exclusive prefix sum over the CTA in thread order; *total gets the sum.
__device__ __forceinline__ int block_exclusive_scan(int v, int* s_warp, int* total) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  int incl = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int n = __shfl_up_sync(kFullMask, incl, off);
    if (lane >= off) incl += n;
  }
  if (lane == 31) s_warp[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int w = lane < nw ? s_warp[lane] : 0;
    int winc = w;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int n = __shfl_up_sync(kFullMask, winc, off);
      if (lane >= off) winc += n;
    }
    s_warp[lane] = winc - w;
    if (lane == 31) s_warp[32] = winc;
  }
  __syncthreads();
  const int res = s_warp[warp] + incl - v;
  *total = s_warp[32];
  __syncthreads();
  return res;
}

inline size_t ec_route_smem(int T, int C) {
  return (((size_t)T * 4 + 15) & ~size_t(15)) + (size_t)next_pow2_host(C) * 8;
}

__global__ void __launch_bounds__(kEcThreads)
    ec_route_kernel(int T, int E, int C, int c_pow2, int32_t* __restrict__ ec_idx,
                    float* __restrict__ ec_score, int32_t* __restrict__ pos) {
  pdl_begin();
  extern __shared__ __align__(16) unsigned char ec_smem[];
  uint32_t* s_key = reinterpret_cast<uint32_t*>(ec_smem);  // ascending = descending logit
  unsigned long long* s_sel = reinterpret_cast<unsigned long long*>(
      ec_smem + (((size_t)T * 4 + 15) & ~size_t(15)));
  __shared__ float scratch[32];
  __shared__ int s_warp[33];
  __shared__ int s_hist[256];
  __shared__ uint32_t s_prefix;
  __shared__ int s_remaining;
  const int e = blockIdx.x;
  const int per = (T + kEcThreads - 1) / kEcThreads;
  const int t0 = min(T, threadIdx.x * per), t1 = min(T, t0 + per);

  int32_t* prow = pos + (size_t)e * T;  // on entry: this expert's logits (fp32 bits)
  float m = -FLT_MAX;
  for (int t = threadIdx.x; t < T; t += blockDim.x) {  // coalesced
    const float v = __int_as_float(prow[t]);
    m = fmaxf(m, v);
    s_key[t] = ~float_order_key(v);
  }
  m = block_reduce_max(m, scratch);  // every read of the row is done past this barrier
  float sum = 0.f;
  for (int t = threadIdx.x; t < T; t += blockDim.x) {
    sum += expf(order_key_float(~s_key[t]) - m);
    prow[t] = -1;
  }
  sum = block_reduce_sum(sum, scratch);  // also publishes the pos writes to the CTA
  if (C <= 0) return;

  // radix select: the C-th smallest key K* and how many keys equal to it to take
  uint32_t prefix = 0, mask = 0;
  int remaining = C;
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int b = threadIdx.x; b < 256; b += blockDim.x) s_hist[b] = 0;
    __syncthreads();
    for (int t = t0; t < t1; ++t) {
      const uint32_t k = s_key[t];
      if ((k & mask) == prefix) atomicAdd(&s_hist[(k >> shift) & 255u], 1);
    }
    __syncthreads();
    if (threadIdx.x < 32) {
      const int lane = threadIdx.x;
      int loc = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) loc += s_hist[lane * 8 + i];
      int incl = loc;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int n = __shfl_up_sync(kFullMask, incl, off);
        if (lane >= off) incl += n;
      }
      int cum = incl - loc;
      if (cum < remaining && remaining <= incl) {
        for (int i = 0; i < 8; ++i) {
          const int h = s_hist[lane * 8 + i];
          if (remaining <= cum + h) {
            s_prefix = prefix | ((uint32_t)(lane * 8 + i) << shift);
            s_remaining = remaining - cum;
            break;
          }
          cum += h;
        }
      }
    }
    __syncthreads();
    prefix = s_prefix;
    remaining = s_remaining;
    mask |= 255u << shift;
  }
  // keep keys < K* and the first `remaining` keys == K* in token order
  int n_eq = 0;
  for (int t = t0; t < t1; ++t) n_eq += s_key[t] == prefix;
  int total;
  int eq_rank = block_exclusive_scan(n_eq, s_warp, &total);
  int n_sel = 0;
  {
    int r = eq_rank;
    for (int t = t0; t < t1; ++t) {
      const uint32_t k = s_key[t];
      if (k < prefix || (k == prefix && r++ < remaining)) ++n_sel;
    }
  }
  int slot = block_exclusive_scan(n_sel, s_warp, &total);
  {
    int r = eq_rank;
    for (int t = t0; t < t1; ++t) {
      const uint32_t k = s_key[t];
      if (k < prefix || (k == prefix && r++ < remaining))
        s_sel[slot++] = ((unsigned long long)k << 32) | (unsigned)t;
    }
  }
  for (int i = C + threadIdx.x; i < c_pow2; i += blockDim.x) s_sel[i] = ~0ull;
  __syncthreads();
  for (int kk = 2; kk <= c_pow2; kk <<= 1) {
    for (int j = kk >> 1; j > 0; j >>= 1) {
      for (int i = threadIdx.x; i < c_pow2; i += blockDim.x) {
        const int ixj = i ^ j;
        if (ixj > i) {
          const unsigned long long a = s_sel[i], b = s_sel[ixj];
          const bool up = (i & kk) == 0;
          if ((a > b) == up) {
            s_sel[i] = b;
            s_sel[ixj] = a;
          }
        }
      }
      __syncthreads();
    }
  }
  const float inv = 1.0f / sum;
  for (int c = threadIdx.x; c < C; c += blockDim.x) {
    const int t = (int)(s_sel[c] & 0xffffffffu);
    const float v = order_key_float((uint32_t)(s_sel[c] >> 32) ^ 0xffffffffu);
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
