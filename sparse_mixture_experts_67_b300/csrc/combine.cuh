// Weighted combine and load-balancing statistics.
//
// Combine: y_t = sum_j w[t,j] * E_{idx[t,j]}(x_t), the accumulation of
// MoELayer.forward in "Mixture of Experts（MoE）の理論と実装" and of
// MoELayerWithAuxLoss.forward in "Sparse Mixture of Experts(MoE) 아키텍처 심층
// 분석".  One warp per token, float4 columns, slots summed in order j = 0..k-1
// (deterministic), skipping slots without a dispatch row (inv_perm < 0:
// dropped by capacity-limited routing).  Expert choice sums the experts that
// picked the token in ascending expert order, weighted by the raw
// dispatch-mask score.
//
// Aux: f_e = count_e / T, p_e = mean_t g[t,e], loss = E * sum_e f_e p_e, the
// load_balancing_loss of the first page; optionally also the convention of
// compute_load_balancing_loss in the second: f_frac_e = count_e / (T k),
// loss_frac = loss / k; and the router z-loss of the second page, the mean of
// the squared log-sum-exps, from the router's per-tile sums.  p is reduced from per-block partial
// sums in a fixed order, so the result does not depend on scheduling.
#pragma once

#include "common.cuh"
#include "router.cuh"

namespace moe {

constexpr int kCombineThreads = 256;

__global__ void __launch_bounds__(kCombineThreads)
    combine_kernel(const float4* __restrict__ y_perm, const int32_t* __restrict__ inv_perm,
                   const float* __restrict__ w, int T, int d4, int k, float4* __restrict__ y) {
  pdl_begin();
  const int lane = threadIdx.x & 31;
  const int warps = gridDim.x * (kCombineThreads / 32);
  for (int t = blockIdx.x * (kCombineThreads / 32) + (threadIdx.x >> 5); t < T; t += warps) {
    for (int c0 = 0; c0 < d4; c0 += 32 * 8) {
      float4 acc[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int j = 0; j < k; ++j) {
        const int row = inv_perm[(size_t)t * k + j];
        if (row < 0) continue;  // dropped by the expert's capacity
        const float wj = w[(size_t)t * k + j];
        const float4* src = y_perm + (size_t)row * d4;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int c = c0 + lane + 32 * i;
          if (c < d4) {
            const float4 v = __ldg(src + c);
            acc[i].x = fmaf(wj, v.x, acc[i].x);
            acc[i].y = fmaf(wj, v.y, acc[i].y);
            acc[i].z = fmaf(wj, v.z, acc[i].z);
            acc[i].w = fmaf(wj, v.w, acc[i].w);
          }
        }
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int c = c0 + lane + 32 * i;
        if (c < d4) y[(size_t)t * d4 + c] = acc[i];
      }
    }
  }
}

__global__ void __launch_bounds__(kCombineThreads)
    ec_combine_kernel(const float4* __restrict__ y_perm, const int32_t* __restrict__ pos,
                      const float* __restrict__ score, int T, int d4, int E,
                      float4* __restrict__ y) {
  pdl_begin();
  const int lane = threadIdx.x & 31;
  const int warps = gridDim.x * (kCombineThreads / 32);
  for (int t = blockIdx.x * (kCombineThreads / 32) + (threadIdx.x >> 5); t < T; t += warps) {
    for (int c0 = 0; c0 < d4; c0 += 32 * 8) {
      float4 acc[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int e0 = 0; e0 < E; e0 += 32) {
        const int e = e0 + lane;
        const int p = (e < E) ? pos[(size_t)e * T + t] : -1;
        unsigned hit = __ballot_sync(kFullMask, p >= 0);
        while (hit) {  // ascending expert order, two experts' rows in flight at a time
          const int la = __ffs(hit) - 1;
          hit &= hit - 1;
          const int lb = hit ? __ffs(hit) - 1 : -1;
          if (hit) hit &= hit - 1;
          const int ra = __shfl_sync(kFullMask, p, la);
          const int rb = __shfl_sync(kFullMask, p, lb < 0 ? la : lb);
          const float sa = score[ra];
          const float sb = lb < 0 ? 0.f : score[rb];
          const float4* srca = y_perm + (size_t)ra * d4;
          const float4* srcb = y_perm + (size_t)rb * d4;
          float4 va[8], vb[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int c = c0 + lane + 32 * i;
            if (c < d4) {
              va[i] = __ldg(srca + c);
              if (lb >= 0) vb[i] = __ldg(srcb + c);
            }
          }
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int c = c0 + lane + 32 * i;
            if (c < d4) {
              acc[i].x = fmaf(sa, va[i].x, acc[i].x);
              acc[i].y = fmaf(sa, va[i].y, acc[i].y);
              acc[i].z = fmaf(sa, va[i].z, acc[i].z);
              acc[i].w = fmaf(sa, va[i].w, acc[i].w);
              if (lb >= 0) {
                acc[i].x = fmaf(sb, vb[i].x, acc[i].x);
                acc[i].y = fmaf(sb, vb[i].y, acc[i].y);
                acc[i].z = fmaf(sb, vb[i].z, acc[i].z);
                acc[i].w = fmaf(sb, vb[i].w, acc[i].w);
              }
            }
          }
        }
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int c = c0 + lane + 32 * i;
        if (c < d4) y[(size_t)t * d4 + c] = acc[i];
      }
    }
  }
}

// Per-block partial column sums of probs [T,E] in the router's block layout
// (blocks of tok tokens).
__global__ void probs_partials_kernel(const float* __restrict__ probs, int T, int E, int tok,
                                      float* __restrict__ partials) {
  pdl_begin();
  const int t0 = blockIdx.x * tok;
  const int t1 = min(T, t0 + tok);
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    float s = 0.f;
    for (int t = t0; t < t1; ++t) s += probs[(size_t)t * E + e];
    partials[(size_t)blockIdx.x * E + e] = s;
  }
}

// One CTA of kAuxThreads.  Below 32 experts warp w reduces experts w, w + 8,
// ...: each lane sums a fixed strided subset of the partial rows, then a fixed
// butterfly.  From 32 experts on the rows are read whole (lanes over experts,
// warp w summing rows w, w + 8, ... in order; coalesced, where the column walk
// touches a line per lane) and the warps' sums are added in warp order.  Both
// orders are fixed: deterministic.
constexpr int kAuxThreads = 256;
__global__ void __launch_bounds__(kAuxThreads)
    aux_finalize_kernel(const float* __restrict__ partials, int rows, const int32_t* __restrict__ counts,
                        int T, int E, int k, float* __restrict__ f, float* __restrict__ p,
                        float* __restrict__ loss, float* __restrict__ f_frac,
                        float* __restrict__ loss_frac, const float* __restrict__ z_partials,
                        float* __restrict__ z_loss) {
  pdl_begin();
  __shared__ float s[MOE_MAX_EXPERTS];
  constexpr int nwarps = kAuxThreads / 32;
  __shared__ float s_w[nwarps][MOE_MAX_EXPERTS];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int e = threadIdx.x; e < MOE_MAX_EXPERTS; e += kAuxThreads) s[e] = 0.f;
  if (E >= 32) {
    for (int e = lane; e < E; e += 32) {
      float acc = 0.f;
      for (int r = warp; r < rows; r += nwarps) acc += partials[(size_t)r * E + e];
      s_w[warp][e] = acc;
    }
  }
  __syncthreads();
  for (int e = warp; e < E; e += nwarps) {
    float acc = 0.f;
    if (E >= 32) {
      if (lane == 0)
        for (int w = 0; w < nwarps; ++w) acc += s_w[w][e];
    } else {
      for (int r = lane; r < rows; r += 32) acc += partials[(size_t)r * E + e];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(kFullMask, acc, off);
    }
    if (lane == 0) {
      const float pe = acc / (float)T;
      const float fe = (float)counts[e] / (float)T;
      if (p) p[e] = pe;
      if (f) f[e] = fe;
      if (f_frac) f_frac[e] = (float)counts[e] / ((float)T * (float)k);
      s[e] = fe * pe;
    }
  }
  __syncthreads();
  for (int off = MOE_MAX_EXPERTS / 2; off > 0; off >>= 1) {
    for (int e = threadIdx.x; e < off; e += kAuxThreads) s[e] += s[e + off];
    __syncthreads();
  }
  if (threadIdx.x == 0 && loss) *loss = (float)E * s[0];
  if (threadIdx.x == 0 && loss_frac) *loss_frac = (float)E * s[0] / (float)k;
  if (warp == 0 && z_partials && z_loss) {  // router z-loss: fixed-order mean
    float acc = 0.f;
    for (int r = lane; r < rows; r += 32) acc += z_partials[r];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(kFullMask, acc, off);
    if (lane == 0) *z_loss = acc / (float)T;
  }
}

}  // namespace moe
