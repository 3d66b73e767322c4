// Dispatch: per-expert histogram, exclusive scan, stable permutation, row gather.
//
// Groups the T*k (token, slot) assignments by expert the way the per-expert
// masks of MoELayerWithAuxLoss and the argsort of ExpertParallelRouter.dispatch
// do in "Sparse Mixture of Experts(MoE) 아키텍처 심층 분석" (youngju.dev), with
// the order inside an expert fixed to ascending assignment id a = t*k + j.
//
// Three small kernels make it deterministic without a global sort:
//   hist:    each tile of kDispatchTile assignments counts its experts with
//            warp-aggregated shared-memory atomics (match_any + popc);
//   scan:    one CTA turns the [tiles, E] count matrix into per-(tile, expert)
//            bases and the expert offsets (exclusive scan over experts);
//   scatter: each tile re-reads its assignments in order and ranks them among
//            equal experts (warp match_any rank + per-warp counts in shared
//            memory), giving perm / inv_perm bit-exactly.
// The row gather then copies x rows into the dispatch order with 16-byte
// vector loads, one warp per row.
#pragma once

#include "common.cuh"

namespace moe {

constexpr int kDispatchTile = 2048;
constexpr int kDispatchThreads = 256;
constexpr int kDispatchWarps = kDispatchThreads / 32;

inline int dispatch_tiles(long long A) { return A == 0 ? 0 : ceil_div(A, kDispatchTile); }

__global__ void __launch_bounds__(kDispatchThreads)
    dispatch_hist_kernel(const int32_t* __restrict__ idx, int A, int E, int32_t* __restrict__ tile_counts) {
  __shared__ int cnt[MOE_MAX_EXPERTS];
  for (int e = threadIdx.x; e < E; e += blockDim.x) cnt[e] = 0;
  __syncthreads();
  const int a0 = blockIdx.x * kDispatchTile;
  const int a1 = min(A, a0 + kDispatchTile);
  const int lane = threadIdx.x & 31;
  for (int base = a0; base < a1; base += kDispatchThreads) {
    const int a = base + threadIdx.x;
    const bool valid = a < a1;
    const int e = valid ? idx[a] : -1;
    const unsigned peers = __match_any_sync(kFullMask, e);
    if (valid && lane == __ffs(peers) - 1) atomicAdd(&cnt[e], __popc(peers));
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) tile_counts[(size_t)blockIdx.x * E + e] = cnt[e];
}

// One CTA of MOE_MAX_EXPERTS threads.  tile_base[tile][e] becomes the first
// dispatch row of expert e's assignments that fall in `tile`.
__global__ void __launch_bounds__(MOE_MAX_EXPERTS)
    dispatch_scan_kernel(const int32_t* __restrict__ tile_counts, int tiles, int E, int A,
                         int32_t* __restrict__ tile_base, int32_t* __restrict__ counts,
                         int32_t* __restrict__ offsets) {
  __shared__ int s[MOE_MAX_EXPERTS];
  const int e = threadIdx.x;
  int total = 0;
  if (e < E) {
    for (int t = 0; t < tiles; ++t) {
      const int c = tile_counts[(size_t)t * E + e];
      tile_base[(size_t)t * E + e] = total;
      total += c;
    }
  }
  s[e] = (e < E) ? total : 0;
  __syncthreads();
  // Hillis-Steele inclusive scan over the (<= 256) experts
  for (int off = 1; off < MOE_MAX_EXPERTS; off <<= 1) {
    const int v = (e >= off) ? s[e - off] : 0;
    __syncthreads();
    s[e] += v;
    __syncthreads();
  }
  if (e < E) {
    const int excl = s[e] - total;
    counts[e] = total;
    offsets[e] = excl;
    for (int t = 0; t < tiles; ++t) tile_base[(size_t)t * E + e] += excl;
  }
  if (e == 0) offsets[E] = A;
}

__global__ void __launch_bounds__(kDispatchThreads)
    dispatch_scatter_kernel(const int32_t* __restrict__ idx, int A, int E,
                            const int32_t* __restrict__ tile_base, int32_t* __restrict__ perm,
                            int32_t* __restrict__ inv_perm) {
  __shared__ int running[MOE_MAX_EXPERTS];
  __shared__ int wcnt[kDispatchWarps][MOE_MAX_EXPERTS];
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    running[e] = tile_base[(size_t)blockIdx.x * E + e];
    for (int w = 0; w < kDispatchWarps; ++w) wcnt[w][e] = 0;
  }
  __syncthreads();
  const int a0 = blockIdx.x * kDispatchTile;
  const int a1 = min(A, a0 + kDispatchTile);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int base = a0; base < a1; base += kDispatchThreads) {
    const int a = base + threadIdx.x;
    const bool valid = a < a1;
    const int e = valid ? idx[a] : -1;
    const unsigned peers = __match_any_sync(kFullMask, e);
    const int rank = __popc(peers & lanemask_lt());
    if (valid && lane == __ffs(peers) - 1) wcnt[warp][e] = __popc(peers);
    __syncthreads();
    if (valid) {
      int row = running[e] + rank;
      for (int w = 0; w < warp; ++w) row += wcnt[w][e];
      perm[row] = a;
      inv_perm[a] = row;
    }
    __syncthreads();
    for (int ee = threadIdx.x; ee < E; ee += blockDim.x) {
      int s = 0;
#pragma unroll
      for (int w = 0; w < kDispatchWarps; ++w) {
        s += wcnt[w][ee];
        wcnt[w][ee] = 0;
      }
      running[ee] += s;
    }
    __syncthreads();
  }
}

// x_perm[r,:] = x[src[r] / div, :]; one warp per row, 16-byte vectors.
constexpr int kGatherThreads = 256;
__global__ void __launch_bounds__(kGatherThreads)
    gather_rows_kernel(const uint4* __restrict__ x, const int32_t* __restrict__ src, int R, int div,
                       int vec_per_row, uint4* __restrict__ out) {
  const int lane = threadIdx.x & 31;
  const int warps = gridDim.x * (kGatherThreads / 32);
  for (int r = blockIdx.x * (kGatherThreads / 32) + (threadIdx.x >> 5); r < R; r += warps) {
    const int t = src[r] / div;
    const uint4* srow = x + (size_t)t * vec_per_row;
    uint4* drow = out + (size_t)r * vec_per_row;
    int v = lane;
    for (; v + 96 < vec_per_row; v += 128) {
      const uint4 a = __ldg(srow + v), b = __ldg(srow + v + 32), c = __ldg(srow + v + 64),
                  dd = __ldg(srow + v + 96);
      drow[v] = a;
      drow[v + 32] = b;
      drow[v + 64] = c;
      drow[v + 96] = dd;
    }
    for (; v < vec_per_row; v += 32) drow[v] = __ldg(srow + v);
  }
}

}  // namespace moe

namespace moe {

// Expert-choice segments are uniform: offsets[e] = e * C, e = 0..E.
__global__ void uniform_offsets_kernel(int32_t* __restrict__ offsets, int E, int C) {
  for (int e = threadIdx.x; e <= E; e += blockDim.x) offsets[e] = e * C;
}

}  // namespace moe
