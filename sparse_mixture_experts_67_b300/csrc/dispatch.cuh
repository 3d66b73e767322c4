// Dispatch: per-expert histogram, exclusive scan, stable permutation, row gather.
//
// Groups the T*k (token, slot) assignments by expert the way the per-expert
// masks of MoELayerWithAuxLoss and the argsort of ExpertParallelRouter.dispatch
// do in "Sparse Mixture of Experts(MoE) 아키텍처 심층 분석" (youngju.dev), with
// the order inside an expert fixed to ascending assignment id a = t*k + j.
//
// Deterministic without a global sort, in tiles of `tile` consecutive
// assignments (the layer uses one tile per router CTA):
//   hist:    per-tile expert counts with warp-aggregated shared-memory
//            atomics (match_any + popc); in the layer the router's epilogue
//            produces them instead;
//   scatter: each tile derives its per-expert bases from the count matrix,
//            re-reads its assignments in order and ranks them among equal
//            experts (warp match_any rank + per-warp counts in shared memory),
//            giving perm / inv_perm bit-exactly, and copies its rows (with
//            few tiles, two CTAs share a tile: both rank, one writes).
#pragma once

#include "common.cuh"

namespace moe {

constexpr int kDispatchThreads = 256;
constexpr int kDispatchWarps = kDispatchThreads / 32;

inline int dispatch_tiles(long long A, int tile) { return A == 0 ? 0 : ceil_div(A, tile); }

__global__ void __launch_bounds__(kDispatchThreads)
    dispatch_hist_kernel(const int32_t* __restrict__ idx, int A, int E, int tile,
                         int32_t* __restrict__ tile_counts) {
  pdl_begin();
  __shared__ int cnt[MOE_MAX_EXPERTS];
  for (int e = threadIdx.x; e < E; e += blockDim.x) cnt[e] = 0;
  __syncthreads();
  const int a0 = blockIdx.x * tile;
  const int a1 = min(A, a0 + tile);
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

// Ranks each assignment of its tile among equal experts and writes perm /
// inv_perm.  The tile's first dispatch row per expert comes from tile_base
// when given (dispatch_scan_kernel), else from the count matrix directly:
// every CTA reduces the [tiles, E] counts itself (totals, and the sum over
// the tiles before its own; below 32 experts a warp per expert with lanes over
// tiles, from 32 on lanes over experts and warps over tiles, so each load
// reads a whole row); the expert
// offsets are the exclusive scan of the totals, and CTA 0 also writes counts /
// offsets and, given aux_partials, the load-balancing statistics (same
// reduction order as aux_finalize_kernel).
// cap (capacity-limited token choice; INT_MAX: none): an expert's segment
// holds its first cap assignments in assignment order, i.e. in token order;
// later ones are dropped (inv_perm -1, no row).  With w_cap != nullptr the
// [T, k] weights of the tile's tokens are then renormalised over their kept
// slots in place (0 on dropped slots; all 0 for a token with none kept).
// dropped (nullable, CTA 0) gets the number of dropped assignments.
// Optional extras:
// x != nullptr copies x[a / k] into x_perm[row] (16-byte vectors, warp per
// row); y_zero != nullptr zeroes the y rows of the tile's tokens
// (tokens_per_tile of them) for an accumulating combine downstream.
// Large count matrices: dispatch_scan_kernel computes every tile's first
// dispatch row per expert (tile_base), the counts and the offsets, over all
// SMs in two launches (or in one CTA); the scatter CTAs then read their row of
// tile_base instead of reducing the whole matrix each.
// cap: per-expert capacity (INT_MAX: none).  Segments hold min(count, cap)
// rows; tile_base[t, e] is the segment start plus the expert's assignments in
// tiles before t, so a row at or past segment start + cap is a dropped one;
// dropped (nullable) gets the number of dropped assignments.
constexpr int kScanThreads = 1024;
// The scan over all SMs uses at most this many CTAs (block sums [nb, E]).
constexpr int kScanBlocks = 160;
// Modes of dispatch_scan_kernel.  kScanWhole: one CTA over all tiles.  Over
// nb CTAs, each owning a contiguous range of tiles: kScanBlockSums writes the
// range's per-expert sums to blk[b, E]; kScanBases (the next launch) takes the
// sums of the ranges before its own and of all ranges from blk and writes its
// rows of tile_base (CTA 0 also the counts, offsets and drops).
enum { kScanWhole = 0, kScanBlockSums = 1, kScanBases = 2 };
// EPL: experts per lane, ceil(E / 32).
template <int EPL>
__global__ void __launch_bounds__(kScanThreads)
    dispatch_scan_kernel(const int32_t* __restrict__ tile_counts, int tiles, int E, int A,
                         int32_t* __restrict__ tile_base, int32_t* __restrict__ counts,
                         int32_t* __restrict__ offsets, int cap, int32_t* __restrict__ dropped,
                         int mode, int32_t* __restrict__ blk) {
  pdl_begin();
  // Rows of the count matrix are read whole (a tile's E counts are contiguous):
  // the CTA's range of tiles is cut into nwarps blocks, warp w owning block w.
  // With E > 32 lane l takes experts l, l + 32, ...; with E <= 32 lane l takes
  // expert l % E of row l / E, so a warp step covers rpw = 32 / E rows (one
  // row from E = 17 on).  Each lane loads U steps before it uses any, to keep
  // several loads in flight.  Pass 1 sums each block per expert; the block
  // sums are scanned per expert (and, over several CTAs, offset by the ranges
  // before this one) and the totals across experts; pass 2 walks each block
  // again with a running base per expert and writes its rows of tile_base.
  constexpr int nwarps = kScanThreads / 32;
  constexpr int U = 4;
  __shared__ int s_tot[MOE_MAX_EXPERTS];
  __shared__ int s_off[MOE_MAX_EXPERTS];
  __shared__ int s_pre[MOE_MAX_EXPERTS];
  __shared__ int s_blk[nwarps][MOE_MAX_EXPERTS];
  __shared__ int s_part[2][kScanThreads];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nb = gridDim.x, bid = blockIdx.x;
  const int BR = (tiles + nb - 1) / nb;  // tiles per CTA range
  const int r0 = min(tiles, bid * BR), r1 = min(tiles, r0 + BR);
  const int B = (r1 - r0 + nwarps - 1) / nwarps;
  const int t0 = min(r1, r0 + warp * B), t1 = min(r1, t0 + B);
  const int rpw = EPL == 1 ? 32 / E : 1;
  const int r = EPL == 1 ? lane / E : 0;  // row of the step (r >= rpw: idle lane)
  int ex[EPL];
  bool on[EPL];
#pragma unroll
  for (int j = 0; j < EPL; ++j) {
    ex[j] = EPL == 1 ? lane % E : lane + 32 * j;
    on[j] = EPL == 1 ? r < rpw : ex[j] < E;
  }
  int sum[EPL];
#pragma unroll
  for (int j = 0; j < EPL; ++j) sum[j] = 0;
  for (int tb = t0; tb < t1; tb += U * rpw) {
    int v[U][EPL];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int t = tb + u * rpw + r;
#pragma unroll
      for (int j = 0; j < EPL; ++j)
        v[u][j] = on[j] && t < t1 ? tile_counts[(size_t)t * E + ex[j]] : 0;
    }
#pragma unroll
    for (int u = 0; u < U; ++u)
#pragma unroll
      for (int j = 0; j < EPL; ++j) sum[j] += v[u][j];
  }
  if constexpr (EPL == 1) {  // add the rows of a step: lane (r, e) takes (r + off, e)
    for (int off = 1; off < rpw; off <<= 1) {
      const int nb2 = __shfl_down_sync(kFullMask, sum[0], off * E);
      if (r + off < rpw) sum[0] += nb2;
    }
    if (lane < E) s_blk[warp][lane] = sum[0];
  } else {
#pragma unroll
    for (int j = 0; j < EPL; ++j)
      if (on[j]) s_blk[warp][ex[j]] = sum[j];
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += kScanThreads) {  // per expert: blocks' exclusive prefix
    int run = 0;
    for (int w = 0; w < nwarps; ++w) {
      const int v = s_blk[w][e];
      s_blk[w][e] = run;
      run += v;
    }
    s_tot[e] = run;  // this CTA's range
    s_pre[e] = 0;
  }
  if (mode == kScanBlockSums) {
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += kScanThreads) blk[(size_t)bid * E + e] = s_tot[e];
    return;
  }
  if (mode == kScanBases) {
    // the ranges before this one and all ranges, from the block sums: G groups
    // of E threads, group g taking ranges g, g + G, ... (integer sums: exact)
    const int G = max(1, kScanThreads / E);
    const int g = (int)threadIdx.x / E, e = (int)threadIdx.x - g * E;
    if (g < G) {
      int pre = 0, tot = 0;
      for (int b2 = g; b2 < nb; b2 += G) {
        const int v = blk[(size_t)b2 * E + e];
        tot += v;
        if (b2 < bid) pre += v;
      }
      s_part[0][threadIdx.x] = pre;
      s_part[1][threadIdx.x] = tot;
    }
    __syncthreads();
    for (int e2 = threadIdx.x; e2 < E; e2 += kScanThreads) {
      int pre = 0, tot = 0;
      for (int g2 = 0; g2 < G; ++g2) {
        pre += s_part[0][g2 * E + e2];
        tot += s_part[1][g2 * E + e2];
      }
      s_pre[e2] = pre;
      s_tot[e2] = tot;
    }
  }
  __syncthreads();
  if (warp == 0) {
    constexpr int per = MOE_MAX_EXPERTS / 32;
    const int e0 = lane * per;
    int run = 0;
    for (int e = e0; e < min(E, e0 + per); ++e) run += min(s_tot[e], cap);
    int incl = run;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int nb2 = __shfl_up_sync(kFullMask, incl, off);
      if (lane >= off) incl += nb2;
    }
    int exc = incl - run;
    for (int e = e0; e < min(E, e0 + per); ++e) {
      s_off[e] = exc;
      exc += min(s_tot[e], cap);
    }
    if (lane == 31 && bid == 0) {
      offsets[E] = exc;  // rows kept
      if (dropped) *dropped = A - exc;
    }
  }
  __syncthreads();
  int run[EPL];
#pragma unroll
  for (int j = 0; j < EPL; ++j)
    run[j] = on[j] ? s_off[ex[j]] + s_pre[ex[j]] + s_blk[warp][ex[j]] : 0;
  for (int tb = t0; tb < t1; tb += U * rpw) {
    int v[U][EPL];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int t = tb + u * rpw + r;
#pragma unroll
      for (int j = 0; j < EPL; ++j)
        v[u][j] = on[j] && t < t1 ? tile_counts[(size_t)t * E + ex[j]] : 0;
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int t = tb + u * rpw + r;
#pragma unroll
      for (int j = 0; j < EPL; ++j) {
        int incl = v[u][j], step = v[u][j];
        if constexpr (EPL == 1) {  // the step's rows before row r, and the step total
          for (int off = 1; off < rpw; off <<= 1) {
            const int nb2 = __shfl_up_sync(kFullMask, incl, off * E);
            if (r >= off) incl += nb2;
          }
          step = __shfl_sync(kFullMask, incl, (rpw - 1) * E + ex[0]);
        }
        if (on[j] && t < t1) tile_base[(size_t)t * E + ex[j]] = run[j] + incl - v[u][j];
        run[j] += step;
      }
    }
  }
  if (bid == 0)
    for (int e = threadIdx.x; e < E; e += kScanThreads) {
      counts[e] = s_tot[e];
      offsets[e] = s_off[e];
    }
}

// The in-CTA reduction reads tiles * E counts per CTA; above this many
// tiles^2 * E reads in total the separate scan is cheaper.
constexpr long long kFusedScanMaxReads = 4LL * 1024 * 1024;

__global__ void __launch_bounds__(kDispatchThreads)
    dispatch_scatter_kernel(const int32_t* __restrict__ idx, int A, int E, int k, int tile,
                            const int32_t* __restrict__ tile_counts,
                            const int32_t* __restrict__ tile_base, int tiles,
                            int32_t* __restrict__ perm, int32_t* __restrict__ inv_perm,
                            int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
                            const uint4* __restrict__ x, int vec_per_row, uint4* __restrict__ x_perm,
                            const float* __restrict__ aux_partials, int T, float* __restrict__ f,
                            float* __restrict__ p, float* __restrict__ loss,
                            float* __restrict__ f_frac, float* __restrict__ loss_frac,
                            float4* __restrict__ y_zero, int d4, int tokens_per_tile, int cap,
                            float* __restrict__ w_cap, int32_t* __restrict__ dropped,
                            const float* __restrict__ z_partials, float* __restrict__ z_loss,
                            int split) {
  pdl_begin();
  __shared__ int running[MOE_MAX_EXPERTS];
  __shared__ int s_tot[MOE_MAX_EXPERTS];
  __shared__ int s_seg[MOE_MAX_EXPERTS];  // segment start of each expert
  __shared__ int wcnt[kDispatchWarps][MOE_MAX_EXPERTS];
  __shared__ int s_row[kDispatchThreads];
  __shared__ int s_tok[kDispatchThreads];
  __shared__ float s_fp[MOE_MAX_EXPERTS];
  __shared__ int s_pre[kDispatchWarps][MOE_MAX_EXPERTS];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  // split CTAs share tile me: each derives the same ranks, part 0 writes perm,
  // inv_perm and the statistics, and the row copy and y's zeroing are shared out
  const int me = blockIdx.x / split, part = blockIdx.x % split;
  const bool fused_scan = tile_base == nullptr;
  for (int e = fused_scan ? E : threadIdx.x; e < E; e += blockDim.x) {
    running[e] = tile_base[(size_t)me * E + e];
    s_seg[e] = offsets[e];  // written by dispatch_scan_kernel
  }
  if (fused_scan && E < 32) {
    // each expert's total over all tiles and over the tiles before this one: a
    // warp per expert, lanes over tiles
    for (int e = warp; e < E; e += kDispatchWarps) {
      int tot = 0, pre = 0;
      for (int t = lane; t < tiles; t += 32) {
        const int c = tile_counts[(size_t)t * E + e];
        tot += c;
        pre += t < me ? c : 0;
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        tot += __shfl_xor_sync(kFullMask, tot, off);
        pre += __shfl_xor_sync(kFullMask, pre, off);
      }
      if (lane == 0) {
        s_tot[e] = tot;
        running[e] = pre;
      }
    }
  } else if (fused_scan) {
    // the same sums read row by row (a tile's E counts are contiguous, so a
    // warp's loads are whole lines): lanes over experts, E / 32 per lane, warps
    // over tiles; per-warp partials are added in shared memory (integers)
    int tot[MOE_MAX_EXPERTS / 32], pre[MOE_MAX_EXPERTS / 32];
#pragma unroll
    for (int j = 0; j < MOE_MAX_EXPERTS / 32; ++j) tot[j] = pre[j] = 0;
    for (int t = warp; t < tiles; t += kDispatchWarps) {
      const int32_t* row = tile_counts + (size_t)t * E;
#pragma unroll
      for (int j = 0; j < MOE_MAX_EXPERTS / 32; ++j) {
        const int e = lane + 32 * j;
        if (e < E) {
          const int c = row[e];
          tot[j] += c;
          pre[j] += t < me ? c : 0;
        }
      }
    }
#pragma unroll
    for (int j = 0; j < MOE_MAX_EXPERTS / 32; ++j) {
      const int e = lane + 32 * j;
      if (e < E) {
        wcnt[warp][e] = tot[j];
        s_pre[warp][e] = pre[j];
      }
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
      int tt = 0, pp = 0;
#pragma unroll
      for (int w = 0; w < kDispatchWarps; ++w) {
        tt += wcnt[w][e];
        pp += s_pre[w][e];
      }
      s_tot[e] = tt;
      running[e] = pp;
    }
    __syncthreads();  // the partials are read before wcnt is cleared below
  }
  for (int e = threadIdx.x; e < E; e += blockDim.x)
    for (int w = 0; w < kDispatchWarps; ++w) wcnt[w][e] = 0;
  __syncthreads();
  if (fused_scan && warp == 0) {  // exclusive scan of the (<= 256) totals, 8 per lane
    constexpr int per = MOE_MAX_EXPERTS / 32;
    const int e0 = lane * per;
    int run = 0;
    for (int e = e0; e < min(E, e0 + per); ++e) run += min(s_tot[e], cap);
    int incl = run;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int nb = __shfl_up_sync(kFullMask, incl, off);
      if (lane >= off) incl += nb;
    }
    int ex = incl - run;
    for (int e = e0; e < min(E, e0 + per); ++e) {
      const int v = s_tot[e];
      if (me == 0 && part == 0) {
        counts[e] = v;
        offsets[e] = ex;
      }
      s_seg[e] = ex;
      running[e] += ex;
      ex += min(v, cap);
    }
    if (me == 0 && part == 0 && lane == 31) {
      offsets[E] = ex;  // rows kept
      if (dropped) *dropped = A - ex;
    }
  }
  if (y_zero != nullptr) {
    const int tk0 = me * tokens_per_tile;
    const int tk1 = min(T, tk0 + tokens_per_tile);
    const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
    const size_t n = tk1 > tk0 ? (size_t)(tk1 - tk0) * d4 : 0;
    const size_t i0 = (size_t)tk0 * d4 + n * part / split, i1 = (size_t)tk0 * d4 + n * (part + 1) / split;
    for (size_t i = i0 + threadIdx.x; i < i1; i += blockDim.x) y_zero[i] = z;
  }
  __syncthreads();
  const int a0 = me * tile;
  const int a1 = min(A, a0 + tile);
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
      if (row - s_seg[e] < cap) {
        if (part == 0) {
          perm[row] = a;
          inv_perm[a] = row;
        }
        s_row[threadIdx.x] = row;
      } else {  // past the expert's capacity: dropped
        if (part == 0) inv_perm[a] = -1;
        s_row[threadIdx.x] = -1;
      }
      s_tok[threadIdx.x] = a / k;
    }
    __syncthreads();
    for (int ee = threadIdx.x; ee < E; ee += blockDim.x) {
      int sum = 0;
#pragma unroll
      for (int w = 0; w < kDispatchWarps; ++w) {
        sum += wcnt[w][ee];
        wcnt[w][ee] = 0;
      }
      running[ee] += sum;
    }
    if (x != nullptr) {  // copy this round's rows, one warp per row, rows shared out by part
      const int nvalid = min(kDispatchThreads, a1 - base);
      for (int i = warp + part * kDispatchWarps; i < nvalid; i += kDispatchWarps * split) {
        if (s_row[i] < 0) continue;  // dropped assignment: no row
        const uint4* src = x + (size_t)s_tok[i] * vec_per_row;
        uint4* dst = x_perm + (size_t)s_row[i] * vec_per_row;
        int v = lane;
        for (; v + 96 < vec_per_row; v += 128) {
          const uint4 q0 = __ldg(src + v), q1 = __ldg(src + v + 32), q2 = __ldg(src + v + 64),
                      q3 = __ldg(src + v + 96);
          dst[v] = q0;
          dst[v + 32] = q1;
          dst[v + 64] = q2;
          dst[v + 96] = q3;
        }
        for (; v < vec_per_row; v += 32) dst[v] = __ldg(src + v);
      }
    }
    __syncthreads();
  }
  if (w_cap != nullptr && part == 0) {  // renormalise the kept weights of this tile's tokens
    for (int t = a0 / k + threadIdx.x; t < (a1 + k - 1) / k; t += blockDim.x) {
      float sum = 0.f;
      for (int j = 0; j < k; ++j)
        if (inv_perm[(size_t)t * k + j] >= 0) sum += w_cap[(size_t)t * k + j];
      for (int j = 0; j < k; ++j) {
        const size_t a = (size_t)t * k + j;
        w_cap[a] = (inv_perm[a] >= 0 && sum > 0.f) ? w_cap[a] / sum : 0.f;
      }
    }
  }
  if (me != 0 || part != 0 || aux_partials == nullptr || !fused_scan) return;
  // CTA 0: aux statistics from the router's per-tile partial sums of g
  for (int e = threadIdx.x; e < MOE_MAX_EXPERTS; e += blockDim.x) s_fp[e] = 0.f;
  __syncthreads();
  if (E >= 32) {
    // column sums of the [tiles, E] partials read row by row: warp w sums rows
    // w, w + 8, ... of lanes' experts, the warps' sums then added in warp order
    // (a fixed order: deterministic)
    for (int j = 0; j * 32 < E; ++j) {
      const int e = lane + 32 * j;
      float acc = 0.f;
      if (e < E)
        for (int r = warp; r < tiles; r += kDispatchWarps) acc += aux_partials[(size_t)r * E + e];
      if (e < E) s_pre[warp][e] = __float_as_int(acc);
    }
    __syncthreads();
  }
  for (int e = warp; e < E; e += kDispatchWarps) {
    float acc = 0.f;
    if (E >= 32) {
      if (lane == 0)
        for (int w = 0; w < kDispatchWarps; ++w) acc += __int_as_float(s_pre[w][e]);
    } else {
      for (int r = lane; r < tiles; r += 32) acc += aux_partials[(size_t)r * E + e];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(kFullMask, acc, off);
    }
    if (lane == 0) {
      const float pe = acc / (float)T;
      const float fe = (float)s_tot[e] / (float)T;
      if (p) p[e] = pe;
      if (f) f[e] = fe;
      if (f_frac) f_frac[e] = (float)s_tot[e] / ((float)T * (float)k);
      s_fp[e] = fe * pe;
    }
  }
  __syncthreads();
  for (int off = MOE_MAX_EXPERTS / 2; off > 0; off >>= 1) {
    for (int e = threadIdx.x; e < off; e += blockDim.x) s_fp[e] += s_fp[e + off];
    __syncthreads();
  }
  if (threadIdx.x == 0 && loss) *loss = (float)E * s_fp[0];
  if (threadIdx.x == 0 && loss_frac) *loss_frac = (float)E * s_fp[0] / (float)k;
  if (warp == 0 && z_partials && z_loss) {  // router z-loss: fixed-order mean
    float acc = 0.f;
    for (int r = lane; r < tiles; r += 32) acc += z_partials[r];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(kFullMask, acc, off);
    if (lane == 0) *z_loss = acc / (float)T;
  }
}

// x_perm[r,:] = x[src[r] / div, :]; one warp per row, 16-byte vectors.
constexpr int kGatherThreads = 256;
__global__ void __launch_bounds__(kGatherThreads)
    gather_rows_kernel(const uint4* __restrict__ x, const int32_t* __restrict__ src, int R, int div,
                       int vec_per_row, uint4* __restrict__ out) {
  pdl_begin();
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
  pdl_begin();
  for (int e = threadIdx.x; e <= E; e += blockDim.x) offsets[e] = e * C;
}

}  // namespace moe
