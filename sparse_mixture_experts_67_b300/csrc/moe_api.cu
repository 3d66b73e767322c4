// C ABI of the MoE layer forward: argument checks, workspace carving and the
// launch sequence.  Every entry point only enqueues on the caller's stream.
#include <limits.h>
#include <math.h>
#include <string.h>

#include "combine.cuh"
#include "common.cuh"
#include "dispatch.cuh"
#include "ec_route.cuh"
#include "grouped_simt.cuh"
#include "grouped_tc.cuh"
#include "router.cuh"
#include "router_tc.cuh"

using namespace moe;

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }
bool valid_dtype(moe_dtype dt) { return dt == MOE_F32 || dt == MOE_BF16; }
size_t elt_size(moe_dtype dt) { return dt == MOE_BF16 ? 2 : 4; }

moe_status cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

// Shape rule shared by every call that reads rows of x / weights.
moe_status check_dims(int d, moe_dtype dt) {
  if (!valid_dtype(dt)) return MOE_ERR_UNSUPPORTED;
  if (d <= 0) return MOE_ERR_INVALID_ARG;
  if (dt == MOE_BF16 && d % 64 != 0) return MOE_ERR_UNSUPPORTED;
  if (dt == MOE_F32 && d % 4 != 0) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

// Top-k layers in bf16 with k <= 2 fuse the weighted combine into the down
// GEMM's epilogue (deterministic: at most two additions onto zero per element).
bool fused_combine(const moe_layer_desc& D) { return D.dtype == MOE_BF16 && D.k <= 2; }

struct Carver {
  char* base;
  size_t used = 0;
  template <typename T>
  T* take(size_t count) {
    T* p = base ? reinterpret_cast<T*>(base + used) : nullptr;
    used += align256(count * sizeof(T));
    return p;
  }
  void* take_bytes(size_t bytes) {
    void* p = base ? base + used : nullptr;
    used += align256(bytes);
    return p;
  }
};

}  // namespace

extern "C" {

const char* moe_status_string(moe_status s) {
  switch (s) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG";
    case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED";
    case MOE_ERR_WORKSPACE: return "MOE_ERR_WORKSPACE";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
  }
  return "MOE_ERR_UNKNOWN";
}

moe_status moe_device_error(uint32_t* word, int clear) {
  if (!word) return MOE_ERR_INVALID_ARG;
  cudaError_t e = cudaMemcpyFromSymbol(word, g_error_word, sizeof(uint32_t));
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  if (clear) {
    const uint32_t zero = 0;
    e = cudaMemcpyToSymbol(g_error_word, &zero, sizeof(uint32_t));
  }
  return cuda_status(e);
}

moe_status moe_selftest_wait_expiry(int T, int E, int C, int32_t* ec_idx, float* ec_score,
                                    int32_t* pos, void* ws, size_t ws_bytes, moe_stream_t stream) {
  if (T <= 0 || E < 1 || E > MOE_MAX_EXPERTS || C < 1 || C > T || !ec_idx || !ec_score || !pos)
    return MOE_ERR_INVALID_ARG;
  if (!ws || ws_bytes < ec_scratch_bytes(T, E, C) + 256) return MOE_ERR_WORKSPACE;
  char* scratch = static_cast<char*>(ws) + ((256 - (reinterpret_cast<uintptr_t>(ws) & 255)) & 255);
  const cudaError_t e = launch_ec_select(T, E, C, ec_idx, ec_score, pos, scratch,
                                         (cudaStream_t)stream, 0x80, true);
  if (e == cudaErrorNotSupported) {
    (void)cudaGetLastError();
    return MOE_ERR_UNSUPPORTED;
  }
  return cuda_status(e);
}

// Rows for the smallest router block (an upper bound for every E).
size_t moe_route_aux_rows(int T) { return T <= 0 ? 0 : (size_t)ceil_div(T, kRouterTokensMin); }

moe_status moe_route(const void* x, const void* w_g, const float* bias, int T, int d, int E, int k,
                     moe_dtype dt, int32_t* topk_idx, float* topk_w, float* logits, float* probs,
                     float* aux_partials, float* z_partials, int flags, moe_stream_t stream) {
  if (T < 0 || E < 1 || E > MOE_MAX_EXPERTS || k < 1 || k > E) return MOE_ERR_INVALID_ARG;
  if (flags & ~MOE_ROUTE_NO_RENORM) return MOE_ERR_INVALID_ARG;
  moe_status st = check_dims(d, dt);
  if (st != MOE_OK) return st;
  if (T == 0) return MOE_OK;
  if (!x || !w_g || !topk_idx || !topk_w) return MOE_ERR_INVALID_ARG;
  if (dt == MOE_BF16 && (!aligned16(x) || !aligned16(w_g))) return MOE_ERR_UNSUPPORTED;
  return cuda_status(launch_router(x, w_g, bias, T, d, E, k, dt == MOE_BF16, topk_idx, topk_w,
                                   logits, probs, aux_partials, (cudaStream_t)stream, nullptr,
                                   nullptr, flags, z_partials));
}

int moe_expert_choice_capacity(int T, int E, float capacity_factor) {
  if (T < 0 || E < 1 || !(capacity_factor > 0.f)) return -1;
  return (int)floor((double)T * (double)capacity_factor / (double)E);
}

size_t moe_expert_choice_workspace_size(int T, int E, float capacity_factor) {
  const int C = moe_expert_choice_capacity(T, E, capacity_factor);
  if (C < 0 || T <= 0 || E > MOE_MAX_EXPERTS) return 0;
  return ec_scratch_bytes(T, E, C) + 256;
}

moe_status moe_expert_choice_route(const void* x, const void* w_g, const float* bias, int T, int d,
                                   int E, float capacity_factor, moe_dtype dt, int32_t* ec_idx,
                                   float* ec_score, int32_t* pos, float* logits, void* ws,
                                   size_t ws_bytes, moe_stream_t stream) {
  if (T < 0 || E < 1 || E > MOE_MAX_EXPERTS || !(capacity_factor > 0.f)) return MOE_ERR_INVALID_ARG;
  moe_status st = check_dims(d, dt);
  if (st != MOE_OK) return st;
  const int C = moe_expert_choice_capacity(T, E, capacity_factor);
  if (C > T) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!x || !w_g || !pos || !logits || (C > 0 && (!ec_idx || !ec_score))) return MOE_ERR_INVALID_ARG;
  if (!ws || ws_bytes < moe_expert_choice_workspace_size(T, E, capacity_factor))
    return MOE_ERR_WORKSPACE;
  if (dt == MOE_BF16 && (!aligned16(x) || !aligned16(w_g))) return MOE_ERR_UNSUPPORTED;
  cudaStream_t s = (cudaStream_t)stream;
  // logits [T, E] for the caller, and transposed into pos for the selection
  cudaError_t e = launch_router(x, w_g, bias, T, d, E, /*k=*/0, dt == MOE_BF16, nullptr, nullptr,
                                logits, nullptr, nullptr, s, nullptr, reinterpret_cast<float*>(pos));
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  char* scratch = static_cast<char*>(ws) + ((256 - (reinterpret_cast<uintptr_t>(ws) & 255)) & 255);
  return cuda_status(launch_ec_select(T, E, C, ec_idx, ec_score, pos, scratch, s));
}

size_t moe_permute_workspace_size(int T, int E, int k) {
  if (T < 0 || E < 1 || k < 1) return 0;
  const int tiles = dispatch_tiles((long long)T * k, router_tokens(E) * k);
  // tile counts | tile bases | the scan's block sums [kScanBlocks, E]
  return 2 * align256((size_t)tiles * E * sizeof(int32_t)) +
         align256((size_t)kScanBlocks * E * sizeof(int32_t)) + 256;
}

moe_status moe_gather_rows(const void* x, const int32_t* src, int R, int div, int T, int d,
                           moe_dtype dt, void* x_perm, moe_stream_t stream) {
  if (R < 0 || div < 1 || T < 0) return MOE_ERR_INVALID_ARG;
  moe_status st = check_dims(d, dt);
  if (st != MOE_OK) return st;
  if (R == 0) return MOE_OK;
  if (!x || !src || !x_perm) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(x_perm)) return MOE_ERR_UNSUPPORTED;
  const int vec = (int)(d * elt_size(dt) / 16);
  const int grid = min(ceil_div(R, kGatherThreads / 32), 148 * 16);
  return cuda_status(launch_k(gather_rows_kernel, dim3(grid), dim3(kGatherThreads), 0,
                              (cudaStream_t)stream, nullptr, 0, static_cast<const uint4*>(x), src, R,
                              div, vec, static_cast<uint4*>(x_perm)));
}

// Dispatch: (histogram when the counts are not ready) + scatter with the row
// copy.  With counts_ready the per-tile counts are already in tile_counts
// (written by the router).  Tiles are `tile` consecutive assignments.  With
// aux_partials the scatter's CTA 0 also writes f, p and loss; with y_zero the
// scatter zeroes y for the fused down+combine.
static moe_status dispatch_launch(const void* x, const int32_t* topk_idx, int T, int d, int E, int k,
                                  moe_dtype dt, void* x_perm, int32_t* counts, int32_t* offsets,
                                  int32_t* perm, int32_t* inv_perm, int32_t* tile_counts,
                                  int32_t* tile_base, int32_t* scan_blk, int tile,
                                  bool counts_ready, cudaStream_t s,
                                  const float* aux_partials = nullptr, float* f = nullptr,
                                  float* p = nullptr, float* loss = nullptr,
                                  float* y_zero = nullptr, float* f_frac = nullptr,
                                  float* loss_frac = nullptr, int cap = INT_MAX,
                                  float* w_cap = nullptr, int32_t* dropped = nullptr,
                                  const float* z_partials = nullptr, float* z_loss = nullptr) {
  const long long A = (long long)T * k;
  const int tiles = dispatch_tiles(A, tile);
  cudaError_t e = cudaSuccess;
  if (!counts_ready)
    e = launch_k(dispatch_hist_kernel, dim3(tiles), dim3(kDispatchThreads), 0, s, nullptr, 0,
                 topk_idx, (int)A, E, tile, tile_counts);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  const bool separate_scan = (long long)tiles * tiles * E > kFusedScanMaxReads;
  if (separate_scan) {
    auto scan = E <= 32 ? dispatch_scan_kernel<1>
              : E <= 64 ? dispatch_scan_kernel<2>
              : E <= 128 ? dispatch_scan_kernel<4> : dispatch_scan_kernel<8>;
    // over all SMs when the block-sum scratch is given: the ranges' sums, then
    // the bases; else one CTA
    const int nb = scan_blk ? std::min(std::min(kScanBlocks, tc::sm_count()), tiles) : 1;
    if (nb > 1) {
      e = launch_k(scan, dim3(nb), dim3(kScanThreads), 0, s, nullptr, 0, tile_counts, tiles, E,
                   (int)A, tile_base, counts, offsets, cap, dropped, (int)kScanBlockSums, scan_blk);
      if (e == cudaSuccess)
        e = launch_k(scan, dim3(nb), dim3(kScanThreads), 0, s, nullptr, 0, tile_counts, tiles, E,
                     (int)A, tile_base, counts, offsets, cap, dropped, (int)kScanBases, scan_blk);
    } else {
      e = launch_k(scan, dim3(1), dim3(kScanThreads), 0, s, nullptr, 0, tile_counts, tiles, E,
                   (int)A, tile_base, counts, offsets, cap, dropped, (int)kScanWhole,
                   (int32_t*)nullptr);
    }
    if (e == cudaSuccess && aux_partials)
      e = launch_k(aux_finalize_kernel, dim3(1), dim3(kAuxThreads), 0, s, nullptr, 0, aux_partials,
                   tiles, counts, T, E, k, f, p, loss, f_frac, loss_frac, z_partials, z_loss);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
  }
  const int32_t* base = separate_scan ? tile_base : nullptr;
  // fewer tiles than two per SM: two CTAs share each tile's row copy (top2_d1024:
  // 256 tiles; measured faster than one CTA per tile)
  const int row_bytes = (int)(d * elt_size(dt));
  const int split = (x != nullptr && tiles < 2 * tc::sm_count()) ? 2 : 1;
  return cuda_status(launch_k(
      dispatch_scatter_kernel, dim3(tiles * split), dim3(kDispatchThreads), 0, s, nullptr, 0, topk_idx,
      (int)A, E, k, tile, tile_counts, base, tiles, perm, inv_perm, counts, offsets,
      static_cast<const uint4*>(x), row_bytes / 16, static_cast<uint4*>(x_perm),
      aux_partials, T, f, p, loss, f_frac, loss_frac, reinterpret_cast<float4*>(y_zero), d / 4,
      tile / k, cap, w_cap, dropped, z_partials, z_loss, split));
}

static moe_status check_permute(const void* x, const void* x_perm, int T, int d, int E, int k,
                                moe_dtype dt, const int32_t* counts, const int32_t* offsets) {
  if (T < 0 || E < 1 || E > MOE_MAX_EXPERTS || k < 1 || k > E) return MOE_ERR_INVALID_ARG;
  moe_status st = check_dims(d, dt);
  if (st != MOE_OK) return st;
  if (!counts || !offsets) return MOE_ERR_INVALID_ARG;
  if ((long long)T * k > INT32_MAX) return MOE_ERR_UNSUPPORTED;
  if (T > 0 && x && x_perm && (!aligned16(x) || !aligned16(x_perm))) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

moe_status moe_permute(const void* x, const int32_t* topk_idx, int T, int d, int E, int k,
                       moe_dtype dt, void* x_perm, int32_t* counts, int32_t* offsets, int32_t* perm,
                       int32_t* inv_perm, void* ws, size_t ws_bytes, moe_stream_t stream) {
  moe_status st = check_permute(x, x_perm, T, d, E, k, dt, counts, offsets);
  if (st != MOE_OK) return st;
  cudaStream_t s = (cudaStream_t)stream;
  if (T == 0) {  // empty: counts = 0, offsets = 0
    cudaError_t e = cudaMemsetAsync(counts, 0, E * sizeof(int32_t), s);
    if (e == cudaSuccess) e = cudaMemsetAsync(offsets, 0, (E + 1) * sizeof(int32_t), s);
    return cuda_status(e);
  }
  if (!x || !topk_idx || !x_perm || !perm || !inv_perm) return MOE_ERR_INVALID_ARG;
  if (!ws || ws_bytes < moe_permute_workspace_size(T, E, k)) return MOE_ERR_WORKSPACE;
  const int tile = router_tokens(E) * k;
  const int tiles = dispatch_tiles((long long)T * k, tile);
  Carver cv{static_cast<char*>(ws)};
  cv.used = (256 - (reinterpret_cast<uintptr_t>(ws) & 255)) & 255;
  int32_t* tile_counts = cv.take<int32_t>((size_t)tiles * E);
  int32_t* tile_base = cv.take<int32_t>((size_t)tiles * E);
  int32_t* scan_blk = cv.take<int32_t>((size_t)kScanBlocks * E);
  return dispatch_launch(x, topk_idx, T, d, E, k, dt, x_perm, counts, offsets, perm, inv_perm,
                         tile_counts, tile_base, scan_blk, tile, false, s);
}

static moe_status check_experts(int R, int d, int F, int E, moe_dtype dt) {
  if (R < 0 || E < 1 || E > MOE_MAX_EXPERTS || F <= 0) return MOE_ERR_INVALID_ARG;
  moe_status st = check_dims(d, dt);
  if (st != MOE_OK) return st;
  return check_dims(F, dt);
}

moe_status moe_grouped_gateup_swiglu(const void* x_perm, const int32_t* offsets, const void* w_gate,
                                     const void* w_up, int R, int d, int F, int E, moe_dtype dt,
                                     void* h, moe_stream_t stream) {
  moe_status st = check_experts(R, d, F, E, dt);
  if (st != MOE_OK) return st;
  if (R == 0) return MOE_OK;
  if (!x_perm || !offsets || !w_gate || !w_up || !h) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x_perm) || !aligned16(w_gate) || !aligned16(w_up) || !aligned16(h))
    return MOE_ERR_UNSUPPORTED;
  cudaStream_t s = (cudaStream_t)stream;
  if (dt == MOE_BF16)
    return cuda_status(launch_gateup_tc(static_cast<const __nv_bfloat16*>(x_perm), offsets,
                                        static_cast<const __nv_bfloat16*>(w_gate),
                                        static_cast<const __nv_bfloat16*>(w_up), R, d, F, E,
                                        static_cast<__nv_bfloat16*>(h), s));
  return cuda_status(launch_grouped_simt<float, true>(
      static_cast<const float*>(x_perm), offsets, static_cast<const float*>(w_gate),
      static_cast<const float*>(w_up), R, F, d, E, h, s));
}

moe_status moe_grouped_gateup_swiglu_gather(const void* x, const int32_t* src, int div, int T,
                                            const int32_t* offsets, const void* w_gate,
                                            const void* w_up, int R, int d, int F, int E,
                                            moe_dtype dt, void* h, moe_stream_t stream) {
  moe_status st = check_experts(R, d, F, E, dt);
  if (st != MOE_OK) return st;
  if (dt != MOE_BF16) return MOE_ERR_UNSUPPORTED;
  if (div < 1 || T < 1) return R == 0 ? MOE_OK : MOE_ERR_INVALID_ARG;
  if (R == 0) return MOE_OK;
  if (!x || !src || !offsets || !w_gate || !w_up || !h) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(w_gate) || !aligned16(w_up) || !aligned16(h))
    return MOE_ERR_UNSUPPORTED;
  return cuda_status(launch_gateup_gather_tc(
      static_cast<const __nv_bfloat16*>(x), T, src, div, offsets,
      static_cast<const __nv_bfloat16*>(w_gate), static_cast<const __nv_bfloat16*>(w_up), R, d, F, E,
      static_cast<__nv_bfloat16*>(h), (cudaStream_t)stream));
}

moe_status moe_grouped_down(const void* h, const int32_t* offsets, const void* w_down, int R, int d,
                            int F, int E, moe_dtype dt, float* y_perm, moe_stream_t stream) {
  moe_status st = check_experts(R, d, F, E, dt);
  if (st != MOE_OK) return st;
  if (R == 0) return MOE_OK;
  if (!h || !offsets || !w_down || !y_perm) return MOE_ERR_INVALID_ARG;
  if (!aligned16(h) || !aligned16(w_down) || !aligned16(y_perm)) return MOE_ERR_UNSUPPORTED;
  cudaStream_t s = (cudaStream_t)stream;
  if (dt == MOE_BF16)
    return cuda_status(launch_down_tc(static_cast<const __nv_bfloat16*>(h), offsets,
                                      static_cast<const __nv_bfloat16*>(w_down), R, d, F, E,
                                      y_perm, s));
  return cuda_status(launch_grouped_simt<float, false>(static_cast<const float*>(h), offsets,
                                                       static_cast<const float*>(w_down), nullptr,
                                                       R, d, F, E, y_perm, s));
}

moe_status moe_experts_swiglu(const void* x_perm, const int32_t* offsets, const void* w_gate,
                              const void* w_up, const void* w_down, int R, int d, int F, int E,
                              moe_dtype dt, void* h, float* y_perm, moe_stream_t stream) {
  // every argument of both stages is checked before the first one is enqueued
  moe_status st = check_experts(R, d, F, E, dt);
  if (st != MOE_OK || R == 0) return st;
  if (!x_perm || !offsets || !w_gate || !w_up || !w_down || !h || !y_perm)
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(x_perm) || !aligned16(w_gate) || !aligned16(w_up) || !aligned16(w_down) ||
      !aligned16(h) || !aligned16(y_perm))
    return MOE_ERR_UNSUPPORTED;
  st = moe_grouped_gateup_swiglu(x_perm, offsets, w_gate, w_up, R, d, F, E, dt, h, stream);
  if (st != MOE_OK) return st;
  return moe_grouped_down(h, offsets, w_down, R, d, F, E, dt, y_perm, stream);
}

moe_status moe_combine(const float* y_perm, const int32_t* inv_perm, const float* topk_w, int T,
                       int d, int k, float* y, moe_stream_t stream) {
  if (T < 0 || k < 1 || d <= 0) return MOE_ERR_INVALID_ARG;
  if (d % 4 != 0) return MOE_ERR_UNSUPPORTED;
  if (T == 0) return MOE_OK;
  if (!y_perm || !inv_perm || !topk_w || !y) return MOE_ERR_INVALID_ARG;
  if (!aligned16(y_perm) || !aligned16(y)) return MOE_ERR_UNSUPPORTED;
  const int grid = min(ceil_div(T, kCombineThreads / 32), 148 * 8);
  return cuda_status(launch_k(combine_kernel, dim3(grid), dim3(kCombineThreads), 0,
                              (cudaStream_t)stream, nullptr, 0,
                              reinterpret_cast<const float4*>(y_perm), inv_perm, topk_w, T, d / 4,
                              k, reinterpret_cast<float4*>(y)));
}

moe_status moe_ec_combine(const float* y_perm, const int32_t* pos, const float* ec_score, int T,
                          int d, int E, int C, float* y, moe_stream_t stream) {
  if (T < 0 || E < 1 || E > MOE_MAX_EXPERTS || C < 0 || C > T || d <= 0) return MOE_ERR_INVALID_ARG;
  if (d % 4 != 0) return MOE_ERR_UNSUPPORTED;
  if (T == 0) return MOE_OK;
  if (!pos || !y || (C > 0 && (!y_perm || !ec_score))) return MOE_ERR_INVALID_ARG;
  if ((y_perm && !aligned16(y_perm)) || !aligned16(y)) return MOE_ERR_UNSUPPORTED;
  const int grid = min(ceil_div(T, kCombineThreads / 32), 148 * 8);
  return cuda_status(launch_k(ec_combine_kernel, dim3(grid), dim3(kCombineThreads), 0,
                              (cudaStream_t)stream, nullptr, 0,
                              reinterpret_cast<const float4*>(y_perm), pos, ec_score, T, d / 4, E,
                              reinterpret_cast<float4*>(y)));
}

moe_status moe_aux_loss(const float* probs, const float* aux_partials, const int32_t* counts, int T,
                        int E, int k, float* f, float* p, float* loss, float* f_frac,
                        float* loss_frac, const float* z_partials, float* z_loss,
                        moe_stream_t stream) {
  if (T < 0 || E < 1 || E > MOE_MAX_EXPERTS || k < 1 || k > E) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!counts || (!probs && !aux_partials)) return MOE_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  const int tok = router_tokens(E);  // the router's block of tokens for this E
  const int rows = ceil_div(T, tok);
  if (probs) {
    // probs given: rebuild the per-block partial sums in place of the router's
    if (!aux_partials) return MOE_ERR_INVALID_ARG;
    cudaError_t e = launch_k(probs_partials_kernel, dim3(rows), dim3(256), 0, s, nullptr, 0, probs, T,
                             E, tok, const_cast<float*>(aux_partials));
    if (e != cudaSuccess) return MOE_ERR_CUDA;
  }
  return cuda_status(launch_k(aux_finalize_kernel, dim3(1), dim3(kAuxThreads), 0, s, nullptr, 0,
                              aux_partials, rows, counts, T, E, k, f, p, loss, f_frac, loss_frac,
                              z_partials, z_loss));
}

size_t moe_layer_workspace_size(const moe_layer_desc* desc) {
  if (!desc) return 0;
  const moe_layer_desc& D = *desc;
  if (D.T < 0 || D.E < 1 || D.E > MOE_MAX_EXPERTS || D.d <= 0 || D.F <= 0 || !valid_dtype(D.dtype))
    return 0;
  Carver cv{nullptr};
  const size_t es = elt_size(D.dtype);
  if (D.routing == MOE_ROUTING_EXPERT_CHOICE) {
    const int C = moe_expert_choice_capacity(D.T, D.E, D.capacity_factor);
    if (C < 0) return 0;
    const size_t R = (size_t)D.E * C;
    cv.take<float>((size_t)D.T * D.E);  // logits
    cv.take<int32_t>(R);                // ec_idx
    cv.take<float>(R);                  // ec_score
    cv.take<int32_t>((size_t)D.E * D.T);  // pos
    cv.take<int32_t>(D.E + 1);          // offsets
    cv.take_bytes(R * D.d * es);        // x_perm
    cv.take_bytes(R * D.F * es);        // h
    cv.take<float>(R * D.d);            // y_perm
    cv.take_bytes(moe_expert_choice_workspace_size(D.T, D.E, D.capacity_factor));  // select
  } else {
    if (D.k < 1 || D.k > D.E) return 0;
    const size_t A = (size_t)D.T * D.k;
    cv.take<int32_t>(A);                                   // topk_idx
    cv.take<float>(A);                                     // topk_w
    cv.take<float>(moe_route_aux_rows(D.T) * D.E);          // aux partials
    cv.take<int32_t>(D.E);                                 // counts
    cv.take<int32_t>(D.E + 1);                             // offsets
    cv.take<float>(2 * D.E + 1);                           // f, p, loss
    cv.take_bytes(moe_permute_workspace_size(D.T, D.E, D.k));
    cv.take<int32_t>(A);                                   // perm
    cv.take<int32_t>(A);                                   // inv_perm
    cv.take_bytes(A * D.d * es);                           // x_perm
    cv.take_bytes(A * D.F * es);                           // h
    cv.take<float>(moe_route_aux_rows(D.T));               // z-loss partials
    if (!fused_combine(D)) cv.take<float>(A * D.d);        // y_perm (separate combine only)
  }
  return cv.used + 256;
}

moe_status moe_layer_forward(const moe_layer_desc* desc, const moe_layer_weights* w, const void* x,
                             float* y, const moe_layer_outputs* out, void* ws, size_t ws_bytes,
                             moe_stream_t stream) {
  if (!desc || !w) return MOE_ERR_INVALID_ARG;
  const moe_layer_desc& D = *desc;
  const bool ec = D.routing == MOE_ROUTING_EXPERT_CHOICE;
  if (D.routing != MOE_ROUTING_TOPK && !ec) return MOE_ERR_INVALID_ARG;
  if (D.T < 0 || D.E < 1 || D.E > MOE_MAX_EXPERTS || D.F <= 0) return MOE_ERR_INVALID_ARG;
  if (!ec && (D.k < 1 || D.k > D.E)) return MOE_ERR_INVALID_ARG;
  if (D.flags & ~(MOE_ROUTE_NO_RENORM | MOE_ROUTE_CAPACITY)) return MOE_ERR_INVALID_ARG;
  const bool capacity = (D.flags & MOE_ROUTE_CAPACITY) != 0;
  if (capacity && (ec || (D.flags & MOE_ROUTE_NO_RENORM) || !(D.capacity_factor > 0.f)))
    return MOE_ERR_INVALID_ARG;
  if (ec && !(D.capacity_factor > 0.f)) return MOE_ERR_INVALID_ARG;
  moe_status st = check_experts(0, D.d, D.F, D.E, D.dtype);
  if (st != MOE_OK) return st;
  if (D.T == 0) return MOE_OK;
  if (!x || !y || !w->w_g || !w->w_gate || !w->w_up || !w->w_down) return MOE_ERR_INVALID_ARG;
  // alignment of every caller pointer a stage reads in 16-byte vectors or TMA
  // boxes, checked here so that an error never leaves earlier stages enqueued
  if (!aligned16(x) || !aligned16(y) || !aligned16(w->w_gate) || !aligned16(w->w_up) ||
      !aligned16(w->w_down) || (D.dtype == MOE_BF16 && !aligned16(w->w_g)))
    return MOE_ERR_UNSUPPORTED;
  const size_t need = moe_layer_workspace_size(desc);
  if (!ws || ws_bytes < need) return MOE_ERR_WORKSPACE;
  moe_layer_outputs none;
  memset(&none, 0, sizeof(none));
  const moe_layer_outputs& O = out ? *out : none;
  Carver cv{static_cast<char*>(ws)};
  cv.used = (256 - (reinterpret_cast<uintptr_t>(ws) & 255)) & 255;
  const size_t es = elt_size(D.dtype);
  cudaStream_t s = (cudaStream_t)stream;

  if (ec) {
    const int C = moe_expert_choice_capacity(D.T, D.E, D.capacity_factor);
    const size_t R = (size_t)D.E * C;
    float* logits = cv.take<float>((size_t)D.T * D.E);
    int32_t* ec_idx = cv.take<int32_t>(R);
    float* ec_score = cv.take<float>(R);
    int32_t* pos = cv.take<int32_t>((size_t)D.E * D.T);
    int32_t* offsets = cv.take<int32_t>(D.E + 1);
    void* x_perm = cv.take_bytes(R * D.d * es);
    void* h = cv.take_bytes(R * D.F * es);
    float* y_perm = cv.take<float>(R * D.d);
    const size_t sel_bytes = moe_expert_choice_workspace_size(D.T, D.E, D.capacity_factor);
    void* sel_ws = cv.take_bytes(sel_bytes);
    if (O.logits) logits = O.logits;
    if (O.ec_idx) ec_idx = O.ec_idx;
    if (O.ec_score) ec_score = O.ec_score;
    if (O.pos) pos = O.pos;
    st = moe_expert_choice_route(x, w->w_g, w->bias, D.T, D.d, D.E, D.capacity_factor, D.dtype,
                                 ec_idx, ec_score, pos, logits, sel_ws, sel_bytes, stream);
    if (st != MOE_OK) return st;
    if (R > 0) {
      // expert e owns dispatch rows [e*C, (e+1)*C)
      if (launch_k(uniform_offsets_kernel, dim3(1), dim3(MOE_MAX_EXPERTS + 1), 0, s, nullptr, 0,
                   offsets, D.E, C) != cudaSuccess)
        return MOE_ERR_CUDA;
      st = moe_gather_rows(x, ec_idx, (int)R, 1, D.T, D.d, D.dtype, x_perm, stream);
      if (st != MOE_OK) return st;
      st = moe_experts_swiglu(x_perm, offsets, w->w_gate, w->w_up, w->w_down, (int)R, D.d, D.F,
                              D.E, D.dtype, h, y_perm, stream);
      if (st != MOE_OK) return st;
    }
    return moe_ec_combine(y_perm, pos, ec_score, D.T, D.d, D.E, C, y, stream);
  }

  const int k = D.k;
  const size_t A = (size_t)D.T * k;
  int32_t* idx = cv.take<int32_t>(A);
  float* tw = cv.take<float>(A);
  float* aux = cv.take<float>(moe_route_aux_rows(D.T) * D.E);
  int32_t* counts = cv.take<int32_t>(D.E);
  int32_t* offsets = cv.take<int32_t>(D.E + 1);
  float* fpl = cv.take<float>(2 * D.E + 1);
  const size_t pws = moe_permute_workspace_size(D.T, D.E, k);
  void* pw = cv.take_bytes(pws);
  int32_t* perm = cv.take<int32_t>(A);
  int32_t* inv_perm = cv.take<int32_t>(A);
  void* x_perm = cv.take_bytes(A * D.d * es);
  void* h = cv.take_bytes(A * D.F * es);
  float* zpart = cv.take<float>(moe_route_aux_rows(D.T));
  // k <= 2 (bf16): the down GEMM accumulates the combine into y, zeroed by the
  // scatter, and no [R, d] y_perm exists
  const bool fused = fused_combine(D);
  float* y_perm = fused ? nullptr : cv.take<float>(A * D.d);
  if (O.topk_idx) idx = O.topk_idx;
  if (O.topk_w) tw = O.topk_w;
  if (O.counts) counts = O.counts;
  if (O.offsets) offsets = O.offsets;
  st = check_permute(x, x_perm, D.T, D.d, D.E, k, D.dtype, counts, offsets);
  if (st != MOE_OK) return st;
  // router CTAs double as dispatch tiles: the router writes the per-tile counts
  const int tile = router_tokens(D.E) * k;
  const int tiles = dispatch_tiles((long long)A, tile);
  int32_t* tile_counts = static_cast<int32_t*>(pw);
  int32_t* tile_base = reinterpret_cast<int32_t*>(static_cast<char*>(pw) +
                                                  align256((size_t)tiles * D.E * sizeof(int32_t)));
  int32_t* scan_blk = reinterpret_cast<int32_t*>(static_cast<char*>(pw) +
                                                 2 * align256((size_t)tiles * D.E * sizeof(int32_t)));
  if (launch_router(x, w->w_g, w->bias, D.T, D.d, D.E, k, D.dtype == MOE_BF16, idx, tw, O.logits,
                    nullptr, aux, s, tile_counts, nullptr, D.flags,
                    O.z_loss ? zpart : nullptr) != cudaSuccess)
    return MOE_ERR_CUDA;
  // the scatter also copies the x rows into dispatch order: contiguous row blocks
  // keep the gate/up operand loads full-width TMA boxes (gathering rows inside
  // the GEMM re-fetches them once per n-block and measured several times slower)
  // capacity-limited token choice: each expert keeps its first `cap` assignments
  // in token order, cap = int(T / E * capacity_factor * k) (double, this order)
  int cap = INT_MAX;
  if (capacity) {
    const double capd =
        floor((double)D.T / (double)D.E * (double)D.capacity_factor * (double)k);
    cap = capd >= (double)A ? (int)A : (int)capd;
  }
  st = dispatch_launch(x, idx, D.T, D.d, D.E, k, D.dtype, x_perm, counts, offsets, perm, inv_perm,
                       tile_counts, tile_base, scan_blk, tile, true, s, aux, O.f ? O.f : fpl,
                       O.p ? O.p : fpl + D.E, O.loss ? O.loss : fpl + 2 * D.E,
                       fused ? y : nullptr, O.f_frac, O.loss_frac, cap,
                       capacity ? tw : nullptr, O.dropped, O.z_loss ? zpart : nullptr, O.z_loss);
  if (st != MOE_OK) return st;
  if (fused) {
    // down projection with the combine in its epilogue (deterministic for k <= 2)
    st = moe_grouped_gateup_swiglu(x_perm, offsets, w->w_gate, w->w_up, (int)A, D.d, D.F, D.E,
                                   D.dtype, h, stream);
    if (st != MOE_OK) return st;
    return cuda_status(launch_down_combine_tc(static_cast<const __nv_bfloat16*>(h), offsets,
                                              static_cast<const __nv_bfloat16*>(w->w_down), (int)A,
                                              D.d, D.F, D.E, perm, tw, k, y, s));
  }
  st = moe_experts_swiglu(x_perm, offsets, w->w_gate, w->w_up, w->w_down, (int)A, D.d, D.F, D.E,
                          D.dtype, h, y_perm, stream);
  if (st != MOE_OK) return st;
  return moe_combine(y_perm, inv_perm, tw, D.T, D.d, k, y, stream);
}

}  // extern "C"

// Allocation-free dispatch variant (static device scratch).
#include "permute_noalloc.cu"
