// Allocation-free variant of the dispatch (moe_permute_noalloc).
//
// Some callers cannot hand the library a workspace: plugin hosts that pass a
// kernel only its input and output buffers, and deployments whose device
// memory is reserved up front by another allocator, so that nothing may call
// cudaMalloc while they run.  This entry point keeps the dispatch scratch (the
// per-tile expert counts and their scanned bases) in a fixed array in the
// library's own device memory instead.
//
// The array is a file-scope __device__ variable, so every GPU that loads the
// library holds it until the process exits.  Host code cannot use the array's
// name as a device address; the first call on each device looks the address
// up with cudaGetSymbolAddress (that device current) and caches it.  All
// calls share the array and it keeps the last call's contents; the kernels
// write every entry they read, so nothing has to start at zero.  Calls whose
// work overlaps on the GPU (several streams, several threads) race on the
// array and must be serialised by the caller.
//
// Included by moe_api.cu (one translation unit with the kernels it reuses).

#include <mutex>

#include "common.cuh"
#include "dispatch.cuh"

namespace {

constexpr size_t kNoAllocScratchInts = MOE_PERMUTE_NOALLOC_SCRATCH_BYTES / sizeof(int32_t);
constexpr size_t kNoAllocHalf = kNoAllocScratchInts / 2;  // tile counts | tile bases
constexpr int kNoAllocMaxDevices = 64;

static __device__ __align__(256) int32_t g_permute_scratch[kNoAllocScratchInts];

std::mutex g_scratch_mu;
int32_t* g_scratch_ptr[kNoAllocMaxDevices] = {};

// Device address of g_permute_scratch on the current device (looked up once per device).
moe_status noalloc_scratch(int32_t** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  if (dev < 0 || dev >= kNoAllocMaxDevices) return MOE_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_permute_scratch) != cudaSuccess || p == nullptr)
      return MOE_ERR_CUDA;
    g_scratch_ptr[dev] = static_cast<int32_t*>(p);
  }
  *out = g_scratch_ptr[dev];
  return MOE_OK;
}

}  // namespace

extern "C" moe_status moe_permute_noalloc(const void* x, const int32_t* topk_idx, int T, int d, int E,
                                          int k, moe_dtype dt, void* x_perm, int32_t* counts,
                                          int32_t* offsets, int32_t* perm, int32_t* inv_perm,
                                          moe_stream_t stream) {
  using namespace moe;
  if (T < 0 || E < 1 || E > MOE_MAX_EXPERTS || k < 1 || k > E) return MOE_ERR_INVALID_ARG;
  if (dt != MOE_F32 && dt != MOE_BF16) return MOE_ERR_UNSUPPORTED;
  if (d <= 0) return MOE_ERR_INVALID_ARG;
  if ((dt == MOE_BF16 && d % 64 != 0) || (dt == MOE_F32 && d % 4 != 0)) return MOE_ERR_UNSUPPORTED;
  const long long A = (long long)T * k;
  if (A > INT32_MAX) return MOE_ERR_UNSUPPORTED;
  constexpr int kTile = 2048;  // assignments per dispatch tile
  const int tiles = dispatch_tiles(A, kTile);
  if ((size_t)tiles * (size_t)E > kNoAllocHalf) return MOE_ERR_WORKSPACE;  // beyond the fixed scratch
  if (!counts || !offsets) return MOE_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  if (T == 0) {
    cudaError_t e = cudaMemsetAsync(counts, 0, E * sizeof(int32_t), s);
    if (e == cudaSuccess) e = cudaMemsetAsync(offsets, 0, (E + 1) * sizeof(int32_t), s);
    return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
  }
  if (!x || !topk_idx || !x_perm || !perm || !inv_perm) return MOE_ERR_INVALID_ARG;
  int32_t* scratch = nullptr;
  moe_status st = noalloc_scratch(&scratch);
  if (st != MOE_OK) return st;
  int32_t* tile_counts = scratch;
  if (!aligned16(x) || !aligned16(x_perm)) return MOE_ERR_UNSUPPORTED;
  // second half of the array holds the tile bases when the separate scan runs
  int32_t* tile_base = scratch + kNoAllocHalf;
  return dispatch_launch(x, topk_idx, T, d, E, k, dt, x_perm, counts, offsets, perm, inv_perm,
                         tile_counts, tile_base, nullptr, kTile, false, s);  // one-CTA scan
}
