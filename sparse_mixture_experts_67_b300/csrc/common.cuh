// Shared device helpers for the MoE kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdlib.h>

#include "../../include/moe.h"

namespace moe {

constexpr unsigned kFullMask = 0xffffffffu;

// Device error word: non-zero once a kernel gave up on a bounded barrier wait.
// Codes: bit 0 = producer wait timed out, bit 1 = MMA wait, bit 2 = epilogue
// wait, bit 3 = drain wait at exit, bit 4 = expert-choice slice wait.
__device__ uint32_t g_error_word;

__device__ __forceinline__ void record_error(uint32_t code) { atomicOr(&g_error_word, code); }

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Programmatic dependent launch.  Every kernel here calls pdl_begin() before
// its first global-memory access: it waits until the previous kernel in the
// stream has completed with its memory visible, then lets the next kernel be
// scheduled.  Launched with programmatic stream serialization (launch_k, when
// enabled), a kernel's CTAs thus start, and run their prologue (barrier setup,
// TMEM allocation), while the previous kernel drains its last CTAs; without
// the launch attribute both instructions are no-ops.
__device__ __forceinline__ void pdl_begin() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// The attribute is off unless MOE_PDL=1 is set in the environment.  Measured
// on top2_d1024: CUDA-graph replay of the layer 0.294 -> 0.300 ms with it (the
// graph already removes the launch gaps), eager launches 0.317 -> 0.313 ms.
inline bool pdl_enabled() {
  const char* v = getenv("MOE_PDL");
  return v && v[0] == '1';
}

// Launch with programmatic stream serialization (see pdl_begin) and optional
// extra attributes (a cluster shape).
template <typename... KArgs, typename... Args>
cudaError_t launch_k(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                     const cudaLaunchAttribute* extra, int n_extra, Args&&... args) {
  cudaLaunchAttribute attrs[4];
  int n = 0;
  for (int i = 0; i < n_extra && n < 3; ++i) attrs[n++] = extra[i];
  if (pdl_enabled()) {
    attrs[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attrs[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attrs;
  cfg.numAttrs = n;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <typename T>
struct Elem;
template <>
struct Elem<float> {
  static __device__ __forceinline__ float to_f32(float v) { return v; }
  static __device__ __forceinline__ float from_f32(float v) { return v; }
};
template <>
struct Elem<__nv_bfloat16> {
  static __device__ __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }
  static __device__ __forceinline__ __nv_bfloat16 from_f32(float v) { return __float2bfloat16_rn(v); }
};

// Unpack 8 bf16 held in a uint4 into fp32.
__device__ __forceinline__ void bf16x8_to_f32(const uint4& v, float* out) {
  const __nv_bfloat162* p = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float2 f = __bfloat1622float2(p[i]);
    out[2 * i] = f.x;
    out[2 * i + 1] = f.y;
  }
}

__device__ __forceinline__ float silu_f32(float a) { return a / (1.0f + expf(-a)); }

__device__ __forceinline__ unsigned lanemask_lt() {
  unsigned m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

inline int ceil_div(long long a, long long b) { return (int)((a + b - 1) / b); }

}  // namespace moe
