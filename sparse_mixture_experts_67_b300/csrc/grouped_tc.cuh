// Grouped bf16 expert GEMMs (placeholder: FFMA tiles until the tensor-core
// kernels land).
#pragma once

#include "grouped_simt.cuh"

namespace moe {

inline cudaError_t launch_gateup_tc(const __nv_bfloat16* x_perm, const int32_t* offsets,
                                    const __nv_bfloat16* w_gate, const __nv_bfloat16* w_up, int R,
                                    int d, int F, int E, __nv_bfloat16* h, cudaStream_t s) {
  return launch_grouped_simt<__nv_bfloat16, true>(x_perm, offsets, w_gate, w_up, R, F, d, E, h, s);
}

inline cudaError_t launch_down_tc(const __nv_bfloat16* h, const int32_t* offsets,
                                  const __nv_bfloat16* w_down, int R, int d, int F, int E,
                                  float* y_perm, cudaStream_t s) {
  return launch_grouped_simt<__nv_bfloat16, false>(h, offsets, w_down, nullptr, R, d, F, E, y_perm, s);
}

}  // namespace moe
