// Grouped expert GEMMs on FFMA: the exact-fp32 path.
//
// SwiGLU expert of "Mixture of Experts（MoE）の理論と実装" (Expert.forward) and
// SwiGLUExpert of "Sparse Mixture of Experts(MoE) 아키텍처 심층 분석":
// h = silu(x W_gate^T) * (x W_up^T), y = h W_down^T, applied per expert
// segment [offsets[e], offsets[e+1]) of the dispatched rows.
//
// 64x64 output tiles, 16-deep k-steps, 4x4 register micro-tiles.  The
// (expert, m-tile) of a CTA is found on the device from the offsets, so the
// host never reads the segment sizes.  fp32 keeps full single precision (the
// tensor cores would round to tf32); bf16 uses the tcgen05 kernels instead.
#pragma once

#include "common.cuh"

namespace moe {

constexpr int kSimtBM = 64, kSimtBN = 64, kSimtBK = 16, kSimtThreads = 256;

// Maps a linear m-tile id to (expert, first row, end row); false if past the end.
__device__ __forceinline__ bool find_segment_tile(const int32_t* __restrict__ offsets, int E,
                                                  int tile, int bm, int* e_out, int* row0,
                                                  int* row_end) {
  int cum = 0;
  for (int e = 0; e < E; ++e) {
    const int lo = offsets[e], hi = offsets[e + 1];
    const int tiles = (hi - lo + bm - 1) / bm;
    if (tile < cum + tiles) {
      *e_out = e;
      *row0 = lo + (tile - cum) * bm;
      *row_end = hi;
      return true;
    }
    cum += tiles;
  }
  return false;
}

template <typename TIn>
__device__ __forceinline__ void load4(const TIn* p, float* v, int valid);
template <>
__device__ __forceinline__ void load4<float>(const float* p, float* v, int valid) {
  if (valid == 4 && (reinterpret_cast<uintptr_t>(p) & 15) == 0) {
    const float4 q = *reinterpret_cast<const float4*>(p);
    v[0] = q.x; v[1] = q.y; v[2] = q.z; v[3] = q.w;
  } else {
#pragma unroll
    for (int i = 0; i < 4; ++i) v[i] = i < valid ? p[i] : 0.f;
  }
}
template <>
__device__ __forceinline__ void load4<__nv_bfloat16>(const __nv_bfloat16* p, float* v, int valid) {
#pragma unroll
  for (int i = 0; i < 4; ++i) v[i] = i < valid ? __bfloat162float(p[i]) : 0.f;
}

// GATEUP: out = TIn h [R,N] from two weight stacks; else out = float y [R,N].
template <typename TIn, bool GATEUP>
__global__ void __launch_bounds__(kSimtThreads)
    grouped_simt_kernel(const TIn* __restrict__ A, const int32_t* __restrict__ offsets,
                        const TIn* __restrict__ B0, const TIn* __restrict__ B1, int N, int K, int E,
                        void* __restrict__ out) {
  pdl_begin();
  __shared__ __align__(16) float As[kSimtBK][kSimtBM + 4];
  __shared__ __align__(16) float Bs0[kSimtBK][kSimtBN + 4];
  __shared__ __align__(16) float Bs1[GATEUP ? kSimtBK : 1][kSimtBN + 4];
  __shared__ int s_tile[3];
  if (threadIdx.x == 0) {
    int e, r0, r1;
    if (!find_segment_tile(offsets, E, blockIdx.x, kSimtBM, &e, &r0, &r1)) e = -1;
    s_tile[0] = e;
    s_tile[1] = r0;
    s_tile[2] = r1;
  }
  __syncthreads();
  const int e = s_tile[0];
  if (e < 0) return;
  const int row0 = s_tile[1], row_end = s_tile[2];
  const int n0 = blockIdx.y * kSimtBN;
  const TIn* b0 = B0 + (size_t)e * N * K;
  const TIn* b1 = GATEUP ? B1 + (size_t)e * N * K : nullptr;

  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const int lr = threadIdx.x >> 2, lk = (threadIdx.x & 3) * 4;
  float acc0[4][4], acc1[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc0[i][j] = acc1[i][j] = 0.f;

  for (int k0 = 0; k0 < K; k0 += kSimtBK) {
    const int kv = max(0, min(4, K - (k0 + lk)));
    float v[4];
    {
      const int r = row0 + lr;
      if (r < row_end) load4<TIn>(A + (size_t)r * K + k0 + lk, v, kv);
      else v[0] = v[1] = v[2] = v[3] = 0.f;
#pragma unroll
      for (int i = 0; i < 4; ++i) As[lk + i][lr] = v[i];
    }
    {
      const int n = n0 + lr;
      if (n < N) load4<TIn>(b0 + (size_t)n * K + k0 + lk, v, kv);
      else v[0] = v[1] = v[2] = v[3] = 0.f;
#pragma unroll
      for (int i = 0; i < 4; ++i) Bs0[lk + i][lr] = v[i];
      if (GATEUP) {
        if (n < N) load4<TIn>(b1 + (size_t)n * K + k0 + lk, v, kv);
        else v[0] = v[1] = v[2] = v[3] = 0.f;
#pragma unroll
        for (int i = 0; i < 4; ++i) Bs1[lk + i][lr] = v[i];
      }
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < kSimtBK; ++kk) {
      const float4 a = *reinterpret_cast<const float4*>(&As[kk][ty * 4]);
      const float4 b = *reinterpret_cast<const float4*>(&Bs0[kk][tx * 4]);
      const float av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc0[i][j] = fmaf(av[i], bv[j], acc0[i][j]);
      if (GATEUP) {
        const float4 c = *reinterpret_cast<const float4*>(&Bs1[kk][tx * 4]);
        const float cv[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int j = 0; j < 4; ++j) acc1[i][j] = fmaf(av[i], cv[j], acc1[i][j]);
      }
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = row0 + ty * 4 + i;
    if (r >= row_end) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int n = n0 + tx * 4 + j;
      if (n >= N) continue;
      if (GATEUP) {
        static_cast<TIn*>(out)[(size_t)r * N + n] = Elem<TIn>::from_f32(silu_f32(acc0[i][j]) * acc1[i][j]);
      } else {
        static_cast<float*>(out)[(size_t)r * N + n] = acc0[i][j];
      }
    }
  }
}

template <typename TIn, bool GATEUP>
cudaError_t launch_grouped_simt(const TIn* A, const int32_t* offsets, const TIn* B0, const TIn* B1,
                                int R, int N, int K, int E, void* out, cudaStream_t st) {
  dim3 grid(ceil_div(R, kSimtBM) + E, ceil_div(N, kSimtBN));
  return launch_k(grouped_simt_kernel<TIn, GATEUP>, grid, dim3(kSimtThreads), 0, st, nullptr, 0, A,
                  offsets, B0, B1, N, K, E, out);
}

}  // namespace moe
