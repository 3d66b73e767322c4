// Tensor-core router for bf16 inputs (sm_103a): the logits GEMM of
// MoELayer.route in "Mixture of Experts（MoE）の理論と実装" and of TopKGating in
// "Sparse Mixture of Experts(MoE) 아키텍처 심층 분석", s = x W_g^T (+ b), on
// tcgen05 with the tokens as the MMA's M, followed by the same softmax,
// top-k, renormalisation and aux partial sums as the warp-MMA router.
//
// One CTA of 16 warps owns 128 tokens:
//   - one thread streams [128 x 64] x tiles and [EN x 64] W_g tiles (EN = E
//     rounded up to 16 .. 256; rows past E read as zero) with 2-D TMA into a
//     shared-memory ring;
//   - one thread issues tcgen05.mma kind::f16 (M = 128, N = EN, K = 16,
//     fp32 accumulate) into TMEM, freeing each stage by tcgen05.commit;
//   - the first 4 warps then read one token's row of logits each from TMEM
//     (TMEM lane = token), add the bias and store the rows to shared memory,
//     where the epilogue of the warp-MMA router runs with 4 threads per token
//     (E > 16) over all 16 warps.  The 128 tokens form 128 / SUB dispatch tiles (SUB =
//     32 or 64 tokens, the tile the dispatch histogram and the aux partial
//     rows are kept per).
// Every barrier wait is bounded; on expiry the kernel records an error code,
// drains its copies and MMAs, frees TMEM and returns without outputs.
#pragma once

#include "grouped_tc.cuh"
#include "router.cuh"

namespace moe {
namespace rtc {

constexpr int kTok = 128;      // tokens per CTA: the MMA's M
constexpr int kThreads = 512;  // 16 warps: warps 0-3 read TMEM (thread = token = lane)
constexpr int kBK = 64;        // K per stage: one 128-byte swizzled row per token

template <int EN>
struct Cfg {
  // epilogue threads per token: 4 (measured 34.8 -> 30.6 us at T=16384, E=64);
  // 1 for E <= 16, where wider groups measured slower
  static constexpr int P = EN > 16 ? kThreads / kTok : 1;
  static constexpr int A_BYTES = kTok * kBK * 2;  // 16 KiB
  static constexpr int B_BYTES = EN * kBK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int LDS = ((EN + 31) / 32) * 32 + P;  // logits tile pitch, = P (mod 32)
  static constexpr int S_BYTES = kTok * LDS * 4;
  // about 192 KiB of ring (one CTA per SM; measured 6% faster than 96 KiB at
  // E = 64); the logits tile reuses the ring once the MMAs are done
  static constexpr int ST0 = (192 * 1024) / STAGE_BYTES;
  static constexpr int STAGES = ST0 > 16 ? 16 : (ST0 < 2 ? 2 : ST0);
  static constexpr int RING0 = STAGES * STAGE_BYTES;
  static constexpr int RING = RING0 >= S_BYTES ? RING0 : ((S_BYTES + 1023) / 1024) * 1024;
  static constexpr uint32_t TMEM_COLS = EN < 32 ? 32 : EN;
};

struct RSmem {  // after the ring
  uint64_t full[16];
  uint64_t empty[16];
  uint64_t done;
  uint32_t tmem_base;
  int abort_flag;
  float s_m[kTok];
  float s_inv[kTok];
  int s_cnt[(kTok / kRouterTokensMin) * MOE_MAX_EXPERTS];
  float s_part[MOE_MAX_EXPERTS > kThreads ? MOE_MAX_EXPERTS : kThreads];
};

template <int EN>
constexpr size_t smem_bytes() {
  return (size_t)Cfg<EN>::RING + sizeof(RSmem) + 1024;
}

template <int EN, int SUB>
__global__ void __launch_bounds__(kThreads)
    router_tc_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                     const float* __restrict__ bias, int T, int d, int E, int k,
                     int32_t* __restrict__ idx_out, float* __restrict__ w_out,
                     float* __restrict__ logits_out, float* __restrict__ probs_out,
                     float* __restrict__ aux_partials, int32_t* __restrict__ tile_counts,
                     float* __restrict__ logitsT, int flags, float* __restrict__ z_partials) {
  using C = Cfg<EN>;
  using namespace tc;
  static_assert(C::STAGES <= 16, "barrier arrays");
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* ring = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  RSmem& S = *reinterpret_cast<RSmem*>(ring + C::RING);
  volatile int* abort_flag = &S.abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tok0 = blockIdx.x * kTok;
  const int nkb = d / kBK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&S.full[s], 1);
      mbar_init(&S.empty[s], 1);
    }
    mbar_init(&S.done, 1);
    S.abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    prefetch_tensormap(&tmX);
    prefetch_tensormap(&tmW);
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(&S.tmem_base)),
                 "r"(C::TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  pdl_begin();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = S.tmem_base;

  // Lanes 1-31 of warps 0 and 1 wait for their lane 0 at __syncwarp.
  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ producer
      int stage = 0;
      uint32_t phase = 0, issued = 0, issued_phase = 0;
      for (int kb = 0; kb < nkb; ++kb) {
        if (!mbar_wait(&S.empty[stage], phase ^ 1u, abort_flag, kErrProducer)) break;
        unsigned char* sA = ring + (size_t)stage * C::STAGE_BYTES;
        mbar_arrive_expect_tx(&S.full[stage], C::STAGE_BYTES);
        tma_load_2d(sA, &tmX, &S.full[stage], kb * kBK, tok0);
        tma_load_2d(sA + C::A_BYTES, &tmW, &S.full[stage], kb * kBK, 0);
        issued |= 1u << stage;
        issued_phase = (issued_phase & ~(1u << stage)) | (phase << stage);
        if (++stage == C::STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
      // every issued load lands before the ring is reused or the CTA exits
      for (int s = 0; s < C::STAGES; ++s) {
        if (!((issued >> s) & 1u)) continue;
        const uint32_t a = smem_u32(&S.full[s]);
        const uint64_t t0 = global_timer_ns();
        while (!mbar_try_wait(a, (issued_phase >> s) & 1u)) {
          if (global_timer_ns() - t0 > kWaitTimeoutNs) {
            record_error(kErrDrain);
            break;
          }
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------------------ MMA issuer
      constexpr uint32_t idesc = make_idesc_bf16(kTok, EN);
      int stage = 0;
      uint32_t phase = 0;
      for (int kb = 0; kb < nkb; ++kb) {
        if (!mbar_wait(&S.full[stage], phase, abort_flag, kErrMma)) break;
        tc_fence_after();
        const uint32_t a0 = smem_u32(ring + (size_t)stage * C::STAGE_BYTES);
        const uint32_t b0 = a0 + C::A_BYTES;
#pragma unroll
        for (int kk = 0; kk < kBK / 16; ++kk)
          tc_mma_f16(tmem, sw128_desc(a0 + kk * 32), sw128_desc(b0 + kk * 32), idesc,
                     (kb | kk) != 0 ? 1u : 0u);
        tc_commit(&S.empty[stage]);
        if (++stage == C::STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
      tc_commit(&S.done);  // arrives once every issued MMA has completed (also after an abort)
    }
    __syncwarp();
  }
  // ------------------------------------------------------------ logits out of TMEM
  mbar_wait(&S.done, 0, abort_flag, kErrEpilogue);
  __syncwarp();
  __syncthreads();  // loads landed and MMAs done: the ring may hold the logits tile
  const bool aborted = *abort_flag != 0;
  float* Sx = reinterpret_cast<float*>(ring);  // [kTok][LDS]
  if (!aborted && warp < 4) {
    tc_fence_after();
    const uint32_t trow = tmem + ((uint32_t)(warp * 32) << 16);
    float* row = Sx + threadIdx.x * C::LDS;
#pragma unroll 1
    for (int c = 0; c < EN; c += 32) {
      uint32_t v[32];
      MOE_TMEM_LD32(trow + c, v);
      tmem_ld_wait();
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const int e = c + i;
        if (e < E) row[e] = __uint_as_float(v[i]) + (bias ? bias[e] : 0.f);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(C::TMEM_COLS)
                 : "memory");
  }
  if (aborted) return;
  constexpr int kSubTiles = kTok / SUB;
  const int tile0 = blockIdx.x * kSubTiles;
  router_epilogue<kTok, SUB, C::P>(Sx, C::LDS, tok0, T, E, k, nullptr, idx_out, w_out, logits_out,
                             probs_out, aux_partials ? aux_partials + (size_t)tile0 * E : nullptr,
                             tile_counts, tile0, S.s_m, S.s_inv, S.s_cnt, S.s_part, logitsT,
                             flags, z_partials ? z_partials + tile0 : nullptr);
}

template <int EN, int SUB>
cudaError_t launch_en(const CUtensorMap& mx, const CUtensorMap& mw, const float* bias, int T, int d,
                      int E, int k, int32_t* idx, float* w, float* logits, float* probs, float* aux,
                      int32_t* tile_counts, float* logitsT, int flags, float* z_partials,
                      cudaStream_t st) {
  constexpr size_t sm = smem_bytes<EN>();
  static_assert(sm <= 227 * 1024, "router shared memory");
  auto kern = router_tc_kernel<EN, SUB>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
  if (e != cudaSuccess) return e;
  return launch_k(kern, dim3(ceil_div(T, kTok)), dim3(kThreads), sm, st, nullptr, 0, mx, mw, bias, T,
                  d, E, k, idx, w, logits, probs, aux, tile_counts, logitsT, flags, z_partials);
}

// Which bf16 router runs: the tensor-core one from E > 16 on (measured, events
// around the launch, L2 flushed: T=16384, d=2048, E=64 34.8 us against 44.8 us
// for the warp-MMA router), the warp-MMA one below (T=8192, d=1024, E=8:
// 12.4 us against 14.7 us; there the fixed launch, TMEM and epilogue costs of
// 64 CTAs of 128 tokens dominate).  MOE_ROUTER_TC=0 / 1 in the environment
// forces one (tests, A/B timing).
inline bool tc_router_enabled(int E) {
  const char* v = getenv("MOE_ROUTER_TC");
  if (v && v[0] == '0') return false;
  if (v && v[0] == '1') return true;
  return E > 16;
}

}  // namespace rtc

// Router launch for every entry point.  bf16 goes to the tensor-core router
// or the warp-MMA router (tc_router_enabled), fp32 to the FFMA router.  All
// keep the aux partial rows and the dispatch histogram per router_tokens(E)
// tokens.  Requires d % 64 == 0 for bf16 (checked by every caller).
// logitsT (nullable): an [E, T] transposed copy of the logits (expert choice).
// flags: MOE_ROUTE_NO_RENORM keeps the selected probabilities as the weights.
// z_partials (nullable): per dispatch tile, the sum of squared log-sum-exps.
inline cudaError_t launch_router(const void* x, const void* wg, const float* bias, int T, int d,
                                 int E, int k, bool bf16, int32_t* idx, float* w, float* logits,
                                 float* probs, float* aux, cudaStream_t st,
                                 int32_t* tile_counts = nullptr, float* logitsT = nullptr,
                                 int flags = 0, float* z_partials = nullptr) {
  if (!bf16 || !rtc::tc_router_enabled(E))
    return launch_router_mma(x, wg, bias, T, d, E, k, bf16, idx, w, logits, probs, aux, st,
                             tile_counts, logitsT, flags, z_partials);
  const int en = E <= 16 ? 16 : E <= 32 ? 32 : E <= 64 ? 64 : E <= 128 ? 128 : 256;
  CUtensorMap mx, mw;
  if (!tc::make_map(&mx, x, (uint64_t)T, (uint64_t)d, rtc::kTok) ||
      !tc::make_map(&mw, wg, (uint64_t)E, (uint64_t)d, (uint32_t)en))
    return cudaErrorInvalidValue;
  switch (en) {
    case 16:
      return rtc::launch_en<16, 32>(mx, mw, bias, T, d, E, k, idx, w, logits, probs, aux,
                                    tile_counts, logitsT, flags, z_partials, st);
    case 32:
      return rtc::launch_en<32, 64>(mx, mw, bias, T, d, E, k, idx, w, logits, probs, aux,
                                    tile_counts, logitsT, flags, z_partials, st);
    case 64:
      return rtc::launch_en<64, 64>(mx, mw, bias, T, d, E, k, idx, w, logits, probs, aux,
                                    tile_counts, logitsT, flags, z_partials, st);
    case 128:
      return rtc::launch_en<128, 64>(mx, mw, bias, T, d, E, k, idx, w, logits, probs, aux,
                                     tile_counts, logitsT, flags, z_partials, st);
    default:
      return rtc::launch_en<256, 64>(mx, mw, bias, T, d, E, k, idx, w, logits, probs, aux,
                                     tile_counts, logitsT, flags, z_partials, st);
  }
}

}  // namespace moe
