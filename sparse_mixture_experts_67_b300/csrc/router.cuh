// Fused router: logits GEMM + softmax + top-k + renormalise + aux partial sums.
//
// Follows MoELayer.route of "Mixture of Experts（MoE）の理論と実装"
// (disassemble-channel.com) and TopKGating of "Sparse Mixture of Experts(MoE)
// 아키텍처 심층 분석" (youngju.dev): s = x W_g^T (+ b), g = softmax(s), the k
// largest entries, weights renormalised over the selection.
//
// One CTA owns TOK = 32 or 64 tokens (warps of 16), chosen by the expert count.  The logits GEMM is narrow (N = E
// <= 256), so bf16 runs on warp-level mma.sync m16n8k16 tiles fed by cp.async
// through a shared-memory ring, 8 warps per CTA splitting tokens and K (see
// router_bf16_kernel); fp32 runs on FFMA.  The 64 x E logits
// tile then goes through shared memory to a thread-per-token epilogue (no
// cross-lane reductions on the critical path): each thread reduces its own
// row for max and sum, and selects its top-k by repeated arg-max.  Outputs
// and the aux column sums are written cooperatively, in a fixed order.
#pragma once

#include <float.h>

#include "common.cuh"

namespace moe {

// Tokens per CTA (and per dispatch tile): 32 for small expert counts (more,
// shorter CTAs stream x faster), 64 from E > 16 on (W_g re-reads per token
// halve).  Threads per CTA: 2 * TOK (TOK / 16 warps of 16-token mma tiles).
constexpr int kRouterTokensMin = 32;
inline int router_tokens(int E) { return E <= 16 ? 32 : 64; }
constexpr int kRouterBK = 64;
constexpr int kRouterLd = kRouterBK + 8;  // bf16 elements per smem row (pad: conflict-free)

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem, bool valid) {
  uint32_t s = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
  int src_bytes = valid ? 16 : 0;
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(s), "l"(gmem), "r"(src_bytes));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N));
}

__device__ __forceinline__ void mma_bf16_16816(float* c, const uint32_t* a, const uint32_t* b) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// Epilogue over the logits tile S[TOK][ldS] (bias not yet added, when given;
// S is modified) with P adjacent threads per token (threads past TOK * P only
// join the cooperative loops): thread r * P + q owns the experts
// e = q, q + P, ... of token row r; row max,
// sum and the top-k arg-max are reduced over the P threads with shuffles (the
// top-k compares (logit desc, index asc), so ties still go to the lower
// index).  ldS = P (mod 32) keeps those reads free of bank conflicts.
// k == 0 writes logits only (expert-choice pre-pass).  The CTA's tokens form
// TOK / SUB dispatch tiles of SUB tokens, numbered from tile0: each gets its
// own row of aux partial sums (aux_rows, the row of tile0, nullable) and of
// per-expert selection counts (tile_counts, the dispatch histogram of its
// SUB*k assignments, nullable).
// Shared scratch: s_m / s_inv TOK floats each; s_cnt (TOK / SUB) *
// MOE_MAX_EXPERTS ints; s_part max(blockDim.x, E) floats.
// logitsT_out (nullable): the logits once more, transposed to [E, T] (row e is
// what the expert-choice selection of expert e reads).
// flags & MOE_ROUTE_NO_RENORM: the weights stay the selected probabilities.
// z_rows (nullable, k > 0): per dispatch tile, the sum over its tokens of
// (log sum_e exp s[t,e])^2 (the router z-loss before the mean), row of tile0.
template <int TOK, int SUB = TOK, int P = 1>
__device__ void router_epilogue(float* S, int ldS, int tok0, int T, int E, int k,
                                const float* __restrict__ bias, int32_t* __restrict__ idx_out,
                                float* __restrict__ w_out, float* __restrict__ logits_out,
                                float* __restrict__ probs_out, float* __restrict__ aux_rows,
                                int32_t* __restrict__ tile_counts, int tile0, float* s_m,
                                float* s_inv, int* s_cnt, float* s_part,
                                float* __restrict__ logitsT_out = nullptr, int flags = 0,
                                float* __restrict__ z_rows = nullptr) {
  static_assert(TOK % SUB == 0, "dispatch tiles split the CTA's tokens");
  static_assert(P >= 1 && P <= 32 && (P & (P - 1)) == 0, "threads per token: a power of two");
  constexpr int NSUB = TOK / SUB;
  const int tid = threadIdx.x, nthr = blockDim.x;
  const int ntok = min(TOK, T - tok0);
  const int nsub = (ntok + SUB - 1) / SUB;  // dispatch tiles holding tokens
  const int r = tid / P, q = tid % P;       // this thread's token row and expert phase
  const bool live = r < ntok;
  if (bias) {
    for (int i = tid; i < ntok * E; i += nthr) {
      const int ri = i / E, e = i - ri * E;
      S[ri * ldS + e] += bias[e];
    }
    __syncthreads();
  }
  if (k > 0) {
    const float* row = S + r * ldS;
    float m = -INFINITY;
    if (live)
      for (int e = q; e < E; e += P) m = fmaxf(m, row[e]);
#pragma unroll
    for (int o = 1; o < P; o <<= 1) m = fmaxf(m, __shfl_xor_sync(kFullMask, m, o));
    float sum = 0.f;
    if (live)
      for (int e = q; e < E; e += P) sum += expf(row[e] - m);
#pragma unroll
    for (int o = 1; o < P; o <<= 1) sum += __shfl_xor_sync(kFullMask, sum, o);
    if (live && q == 0) {
      s_m[r] = m;
      s_inv[r] = 1.0f / sum;
      if (z_rows) s_part[r] = m + logf(sum);  // log-sum-exp, read just below
    }
  }
  __syncthreads();
  if (k > 0 && z_rows) {  // per dispatch tile: sum of lse^2 in token order
    for (int st = tid; st < nsub; st += nthr) {
      float acc = 0.f;
      for (int ri = st * SUB; ri < min(ntok, st * SUB + SUB); ++ri) acc += s_part[ri] * s_part[ri];
      z_rows[st] = acc;
    }
    __syncthreads();  // s_part is reused by the aux sums
  }
  // coalesced optional outputs: element i of the CTA's [ntok, E] block
  if (logits_out || probs_out) {
    const size_t base = (size_t)tok0 * E;
    for (int i = tid; i < ntok * E; i += nthr) {
      const int ri = i / E, e = i - ri * E;
      const float v = S[ri * ldS + e];
      if (logits_out) logits_out[base + i] = v;
      if (probs_out) probs_out[base + i] = expf(v - s_m[ri]) * s_inv[ri];
    }
  }
  if (logitsT_out) {  // element i of the CTA's [E, ntok] block, tokens fastest
    for (int i = tid; i < ntok * E; i += nthr) {
      const int e = i / ntok, ri = i - e * ntok;
      logitsT_out[(size_t)e * T + tok0 + ri] = S[ri * ldS + e];
    }
  }
  if (k == 0) return;
  if (tile_counts)
    for (int i = tid; i < NSUB * MOE_MAX_EXPERTS; i += nthr) s_cnt[i] = 0;
  if (aux_rows) {
    // column sums of g over each dispatch tile's tokens: G row groups per
    // expert sum strided rows, then one thread per expert adds the G partials
    // in order
    const int G = max(1, nthr / E);
    for (int st = 0; st < nsub; ++st) {
      const int r0 = st * SUB, r1 = min(ntok, r0 + SUB);
      for (int c = tid; c < G * E; c += nthr) {
        const int e = c % E, gi = c / E;
        float acc = 0.f;
        for (int ri = r0 + gi; ri < r1; ri += G) acc += expf(S[ri * ldS + e] - s_m[ri]) * s_inv[ri];
        s_part[gi * E + e] = acc;
      }
      __syncthreads();
      for (int e = tid; e < E; e += nthr) {
        float acc = 0.f;
        for (int gi = 0; gi < G; ++gi) acc += s_part[gi * E + e];
        aux_rows[(size_t)st * E + e] = acc;
      }
      __syncthreads();
    }
  }
  __syncthreads();  // the top-k below overwrites selected entries of S
  {
    float* row = S + r * ldS;
    const float m = live ? s_m[r] : 0.f, inv = live ? s_inv[r] : 0.f;
    const int t = tok0 + r;
    float selsum = 0.f;
    for (int j = 0; j < k; ++j) {
      float best = -INFINITY;
      int bi = -1;
      if (live)
        for (int e = q; e < E; e += P) {  // ascending e + strict '>': lower index on ties
          const float v = row[e];
          if (bi < 0 ? v > -INFINITY : v > best) {
            best = v;
            bi = e;
          }
        }
#pragma unroll
      for (int o = 1; o < P; o <<= 1) {  // (larger logit, then lower index); none loses
        const float ob = __shfl_xor_sync(kFullMask, best, o);
        const int oi = __shfl_xor_sync(kFullMask, bi, o);
        if (oi >= 0 && (bi < 0 || ob > best || (ob == best && oi < bi))) {
          best = ob;
          bi = oi;
        }
      }
      if (bi < 0) {  // only for non-finite logits (NaN / -inf everywhere): stay in range
        bi = j;
        best = live ? row[bi] : 0.f;
      }
      if (live && bi % P == q) row[bi] = -INFINITY;  // taken; only this thread reads it again
      const float gsel = expf(best - m) * inv;  // same arithmetic as probs
      selsum += gsel;
      if (live && q == 0) {
        idx_out[(size_t)t * k + j] = bi;
        w_out[(size_t)t * k + j] = gsel;
        if (tile_counts) atomicAdd(&s_cnt[(r / SUB) * MOE_MAX_EXPERTS + bi], 1);
      }
    }
    if (live && q == 0 && !(flags & MOE_ROUTE_NO_RENORM)) {
      const float rs = 1.0f / selsum;
      for (int j = 0; j < k; ++j) w_out[(size_t)t * k + j] *= rs;
    }
  }
  if (tile_counts) {
    __syncthreads();
    for (int i = tid; i < nsub * E; i += nthr) {
      const int st = i / E, e = i - st * E;
      tile_counts[(size_t)(tile0 + st) * E + e] = s_cnt[st * MOE_MAX_EXPERTS + e];
    }
  }
}

// bf16 router CTA: 8 warps = TOK/16 token groups x K groups.  Each stage holds
// one 64-column chunk per K group; every warp runs its 16 tokens over its own
// chunk, and the K groups' partial logits are summed in a fixed order at the
// end (more warps per SM than one warp per token group: the small GEMM and
// the epilogue are latency-bound, not bandwidth-bound).
constexpr int kRouterWarps = 8;
constexpr int kRouterThreadsBf16 = 32 * kRouterWarps;

template <int NT, int TOK>
struct RouterBf16 {
  static constexpr int EP = 8 * NT;
  static constexpr int TG = TOK / 16;            // token groups
  static constexpr int KG = kRouterWarps / TG;   // K groups
  static constexpr int SBK = kRouterBK * KG;     // columns per stage
  static constexpr int LD = SBK + 8;             // bf16 row pitch (conflict-free fragments)
  static constexpr int STAGE_ELEMS = (TOK + EP) * LD;
  static constexpr size_t STAGE_BYTES = (size_t)STAGE_ELEMS * 2;
  // up to 8 stages within ~110 KB (two CTAs per SM); at least 3 while they fit
  // in 200 KB; 2 for the widest expert counts
  static constexpr size_t FIT2 = (110u * 1024u) / STAGE_BYTES;
  static constexpr size_t FIT1 = (200u * 1024u) / STAGE_BYTES;
  static constexpr int STAGES =
      FIT2 >= 3 ? (FIT2 > 8 ? 8 : (int)FIT2) : (FIT1 >= 3 ? 3 : (FIT1 < 2 ? 2 : (int)FIT1));
  static constexpr size_t RING = (size_t)STAGES * STAGE_BYTES;
  // epilogue threads per token: 4 from E > 16 on (TOK = 64; measured 44.8 -> 39.2 us at
  // T=16384, E=64), 1 below (TOK = 32; 4-8 threads per token measured slower at E=8)
  static constexpr int P = TOK == 64 ? 4 : 1;
  static constexpr int LDS = ((EP + 31) / 32) * 32 + P;  // = P (mod 32): conflict-free epilogue
  static constexpr size_t PART = (size_t)KG * TOK * LDS * 4;  // per-K-group partial logits
  static constexpr size_t TILE = (size_t)TOK * LDS * 4;
  static constexpr size_t MAIN = RING > PART + TILE ? RING : PART + TILE;
  static constexpr size_t SMEM = MAIN + 2 * TOK * 4 + MOE_MAX_EXPERTS * 4 + kRouterThreadsBf16 * 4;
  static_assert(SMEM <= 227 * 1024, "router shared memory");
};

template <int NT, int TOK>
constexpr size_t router_smem_bytes_bf16() {
  return RouterBf16<NT, TOK>::SMEM;
}

template <int NT, int TOK>
__global__ void __launch_bounds__(kRouterThreadsBf16)
    router_bf16_kernel(const __nv_bfloat16* __restrict__ x, const __nv_bfloat16* __restrict__ wg,
                       const float* __restrict__ bias, int T, int d, int E, int k,
                       int32_t* __restrict__ idx_out, float* __restrict__ w_out,
                       float* __restrict__ logits_out, float* __restrict__ probs_out,
                       float* __restrict__ aux_partials, int32_t* __restrict__ tile_counts,
                       float* __restrict__ logitsT, int flags, float* __restrict__ z_partials) {
  pdl_begin();
  using C = RouterBf16<NT, TOK>;
  constexpr int EP = C::EP, LD = C::LD, SBK = C::SBK, STAGES = C::STAGES;
  extern __shared__ __align__(16) unsigned char smem[];
  __nv_bfloat16* ring = reinterpret_cast<__nv_bfloat16*>(smem);
  float* s_m = reinterpret_cast<float*>(smem + C::MAIN);
  float* s_inv = s_m + TOK;
  int* s_cnt = reinterpret_cast<int*>(s_inv + TOK);
  float* s_part = reinterpret_cast<float*>(s_cnt + MOE_MAX_EXPERTS);

  const int tok0 = blockIdx.x * TOK;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tg = warp % C::TG, kg = warp / C::TG;
  const int nsc = (d + SBK - 1) / SBK;  // stages of SBK columns (the last may be partial)

  auto load_stage = [&](int stage, int sc) {
    __nv_bfloat16* xs = ring + stage * C::STAGE_ELEMS;
    __nv_bfloat16* ws = xs + TOK * LD;
    const int kof = sc * SBK;
    constexpr int CH = SBK / 8;  // 16-byte chunks per row
    for (int c = threadIdx.x; c < TOK * CH; c += kRouterThreadsBf16) {
      const int r = c / CH, ch = c % CH;
      const int t = tok0 + r, col = kof + ch * 8;
      const bool ok = t < T && col < d;
      const __nv_bfloat16* src = ok ? x + (size_t)t * d + col : x;
      cp_async16(xs + r * LD + ch * 8, src, ok);
    }
    for (int c = threadIdx.x; c < EP * CH; c += kRouterThreadsBf16) {
      const int r = c / CH, ch = c % CH;
      const int col = kof + ch * 8;
      const bool ok = r < E && col < d;
      const __nv_bfloat16* src = ok ? wg + (size_t)r * d + col : wg;
      cp_async16(ws + r * LD + ch * 8, src, ok);
    }
  };

  float acc[NT][4];
#pragma unroll
  for (int n = 0; n < NT; ++n)
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[n][i] = 0.f;

#pragma unroll
  for (int s = 0; s < STAGES - 1; ++s) {
    if (s < nsc) load_stage(s, s);
    cp_async_commit();
  }
  const int g = lane >> 2, c4 = lane & 3;
  for (int sc = 0; sc < nsc; ++sc) {
    cp_async_wait<STAGES - 2>();
    __syncthreads();
    {
      const int nxt = sc + STAGES - 1;
      if (nxt < nsc) load_stage(nxt % STAGES, nxt);
      cp_async_commit();
    }
    const __nv_bfloat16* xs = ring + (sc % STAGES) * C::STAGE_ELEMS;
    const __nv_bfloat16* ws = xs + TOK * LD + kg * kRouterBK;
    const __nv_bfloat16* xw = xs + tg * 16 * LD + kg * kRouterBK;
#pragma unroll
    for (int kk = 0; kk < kRouterBK; kk += 16) {
      uint32_t a[4];
      a[0] = *reinterpret_cast<const uint32_t*>(xw + g * LD + kk + 2 * c4);
      a[1] = *reinterpret_cast<const uint32_t*>(xw + (g + 8) * LD + kk + 2 * c4);
      a[2] = *reinterpret_cast<const uint32_t*>(xw + g * LD + kk + 8 + 2 * c4);
      a[3] = *reinterpret_cast<const uint32_t*>(xw + (g + 8) * LD + kk + 8 + 2 * c4);
#pragma unroll
      for (int n = 0; n < NT; ++n) {
        uint32_t b[2];
        const __nv_bfloat16* wr = ws + (n * 8 + g) * LD + kk + 2 * c4;
        b[0] = *reinterpret_cast<const uint32_t*>(wr);
        b[1] = *reinterpret_cast<const uint32_t*>(wr + 8);
        mma_bf16_16816(acc[n], a, b);
      }
    }
  }
  cp_async_wait<0>();
  __syncthreads();  // ring no longer read: the partial tiles may alias it

  constexpr int ldS = C::LDS;
  float* P = reinterpret_cast<float*>(smem);  // [KG][TOK][ldS]
  float* S = P + C::KG * TOK * ldS;           // [TOK][ldS]
  {
    float* Pk = P + kg * TOK * ldS;
#pragma unroll
    for (int n = 0; n < NT; ++n) {
      const int col = n * 8 + 2 * c4;
      const int r0 = tg * 16 + g;
      Pk[r0 * ldS + col] = acc[n][0];
      Pk[r0 * ldS + col + 1] = acc[n][1];
      Pk[(r0 + 8) * ldS + col] = acc[n][2];
      Pk[(r0 + 8) * ldS + col + 1] = acc[n][3];
    }
  }
  __syncthreads();
  for (int i = threadIdx.x; i < TOK * EP; i += kRouterThreadsBf16) {
    const int r = i / EP, e = i % EP;
    float v = P[r * ldS + e];
#pragma unroll
    for (int q = 1; q < C::KG; ++q) v += P[(q * TOK + r) * ldS + e];  // fixed K-group order
    S[r * ldS + e] = v;
  }
  __syncthreads();
  router_epilogue<TOK, TOK, C::P>(S, ldS, tok0, T, E, k, bias, idx_out, w_out, logits_out, probs_out,
                       aux_partials ? aux_partials + (size_t)blockIdx.x * E : nullptr, tile_counts,
                       blockIdx.x,
                       s_m, s_inv, s_cnt, s_part, logitsT, flags,
                       z_partials ? z_partials + blockIdx.x : nullptr);
}

// fp32 router: FFMA over 32-wide d chunks, same epilogue.
constexpr int kRouterBKf = 32;
template <int NT, int TOK>
constexpr size_t router_smem_bytes_f32() {
  constexpr size_t ld = kRouterBKf + 1;
  constexpr size_t tiles = (size_t)(TOK + 8 * NT) * ld * 4;
  constexpr size_t acc = (size_t)TOK * (((8 * NT + 31) / 32) * 32 + (TOK == 64 ? 2 : 1)) * 4;  // S
  // s_m, s_inv; s_cnt; s_part (max(threads, E) floats)
  return tiles + acc + 2 * TOK * 4 + MOE_MAX_EXPERTS * 4 +
         (2 * TOK > MOE_MAX_EXPERTS ? 2 * TOK : MOE_MAX_EXPERTS) * 4;
}

template <int NT, int TOK>
__global__ void __launch_bounds__(2 * TOK)
    router_f32_kernel(const float* __restrict__ x, const float* __restrict__ wg,
                      const float* __restrict__ bias, int T, int d, int E, int k,
                      int32_t* __restrict__ idx_out, float* __restrict__ w_out,
                      float* __restrict__ logits_out, float* __restrict__ probs_out,
                      float* __restrict__ aux_partials, int32_t* __restrict__ tile_counts,
                      float* __restrict__ logitsT, int flags, float* __restrict__ z_partials) {
  pdl_begin();
  constexpr int EP = 8 * NT;
  constexpr int ld = kRouterBKf + 1;
  constexpr int kPf = TOK == 64 ? 2 : 1;               // epilogue threads per token
  constexpr int ldS = ((EP + 31) / 32) * 32 + kPf;  // = kPf (mod 32)
  extern __shared__ __align__(16) unsigned char smem[];
  float* xs = reinterpret_cast<float*>(smem);
  constexpr int kThr = 2 * TOK;
  float* ws = xs + TOK * ld;
  float* S = ws + EP * ld;
  float* s_m = S + TOK * ldS;
  float* s_inv = s_m + TOK;
  int* s_cnt = reinterpret_cast<int*>(s_inv + TOK);
  float* s_part = reinterpret_cast<float*>(s_cnt + MOE_MAX_EXPERTS);
  const int tok0 = blockIdx.x * TOK;
  // thread -> (token, expert group): token = tid % TOK, experts eh + 2*i
  const int tt = threadIdx.x % TOK, eh = threadIdx.x / TOK;
  float acc[4 * NT];
#pragma unroll
  for (int i = 0; i < 4 * NT; ++i) acc[i] = 0.f;
  for (int kof = 0; kof < d; kof += kRouterBKf) {
    __syncthreads();
    for (int c = threadIdx.x; c < TOK * kRouterBKf; c += kThr) {
      const int r = c / kRouterBKf, cc = c % kRouterBKf;
      const int t = tok0 + r;
      xs[r * ld + cc] = (t < T && kof + cc < d) ? x[(size_t)t * d + kof + cc] : 0.f;
    }
    for (int c = threadIdx.x; c < EP * kRouterBKf; c += kThr) {
      const int r = c / kRouterBKf, cc = c % kRouterBKf;
      ws[r * ld + cc] = (r < E && kof + cc < d) ? wg[(size_t)r * d + kof + cc] : 0.f;
    }
    __syncthreads();
#pragma unroll 4
    for (int kk = 0; kk < kRouterBKf; ++kk) {
      const float xv = xs[tt * ld + kk];
#pragma unroll
      for (int i = 0; i < 4 * NT; ++i) acc[i] = fmaf(xv, ws[(eh + 2 * i) * ld + kk], acc[i]);
    }
  }
#pragma unroll
  for (int i = 0; i < 4 * NT; ++i) S[tt * ldS + eh + 2 * i] = acc[i];
  __syncthreads();
  router_epilogue<TOK, TOK, kPf>(S, ldS, tok0, T, E, k, bias, idx_out, w_out, logits_out, probs_out,
                       aux_partials ? aux_partials + (size_t)blockIdx.x * E : nullptr, tile_counts,
                       blockIdx.x,
                       s_m, s_inv, s_cnt, s_part, logitsT, flags,
                       z_partials ? z_partials + blockIdx.x : nullptr);
}

inline int router_nt(int E) {
  int ep = 8;
  while (ep < E) ep <<= 1;
  return ep / 8;
}

template <int NT, int TOK>
cudaError_t launch_router_nt(const void* x, const void* wg, const float* bias, int T, int d, int E,
                             int k, bool bf16, int32_t* idx, float* w, float* logits, float* probs,
                             float* aux, int32_t* tile_counts, float* logitsT, int flags,
                             float* z_partials, cudaStream_t st) {
  const int grid = ceil_div(T, TOK);
  if (bf16) {
    const size_t sm = router_smem_bytes_bf16<NT, TOK>();
    cudaError_t e = cudaFuncSetAttribute(router_bf16_kernel<NT, TOK>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
    if (e != cudaSuccess) return e;
    return launch_k(router_bf16_kernel<NT, TOK>, dim3(grid), dim3(kRouterThreadsBf16), sm, st,
                    nullptr, 0, static_cast<const __nv_bfloat16*>(x),
                    static_cast<const __nv_bfloat16*>(wg), bias, T, d, E, k, idx, w, logits, probs,
                    aux, tile_counts, logitsT, flags, z_partials);
  } else {
    const size_t sm = router_smem_bytes_f32<NT, TOK>();
    cudaError_t e = cudaFuncSetAttribute(router_f32_kernel<NT, TOK>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
    if (e != cudaSuccess) return e;
    return launch_k(router_f32_kernel<NT, TOK>, dim3(grid), dim3(2 * TOK), sm, st, nullptr, 0,
                    static_cast<const float*>(x), static_cast<const float*>(wg), bias, T, d, E, k,
                    idx, w, logits, probs, aux, tile_counts, logitsT, flags, z_partials);
  }
}

inline cudaError_t launch_router_mma(const void* x, const void* wg, const float* bias, int T, int d,
                                 int E, int k, bool bf16, int32_t* idx, float* w, float* logits,
                                 float* probs, float* aux, cudaStream_t st,
                                 int32_t* tile_counts = nullptr, float* logitsT = nullptr,
                                 int flags = 0, float* z_partials = nullptr) {
#define MOE_ROUTER_CASE(NT_)                                                                     \
  case NT_:                                                                                      \
    return router_tokens(E) == 32                                                                \
               ? launch_router_nt<NT_, 32>(x, wg, bias, T, d, E, k, bf16, idx, w, logits, probs, \
                                           aux, tile_counts, logitsT, flags, z_partials, st)                                 \
               : launch_router_nt<NT_, 64>(x, wg, bias, T, d, E, k, bf16, idx, w, logits, probs, \
                                           aux, tile_counts, logitsT, flags, z_partials, st);
  switch (router_nt(E)) {
    MOE_ROUTER_CASE(1)
    MOE_ROUTER_CASE(2)
    MOE_ROUTER_CASE(4)
    MOE_ROUTER_CASE(8)
    MOE_ROUTER_CASE(16)
    default:
      return launch_router_nt<32, 64>(x, wg, bias, T, d, E, k, bf16, idx, w, logits, probs, aux,
                                      tile_counts, logitsT, flags, z_partials, st);
  }
#undef MOE_ROUTER_CASE
}

}  // namespace moe
