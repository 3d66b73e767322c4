// Tensor-core router for bf16 inputs (sm_103a): the logits GEMM of
// MoELayer.route in "Mixture of Experts（MoE）の理論と実装" and of TopKGating in
// "Sparse Mixture of Experts(MoE) 아키텍처 심층 분석", s = x W_g^T (+ b), on
// tcgen05 with the tokens as the MMA's M, then the softmax, the top-k with
// lower-index ties, the renormalisation and the per-dispatch-tile statistics
// (expert counts, column sums of g, sums of squared log-sum-exps).
//
// Persistent, one CTA per SM, each owning a contiguous range of dispatch tiles
// (SUB = 32 or 64 tokens; the ranges of all SMs differ by one tile at most)
// and taking them in MMA tiles of up to 128 tokens:
//   warp 0     one thread streams, per 64-column k-block, the tile's x rows
//              (one TMA box; a CTA's shorter last tile one box per dispatch
//              tile) and the W_g k-block ([NM x 64],
//              rows past E zero-filled) into a ring of about 180 KiB; the whole
//              range is requested as fast as the ring frees, so HBM sees every
//              CTA's reads from the start;
//   warp 1     allocates TMEM; one thread issues tcgen05.mma kind::f16
//              (M = 128, N = NM, K = 16) into one of two accumulators;
//   warps 2-9  epilogue, thread = token (TMEM lane): reads its logits row
//              straight from TMEM, reduces max and sum of exponentials,
//              selects the top-k by repeated arg-max on (logit desc, index
//              asc), and reduces the statistics of its 32 tokens with warp
//              butterflies.
// The epilogue has two forms.  Up to 16 experts (EN = 8 or 16 columns read,
// the MMA N at least 16) one warp holds a token's whole row: warps 2-5 take
// the tiles of accumulator 0 and warps 6-9 those of accumulator 1, one warp per
// TMEM lane quarter, and no warp exchanges anything with another.  From 32
// experts on, two warps share each lane quarter, each holding half of every
// row, and exchange partial maxima, sums and top-k candidates through shared
// memory; for SUB = 64 two quarters' statistics are added in a fixed order.
// With two accumulators the epilogue of one MMA tile overlaps the loads and
// MMAs of the next.  Rows of a partial MMA tile beyond its tokens hold stale
// shared memory; the MMA rows are independent, so only those TMEM lanes carry
// garbage and no thread reads them.
// Every barrier wait is bounded; on expiry the kernel records an error code,
// drains its copies and MMAs, frees TMEM and returns.
#pragma once

#include "grouped_tc.cuh"
#include "router.cuh"

namespace moe {
namespace rtc {

constexpr int kMmaTok = 128;   // tokens per MMA tile at most: the MMA's M
constexpr int kThreads = 320;  // 10 warps: producer, MMA, 8 epilogue warps
constexpr int kEpiThreads = 256;
constexpr int kBK = 64;        // K per stage: one 128-byte swizzled row per token

#define MOE_TMEM_LD8(taddr, r)                                                                    \
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"            \
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),         \
                 "=r"(r[6]), "=r"(r[7])                                                           \
               : "r"(taddr))

#define MOE_TMEM_LD16(taddr, r)                                                                   \
  asm volatile(                                                                                   \
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14," \
      "%15}, [%16];"                                                                              \
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),       \
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),   \
        "=r"(r[14]), "=r"(r[15])                                                                  \
      : "r"(taddr))

// The ring is cut at run time into stages of [a_rows x 64] x plus [NM x 64] W_g
// (1 KiB-aligned), a_rows the most tokens any CTA's MMA tile holds, so that a
// launch of small tiles keeps as many x bytes in flight as one of full tiles.
// The MMA still reads 128 rows of A from a stage's start; rows past the tile's
// tokens lie in the next stage or, for the last one, in the pad after the
// ring, and only reach TMEM lanes no thread reads.
constexpr int kRingBytes = 180 * 1024;
constexpr int kRingPad = kMmaTok * kBK * 2;  // 16 KiB
constexpr int kMaxStages = 32;

// EN: logit columns the epilogue reads (8, 16, ... 256); NM: the MMA's N
// (the smallest legal N for M = 128 is 16); SOLO: the one-warp-per-row epilogue.
template <int EN>
struct Cfg {
  static constexpr int NM = EN < 16 ? 16 : EN;
  static constexpr bool SOLO = EN <= 16;
  static constexpr int B_BYTES = NM * kBK * 2;
  static constexpr uint32_t TMEM_COLS = 2 * NM < 32 ? 32 : 2 * NM;  // two accumulators
};

__host__ __device__ constexpr int stage_bytes_for(int a_rows, int b_bytes) {
  return ((a_rows * kBK * 2 + b_bytes) + 1023) / 1024 * 1024;
}
__host__ __device__ constexpr int stages_for(int stage_bytes) {
  return kRingBytes / stage_bytes > kMaxStages ? kMaxStages : kRingBytes / stage_bytes;
}

struct RSmem {  // after the ring and its pad
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  uint64_t tmem_full[2];
  uint64_t tmem_empty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
  float bias[MOE_MAX_EXPERTS];
  int cnt[4][MOE_MAX_EXPERTS];    // per lane quarter: expert counts of its 32 tokens
  int cnt16[8][16];               // one-warp rows (E <= 16): per epilogue warp
  float gsum[4][MOE_MAX_EXPERTS]; // per lane quarter: column sums of g (SUB = 64 pairs)
  float zsum[4];
  float xf[2][2][kMmaTok];        // pair exchange of floats: [parity][half][row]
  int xi[2][2][kMmaTok];          // pair exchange of indices
};

// Exchange between the two warps of a lane quarter: half h posts (v, i) for
// tile row r and reads the other half's after the quarter's barrier.  The
// buffer alternates with the exchange count xc (kept across tiles), so each
// exchange needs one barrier: a thread writes a buffer again only after the
// barrier that follows its partner's read of it.
__device__ __forceinline__ void pair_xchg(RSmem& S, float v, int i, float& ov, int& oi, int h, int q,
                                          int r, int& xc) {
  const int p = xc & 1;
  ++xc;
  S.xf[p][h][r] = v;
  S.xi[p][h][r] = i;
  asm volatile("bar.sync %0, 64;" ::"r"(2 + q) : "memory");
  ov = S.xf[p][h ^ 1][r];
  oi = S.xi[p][h ^ 1][r];
}

template <int EN>
constexpr size_t smem_bytes() {
  return (size_t)kRingBytes + kRingPad + sizeof(RSmem) + 1024;
}

// One chunk of a thread's logits row from TMEM: CH fp32 columns from taddr.
template <int CH>
__device__ __forceinline__ void tmem_chunk(uint32_t taddr, uint32_t (&v)[CH]) {
  static_assert(CH == 8 || CH == 16 || CH == 32, "chunk width");
  if constexpr (CH == 8) {
    MOE_TMEM_LD8(taddr, v);
  } else if constexpr (CH == 16) {
    MOE_TMEM_LD16(taddr, v);
  } else {
    MOE_TMEM_LD32(taddr, v);
  }
  tc::tmem_ld_wait();
}

// Sum over the 32 lanes of each of the N values v[0..N-1] (N = 8, 16 or 32):
// a transpose within aligned groups of N lanes, then a butterfly across the
// groups.  On return lane l holds, in v[0], the sum over all lanes of
// v[l % N]; the order of the additions is fixed and every lane holding the
// same column gets the same value.
template <int N>
__device__ __forceinline__ float warp_transpose_sum(float (&v)[N]) {
  static_assert(N == 8 || N == 16 || N == 32, "row width");
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int s = N / 2; s >= 1; s >>= 1) {
    const bool hi = (lane & s) != 0;
#pragma unroll
    for (int i = 0; i < s; ++i) {
      const float send = hi ? v[i] : v[i + s];
      const float recv = __shfl_xor_sync(kFullMask, send, s);
      v[i] = (hi ? v[i + s] : v[i]) + recv;
    }
  }
#pragma unroll
  for (int o = N; o < 32; o <<= 1) v[0] += __shfl_xor_sync(kFullMask, v[0], o);
  return v[0];
}

// Pairwise trees over a row held in registers (N a power of two): depth
// log2 N instead of a chain of N dependent steps.  The order of the additions
// is fixed, so the sum is deterministic.
template <int N>
__device__ __forceinline__ float tree_max(const float (&v)[N]) {
  float t[N];
#pragma unroll
  for (int i = 0; i < N; ++i) t[i] = v[i];
#pragma unroll
  for (int w = N / 2; w >= 1; w >>= 1)
#pragma unroll
    for (int i = 0; i < w; ++i) t[i] = fmaxf(t[2 * i], t[2 * i + 1]);
  return t[0];
}
template <int N>
__device__ __forceinline__ float tree_sum(const float (&v)[N]) {
  float t[N];
#pragma unroll
  for (int i = 0; i < N; ++i) t[i] = v[i];
#pragma unroll
  for (int w = N / 2; w >= 1; w >>= 1)
#pragma unroll
    for (int i = 0; i < w; ++i) t[i] = t[2 * i] + t[2 * i + 1];
  return t[0];
}
// Largest entry and its index; the left operand of every comparison holds the
// lower indices, and it keeps ties, so equal values go to the lower index.
template <int N>
__host__ __device__ __forceinline__ float tree_argmax(const float (&v)[N], int& idx) {
  float t[N];
  int ix[N];
#pragma unroll
  for (int i = 0; i < N; ++i) {
    t[i] = v[i];
    ix[i] = i;
  }
#pragma unroll
  for (int w = N / 2; w >= 1; w >>= 1)
#pragma unroll
    for (int i = 0; i < w; ++i) {
      const bool right = t[2 * i + 1] > t[2 * i];
      t[i] = right ? t[2 * i + 1] : t[2 * i];
      ix[i] = right ? ix[2 * i + 1] : ix[2 * i];
    }
  idx = ix[0];
  return t[0];
}

// The top-k of a row of N logits held in registers (N = 8 G, G <= 4): the
// best remaining entry of each group of 8 columns is kept, so a pick re-scans
// only the 8 columns of its own group instead of the row.  Comparisons keep
// the left (lower-column) operand on ties, within a group and across groups,
// so equal logits go to the lower column, as with a scan of the whole row.
template <int N>
struct RowTopK {
  static_assert(N % 8 == 0 && N <= 32, "groups of 8 columns, at most 32");
  static constexpr int G = N / 8;
  float gv[G];     // best remaining logit of each group
  int gi[G];       // its column
  uint32_t taken;  // columns picked so far

  __host__ __device__ __forceinline__ void init(const float (&v)[N]) {
    taken = 0u;
#pragma unroll
    for (int g = 0; g < G; ++g) {
      float t[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) t[i] = v[8 * g + i];
      int li;
      gv[g] = tree_argmax(t, li);
      gi[g] = 8 * g + li;
    }
  }
  // the best remaining (logit, column)
  __host__ __device__ __forceinline__ float best(int& col) const {
    float t[G];
    int c[G];
#pragma unroll
    for (int g = 0; g < G; ++g) {
      t[g] = gv[g];
      c[g] = gi[g];
    }
#pragma unroll
    for (int w = G / 2; w >= 1; w >>= 1)
#pragma unroll
      for (int g = 0; g < w; ++g) {
        const bool right = t[2 * g + 1] > t[2 * g];
        t[g] = right ? t[2 * g + 1] : t[2 * g];
        c[g] = right ? c[2 * g + 1] : c[2 * g];
      }
    col = c[0];
    return t[0];
  }
  // when pick holds: mark column col taken and re-scan its group
  __host__ __device__ __forceinline__ void take(const float (&v)[N], int col, bool pick) {
    taken |= pick ? 1u << col : 0u;
    const int grp = col >> 3;
    const uint32_t tk = taken >> (8 * grp);
    float t[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      float x = v[i];
#pragma unroll
      for (int g = 1; g < G; ++g) x = grp == g ? v[8 * g + i] : x;
      t[i] = (tk >> i) & 1u ? -INFINITY : x;
    }
    int li;
    const float nv = tree_argmax(t, li);
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const bool upd = pick && g == grp;
      gv[g] = upd ? nv : gv[g];
      gi[g] = upd ? 8 * grp + li : gi[g];
    }
  }
};

__device__ __forceinline__ void epi_bar() {  // the eight epilogue warps
  asm volatile("bar.sync 1, 256;" ::: "memory");
}


// Work split (host side, RouterPlan): the ndt dispatch tiles of SUB tokens
// are dealt over grid = min(SMs, ndt) CTAs in consecutive ranges, base tiles
// each and one more for the first `extra` CTAs, so every SM streams and no
// two ranges differ by more than one tile.  A CTA takes its range in MMA
// tiles of up to tpm dispatch tiles (tpm * SUB <= 128 tokens); per k-block a
// shorter tile's dispatch tiles come in one TMA box of SUB rows each, so no CTA reads
// another's rows, and the last tile's box reads past T as zeros.  A full MMA
// tile's rows come in one box of tpm * SUB rows instead (measured faster than
// tpm boxes at E <= 16).
struct RouterPlan {
  int sub, ndt, grid, base, extra, tpm;
  RouterPlan(int T, int E, int sms) {
    sub = E <= 16 ? 32 : 64;
    ndt = T <= 0 ? 0 : (T + sub - 1) / sub;
    grid = ndt <= 0 ? 0 : std::min(sms, ndt);
    base = grid > 0 ? ndt / grid : 0;
    extra = grid > 0 ? ndt % grid : 0;
    tpm = std::max(1, std::min(base + (extra > 0 ? 1 : 0), kMmaTok / sub));
  }
};

template <int EN, int SUB>
__global__ void __launch_bounds__(kThreads, 1)
    router_tc_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmXs,
                     const __grid_constant__ CUtensorMap tmW,
                     const float* __restrict__ bias, int T, int d, int E, int k,
                     int32_t* __restrict__ idx_out, float* __restrict__ w_out,
                     float* __restrict__ logits_out, float* __restrict__ probs_out,
                     float* __restrict__ aux_partials, int32_t* __restrict__ tile_counts,
                     float* __restrict__ logitsT, int flags, float* __restrict__ z_partials,
                     int base, int extra, int tpm) {
  using C = Cfg<EN>;
  using namespace tc;
  constexpr int HC = EN / 2;  // columns per epilogue half (two-warp rows)
  static_assert(SUB == 32 || SUB == 64, "dispatch tile");
  static_assert(!C::SOLO || SUB == 32, "one-warp rows keep 32-token dispatch tiles");
  static_assert(stages_for(stage_bytes_for(kMmaTok, C::B_BYTES)) >= 2, "ring depth");
  const int a_rows = tpm * SUB;  // tokens of the largest MMA tile
  const int STAGE_BYTES = stage_bytes_for(a_rows, C::B_BYTES);
  const int A_BYTES = a_rows * kBK * 2;
  const int STAGES = stages_for(STAGE_BYTES);
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* ring = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  RSmem& S = *reinterpret_cast<RSmem*>(ring + kRingBytes + kRingPad);
  volatile int* abort_flag = &S.abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nkb = d / kBK;
  const int ndt = (T + SUB - 1) / SUB;
  // this CTA's dispatch tiles [dt0, dt1)
  const int dt0 = (int)blockIdx.x * base + min((int)blockIdx.x, extra);
  const int dt1 = min(ndt, dt0 + base + ((int)blockIdx.x < extra ? 1 : 0));

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&S.full[s], 1);
      mbar_init(&S.empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&S.tmem_full[b], 1);
      mbar_init(&S.tmem_empty[b], C::SOLO ? 4 : 8);  // one arrival per epilogue warp of the tile
    }
    mbar_init(&S.drain, 1);
    S.abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    prefetch_tensormap(&tmX);
    prefetch_tensormap(&tmXs);
    prefetch_tensormap(&tmW);
  }
  if (warp == 1) {
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
  // The ring waits below pass no suspend-time hint: here every stage's round
  // trip (TMA, a few small MMAs, the commit) is on the critical path of the
  // stream, and a suspended waiter wakes late.

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ producer
      int stage = 0;
      uint32_t phase = 0, issued = 0, issued_phase = 0;
      bool ok = true;
      for (int u = dt0; u < dt1 && ok; u += tpm) {
        const int nsub = min(tpm, dt1 - u);  // dispatch tiles in this MMA tile
        const uint32_t bytes = (uint32_t)(nsub * SUB * kBK * 2 + C::B_BYTES);
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait<false, true>(&S.empty[stage], phase ^ 1u, abort_flag, kErrProducer)) {
            ok = false;
            break;
          }
          unsigned char* sA = ring + (size_t)stage * STAGE_BYTES;
          mbar_arrive_expect_tx(&S.full[stage], bytes);
          if (nsub == tpm) {  // a full tile: one box of a_rows rows
            tma_load_2d(sA, &tmX, &S.full[stage], kb * kBK, u * SUB);
          } else {
            for (int j = 0; j < nsub; ++j)
              tma_load_2d(sA + j * SUB * kBK * 2, &tmXs, &S.full[stage], kb * kBK, (u + j) * SUB);
          }
          tma_load_2d(sA + A_BYTES, &tmW, &S.full[stage], kb * kBK, 0);
          issued |= 1u << stage;
          issued_phase = (issued_phase & ~(1u << stage)) | (phase << stage);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // every issued load lands before the CTA exits
      for (int s = 0; s < STAGES; ++s) {
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
      constexpr uint32_t idesc = make_idesc_bf16(kMmaTok, C::NM);
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      for (int u = dt0; u < dt1 && ok; u += tpm) {
        if (!mbar_wait<false, true>(&S.tmem_empty[acc], acc_phase ^ 1u, abort_flag, kErrMma)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem + (uint32_t)(acc * C::NM);
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait<false, true>(&S.full[stage], phase, abort_flag, kErrMma)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = smem_u32(ring + (size_t)stage * STAGE_BYTES);
          const uint32_t b0 = a0 + A_BYTES;
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk)
            tc_mma_f16(d_tmem, sw128_desc(a0 + kk * 32), sw128_desc(b0 + kk * 32), idesc,
                       (kb | kk) != 0 ? 1u : 0u);
          tc_commit(&S.empty[stage]);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        tc_commit(&S.tmem_full[acc]);
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      // every issued MMA completes before TMEM is released
      tc_commit(&S.drain);
      const uint32_t a = smem_u32(&S.drain);
      const uint64_t t0 = global_timer_ns();
      while (!mbar_try_wait(a, 0)) {
        if (global_timer_ns() - t0 > kWaitTimeoutNs) {
          record_error(kErrDrain);
          break;
        }
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int ew = warp - 2;          // 0..7
    const int q = warp & 3;           // TMEM lane quarter: tile rows 32q .. 32q + 31
    const int h = ew >> 2;            // warps 2-5: 0, warps 6-9: 1
    for (int e = threadIdx.x - 64; e < MOE_MAX_EXPERTS; e += kEpiThreads)
      S.bias[e] = (bias != nullptr && e < E) ? bias[e] : 0.f;
    epi_bar();
    if constexpr (C::SOLO) {
      // One warp per lane quarter and tile: thread (q, lane) holds all EN
      // columns of token row 32q + lane; group h takes the MMA tiles of
      // accumulator h (the even or the odd tiles of this CTA).
      int ord = 0;  // MMA tiles of this CTA so far
      for (int u = dt0; u < dt1; u += tpm, ++ord) {
        const int acc = ord & 1;
        if (acc != h) continue;
        const uint32_t acc_phase = (uint32_t)(ord >> 1) & 1u;
        const int tok0 = u * SUB;
        const int ntok = min(min(dt1, u + tpm) * SUB, T) - tok0;
        // a wait that gives up sets the abort flag (the error word records it)
        mbar_wait<false, true>(&S.tmem_full[acc], acc_phase, abort_flag, kErrEpilogue);
        tc_fence_after();
        const bool qlive = q * 32 < ntok;  // warp-uniform: dispatch tile u + q is this CTA's
        const int r = q * 32 + lane;       // tile row = TMEM lane
        const bool live = qlive && r < ntok;
        const int t = tok0 + r;
        float sr[EN];
        if (qlive) {
          uint32_t v[EN];
          tmem_chunk<EN>(tmem + (uint32_t)(acc * C::NM) + ((uint32_t)(q * 32) << 16), v);
#pragma unroll
          for (int i = 0; i < EN; ++i) sr[i] = i < E ? __uint_as_float(v[i]) + S.bias[i] : -INFINITY;
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.tmem_empty[acc]);
        if (!qlive) continue;
        float m = -INFINITY, inv = 0.f, lse = 0.f;
        float ex[EN];
        if (k > 0) {
          m = tree_max(sr);
#pragma unroll
          for (int i = 0; i < EN; ++i) ex[i] = i < E ? expf(sr[i] - m) : 0.f;
          const float sum = tree_sum(ex);
          inv = 1.0f / sum;
          lse = m + logf(sum);
        }
        if (live) {
#pragma unroll
          for (int i = 0; i < EN; ++i) {
            if (i < E) {
              if (logits_out) logits_out[(size_t)t * E + i] = sr[i];
              if (logitsT) logitsT[(size_t)i * T + t] = sr[i];
              if (k > 0 && probs_out) probs_out[(size_t)t * E + i] = ex[i] * inv;
            }
          }
        }
        if (k == 0) continue;
        const int tile = u + q;  // the dispatch tile of this quarter
        if (aux_partials) {
          float g[EN];
#pragma unroll
          for (int i = 0; i < EN; ++i) g[i] = live ? ex[i] * inv : 0.f;
          const float colsum = warp_transpose_sum<EN>(g);  // lane l: column l % EN
          if (lane < E) aux_partials[(size_t)tile * E + lane] = colsum;
        }
        if (tile_counts) {
          if (lane < 16) S.cnt16[ew][lane] = 0;
          __syncwarp();
        }
        // top-k: repeated arg-max over the remaining columns (ties to the lower index)
        RowTopK<EN> tk;
        tk.init(sr);
        float gk[8];
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) gk[jj] = 0.f;
        float selsum = 0.f;
#pragma unroll 1
        for (int j = 0; j < k; ++j) {
          int sel;
          float best = tk.best(sel);
          tk.take(sr, sel, true);
          if (!(best > -INFINITY)) {  // only for non-finite logits: stay in range
            sel = j < E ? j : 0;
            best = -INFINITY;
          }
          const float gs = expf(best - m) * inv;  // same arithmetic as the probabilities
          selsum += gs;
#pragma unroll
          for (int jj = 0; jj < 8; ++jj) gk[jj] = jj == j ? gs : gk[jj];
          if (live) {
            idx_out[(size_t)t * k + j] = sel;
            w_out[(size_t)t * k + j] = gs;
          }
          if (tile_counts) {  // one shared atomic per distinct expert of the warp
            const unsigned peers = __match_any_sync(kFullMask, live ? sel : -1);
            if (live && lane == __ffs(peers) - 1) atomicAdd(&S.cnt16[ew][sel], __popc(peers));
          }
        }
        if (live && !(flags & MOE_ROUTE_NO_RENORM)) {
          const float rs = 1.0f / selsum;
#pragma unroll
          for (int jj = 0; jj < 8; ++jj)
            if (jj < k) w_out[(size_t)t * k + jj] = gk[jj] * rs;
          for (int j = 8; j < k; ++j) w_out[(size_t)t * k + j] *= rs;
        }
        // per-dispatch-tile expert counts and z sums
        float z = (live && z_partials) ? lse * lse : 0.f;
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) z += __shfl_xor_sync(kFullMask, z, o);
        if (tile_counts) {
          __syncwarp();
          if (lane < E) tile_counts[(size_t)tile * E + lane] = S.cnt16[ew][lane];
        }
        if (z_partials && lane == 0) z_partials[tile] = z;
      }
    } else {
      // Two warps per TMEM lane quarter: thread (q, h, lane) handles token row
      // 32q + lane and the expert columns [h * HC, (h + 1) * HC) of it.  The
      // pair exchanges its partial max and sum and, per top-k pass, its best
      // candidate through shared memory (a named barrier per quarter); half 0
      // writes the selection, counts and z sums.  Both warps of a pair run the
      // same sequence of barriers whatever happens to a wait, so none can hang.
      const int col0 = h * HC;
      int acc = 0;
      uint32_t acc_phase = 0;
      int xc = 0;  // pair exchanges so far
      // the pair's max (either order gives the same value) and sum (half 0's first)
      auto pair_max = [&](float v, int r) {
        float o;
        int oi;
        pair_xchg(S, v, 0, o, oi, h, q, r, xc);
        return fmaxf(v, o);
      };
      auto pair_sum = [&](float v, int r) {
        float o;
        int oi;
        pair_xchg(S, v, 0, o, oi, h, q, r, xc);
        return h == 0 ? v + o : o + v;
      };
      for (int u = dt0; u < dt1; u += tpm) {
        const int tok0 = u * SUB;
        const int ntok = min(min(dt1, u + tpm) * SUB, T) - tok0;
        // a wait that gives up sets the abort flag (the error word records it); the
        // warp still runs the tile's barriers, with garbage values
        mbar_wait<false, true>(&S.tmem_full[acc], acc_phase, abort_flag, kErrEpilogue);
        tc_fence_after();
        const bool qlive = q * 32 < ntok;  // uniform over the pair
        const int r = q * 32 + lane;       // tile row = TMEM lane
        const bool live = qlive && r < ntok;
        const int t = tok0 + r;
        const uint32_t trow = tmem + (uint32_t)(acc * EN + col0) + ((uint32_t)(q * 32) << 16);
        float m = -INFINITY, inv = 0.f, lse = 0.f;
        float gk[8];  // half 0: the first 8 selected probabilities
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) gk[jj] = 0.f;
        if (k > 0 && tile_counts && h == 0) {  // expert counts, filled by the top-k below
          __syncwarp();  // the previous tile's counts have been read
          for (int e = lane; e < E; e += 32) S.cnt[q][e] = 0;
          __syncwarp();
        }
        if constexpr (HC <= 32) {
          // this half's columns in registers; TMEM is released before any arithmetic
          float sr[HC];
          if (qlive) {
            uint32_t v[HC];
            tmem_chunk<HC>(trow, v);
#pragma unroll
            for (int i = 0; i < HC; ++i)
              sr[i] = col0 + i < E ? __uint_as_float(v[i]) + S.bias[col0 + i] : -INFINITY;
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&S.tmem_empty[acc]);
          if (qlive) {
            float ex[HC];
            if (k > 0) {
              m = pair_max(tree_max(sr), r);
#pragma unroll
              for (int i = 0; i < HC; ++i) ex[i] = col0 + i < E ? expf(sr[i] - m) : 0.f;
              const float sum = pair_sum(tree_sum(ex), r);
              inv = 1.0f / sum;
              lse = m + logf(sum);
            }
            if (live) {
#pragma unroll
              for (int i = 0; i < HC; ++i) {
                const int e = col0 + i;
                if (e < E) {
                  if (logits_out) logits_out[(size_t)t * E + e] = sr[i];
                  if (logitsT) logitsT[(size_t)e * T + t] = sr[i];
                  if (k > 0 && probs_out) probs_out[(size_t)t * E + e] = ex[i] * inv;
                }
              }
            }
            if (k > 0 && aux_partials) {
              float g[HC];
#pragma unroll
              for (int i = 0; i < HC; ++i) g[i] = live ? ex[i] * inv : 0.f;
              const float colsum = warp_transpose_sum<HC>(g);  // lane l: column col0 + l % HC
              if (lane < HC && col0 + lane < E) {
                if (SUB == 32) aux_partials[(size_t)(u + q) * E + col0 + lane] = colsum;
                else S.gsum[q][col0 + lane] = colsum;
              }
            }
            if (k > 0) {
              // top-k: each pass takes the better of the two halves' best remaining
              // columns (ties to the lower index, which half 0 holds); the winner
              // marks its pick taken
              RowTopK<HC> tk;
              tk.init(sr);
              float selsum = 0.f;
#pragma unroll 1
              for (int j = 0; j < k; ++j) {
                int bi;
                float bv = tk.best(bi);  // bi: column within this half
                float ov;
                int oi;
                pair_xchg(S, bv, col0 + bi, ov, oi, h, q, r, xc);
                const bool mine = h == 0 ? !(ov > bv) : (bv > ov);
                tk.take(sr, bi, mine);
                float best = mine ? bv : ov;
                int sel = mine ? col0 + bi : oi;
                if (!(best > -INFINITY)) {  // only for non-finite logits: stay in range
                  sel = j < E ? j : 0;
                  best = -INFINITY;
                }
                const float gs = expf(best - m) * inv;  // same arithmetic as the probabilities
                selsum += gs;
#pragma unroll
                for (int jj = 0; jj < 8; ++jj) gk[jj] = jj == j ? gs : gk[jj];
                if (live && h == 0) {
                  idx_out[(size_t)t * k + j] = sel;
                  w_out[(size_t)t * k + j] = gs;
                }
                if (tile_counts && h == 0) {  // one shared atomic per distinct expert of the warp
                  const unsigned peers = __match_any_sync(kFullMask, live ? sel : -1);
                  if (live && lane == __ffs(peers) - 1) atomicAdd(&S.cnt[q][sel], __popc(peers));
                }
              }
              if (live && h == 0 && !(flags & MOE_ROUTE_NO_RENORM)) {
                const float rs = 1.0f / selsum;
#pragma unroll
                for (int jj = 0; jj < 8; ++jj)
                  if (jj < k) w_out[(size_t)t * k + jj] = gk[jj] * rs;
                for (int j = 8; j < k; ++j) w_out[(size_t)t * k + j] *= rs;
              }
            }
          }
        } else {
          // wide rows (E > 64): this half's columns in 32-column chunks, read from
          // TMEM once per pass
          if (qlive) {
            if (k > 0) {
              float mh = -INFINITY;
#pragma unroll 1
              for (int c = 0; c < HC; c += 32) {
                uint32_t v[32];
                tmem_chunk<32>(trow + c, v);
#pragma unroll
                for (int i = 0; i < 32; ++i)
                  if (col0 + c + i < E) mh = fmaxf(mh, __uint_as_float(v[i]) + S.bias[col0 + c + i]);
              }
              m = pair_max(mh, r);
              float sh = 0.f;
#pragma unroll 1
              for (int c = 0; c < HC; c += 32) {
                uint32_t v[32];
                tmem_chunk<32>(trow + c, v);
#pragma unroll
                for (int i = 0; i < 32; ++i)
                  if (col0 + c + i < E) sh += expf(__uint_as_float(v[i]) + S.bias[col0 + c + i] - m);
              }
              const float sum = pair_sum(sh, r);
              inv = 1.0f / sum;
              lse = m + logf(sum);
            }
#pragma unroll 1
            for (int c = 0; c < HC; c += 32) {
              uint32_t v[32];
              tmem_chunk<32>(trow + c, v);
              float g[32];
#pragma unroll
              for (int i = 0; i < 32; ++i) {
                const int e = col0 + c + i;
                const float s = __uint_as_float(v[i]) + S.bias[e < E ? e : 0];
                g[i] = 0.f;
                if (live && e < E) {
                  if (logits_out) logits_out[(size_t)t * E + e] = s;
                  if (logitsT) logitsT[(size_t)e * T + t] = s;
                  if (k > 0) {
                    const float p = expf(s - m) * inv;
                    if (probs_out) probs_out[(size_t)t * E + e] = p;
                    g[i] = p;
                  }
                }
              }
              if (k > 0 && aux_partials) {
                const float colsum = warp_transpose_sum<32>(g);  // lane l: column col0 + c + l
                if (col0 + c + lane < E) {
                  if (SUB == 32) aux_partials[(size_t)(u + q) * E + col0 + c + lane] = colsum;
                  else S.gsum[q][col0 + c + lane] = colsum;
                }
              }
            }
            if (k > 0) {
              // the j-th pick is the largest (logit, -index) strictly after the
              // previous one, the better of the two halves' candidates
              float pv = INFINITY, selsum = 0.f;
              int pi = -1;
#pragma unroll 1
              for (int j = 0; j < k; ++j) {
                float bv = -INFINITY;
                int bi = -1;
#pragma unroll 1
                for (int c = 0; c < HC; c += 32) {
                  uint32_t v[32];
                  tmem_chunk<32>(trow + c, v);
#pragma unroll
                  for (int i = 0; i < 32; ++i) {
                    const int e = col0 + c + i;
                    if (e < E) {
                      const float s = __uint_as_float(v[i]) + S.bias[e];
                      const bool after = s < pv || (s == pv && e > pi);
                      if (after && (bi < 0 ? s > -INFINITY : s > bv)) {
                        bv = s;
                        bi = e;
                      }
                    }
                  }
                }
                float ov;
                int oi;
                pair_xchg(S, bv, bi, ov, oi, h, q, r, xc);
                // half 0 holds the lower indices: it wins ties; no candidate loses
                const bool mine = bi >= 0 && (oi < 0 || (h == 0 ? !(ov > bv) : (bv > ov)));
                float best = mine ? bv : ov;
                int sel = mine ? bi : oi;
                if (sel < 0) {  // only for non-finite logits: stay in range
                  sel = j < E ? j : 0;
                  best = -INFINITY;
                } else {
                  pv = best;
                  pi = sel;
                }
                const float gs = expf(best - m) * inv;  // same arithmetic as the probabilities
                selsum += gs;
#pragma unroll
                for (int jj = 0; jj < 8; ++jj) gk[jj] = jj == j ? gs : gk[jj];
                if (live && h == 0) {
                  idx_out[(size_t)t * k + j] = sel;
                  w_out[(size_t)t * k + j] = gs;
                }
                if (tile_counts && h == 0) {  // one shared atomic per distinct expert of the warp
                  const unsigned peers = __match_any_sync(kFullMask, live ? sel : -1);
                  if (live && lane == __ffs(peers) - 1) atomicAdd(&S.cnt[q][sel], __popc(peers));
                }
              }
              if (live && h == 0 && !(flags & MOE_ROUTE_NO_RENORM)) {
                const float rs = 1.0f / selsum;
#pragma unroll
                for (int jj = 0; jj < 8; ++jj)
                  if (jj < k) w_out[(size_t)t * k + jj] = gk[jj] * rs;
                for (int j = 8; j < k; ++j) w_out[(size_t)t * k + j] *= rs;
              }
            }
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&S.tmem_empty[acc]);
        }
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1u;
        }
        if (k == 0) continue;
        // per-dispatch-tile expert counts (counted during the top-k) and z sums (half 0)
        float z = (live && z_partials) ? lse * lse : 0.f;
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) z += __shfl_xor_sync(kFullMask, z, o);
        if (SUB == 32) {
          if (qlive && h == 0) {
            __syncwarp();
            const int tile = u + q;
            if (tile_counts)
              for (int e = lane; e < E; e += 32) tile_counts[(size_t)tile * E + e] = S.cnt[q][e];
            if (z_partials && lane == 0) z_partials[tile] = z;
          }
        } else {
          if (h == 0) {
            if (lane == 0) S.zsum[q] = z;
            if (!qlive)  // an empty quarter contributes nothing to its pair
              for (int e = lane; e < E; e += 32) S.cnt[q][e] = 0;
          }
          if (!qlive)
            for (int e = col0 + lane; e < col0 + HC && e < E; e += 32) S.gsum[q][e] = 0.f;
          epi_bar();
          if ((q & 1) == 0 && qlive && h == 0) {  // quarters q, q+1 form dispatch tile u + q / 2
            const int tile = u + (q >> 1);
            for (int e = lane; e < E; e += 32) {
              if (tile_counts) tile_counts[(size_t)tile * E + e] = S.cnt[q][e] + S.cnt[q + 1][e];
              if (aux_partials) aux_partials[(size_t)tile * E + e] = S.gsum[q][e] + S.gsum[q + 1][e];
            }
            if (z_partials && lane == 0) z_partials[tile] = S.zsum[q] + S.zsum[q + 1];
          }
          epi_bar();  // the staging arrays are reused by the next tile
        }
      }
    }  // two-warp rows
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(C::TMEM_COLS)
                 : "memory");
  }
}

template <int EN, int SUB>
cudaError_t launch_en(const RouterPlan& P, const CUtensorMap& mx, const CUtensorMap& mxs,
                      const CUtensorMap& mw, const float* bias, int T, int d, int E, int k,
                      int32_t* idx, float* w, float* logits, float* probs, float* aux,
                      int32_t* tile_counts, float* logitsT, int flags, float* z_partials,
                      cudaStream_t st) {
  constexpr size_t sm = smem_bytes<EN>();
  static_assert(sm <= 227 * 1024, "router shared memory");
  auto kern = router_tc_kernel<EN, SUB>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
  if (e != cudaSuccess) return e;
  return launch_k(kern, dim3(P.grid), dim3(kThreads), sm, st, nullptr, 0, mx, mxs, mw, bias, T, d, E, k,
                  idx, w, logits, probs, aux, tile_counts, logitsT, flags, z_partials, P.base, P.extra,
                  P.tpm);
}

// Which bf16 router runs (measured, CUDA events with the stream held, L2
// flushed): the tensor-core one from E > 16 on (T=16384, d=2048, E=64: 28.7 us
// against 38.9 us for the warp-MMA router) and for inputs of 32 MiB or more
// (T=16384, d=4096, E=8: 41.0 against 45.1 us); the warp-MMA router below that
// (T=8192, d=1024, E=8: 12.3 against 14.3 us: a short read, where the
// persistent kernel's set-up and epilogue tail dominate).  MOE_ROUTER_TC=0 / 1
// in the environment forces one (tests, A/B timing).
inline bool tc_router_enabled(int T, int d, int E) {
  const char* v = getenv("MOE_ROUTER_TC");
  if (v && v[0] == '0') return false;
  if (v && v[0] == '1') return true;
  return E > 16 || (long long)T * d >= (16LL << 20);
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
  if (!bf16 || !rtc::tc_router_enabled(T, d, E))
    return launch_router_mma(x, wg, bias, T, d, E, k, bf16, idx, w, logits, probs, aux, st,
                             tile_counts, logitsT, flags, z_partials);
  const int en = E <= 8 ? 8 : E <= 16 ? 16 : E <= 32 ? 32 : E <= 64 ? 64 : E <= 128 ? 128 : 256;
  const int nm = en < 16 ? 16 : en;  // the MMA's N: W_g rows per box, past E zero-filled
  // the dispatch tile: router_tokens(E) tokens (32 up to E = 16, 64 above)
  const rtc::RouterPlan P(T, E, tc::sm_count());
  CUtensorMap mx, mxs, mw;
  if (!tc::make_map(&mx, x, (uint64_t)T, (uint64_t)d, (uint32_t)(P.tpm * P.sub)) ||
      !tc::make_map(&mxs, x, (uint64_t)T, (uint64_t)d, (uint32_t)P.sub) ||
      !tc::make_map(&mw, wg, (uint64_t)E, (uint64_t)d, (uint32_t)nm))
    return cudaErrorInvalidValue;
  switch (en) {
    case 8:
      return rtc::launch_en<8, 32>(P, mx, mxs, mw, bias, T, d, E, k, idx, w, logits, probs, aux,
                                   tile_counts, logitsT, flags, z_partials, st);
    case 16:
      return rtc::launch_en<16, 32>(P, mx, mxs, mw, bias, T, d, E, k, idx, w, logits, probs, aux,
                                    tile_counts, logitsT, flags, z_partials, st);
    case 32:
      return rtc::launch_en<32, 64>(P, mx, mxs, mw, bias, T, d, E, k, idx, w, logits, probs, aux,
                                    tile_counts, logitsT, flags, z_partials, st);
    case 64:
      return rtc::launch_en<64, 64>(P, mx, mxs, mw, bias, T, d, E, k, idx, w, logits, probs, aux,
                                    tile_counts, logitsT, flags, z_partials, st);
    case 128:
      return rtc::launch_en<128, 64>(P, mx, mxs, mw, bias, T, d, E, k, idx, w, logits, probs, aux,
                                     tile_counts, logitsT, flags, z_partials, st);
    default:
      return rtc::launch_en<256, 64>(P, mx, mxs, mw, bias, T, d, E, k, idx, w, logits, probs, aux,
                                     tile_counts, logitsT, flags, z_partials, st);
  }
}

}  // namespace moe
