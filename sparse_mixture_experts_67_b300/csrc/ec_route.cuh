// Expert-choice routing: ExpertChoiceGating.forward of "Sparse Mixture of
// Experts(MoE) 아키텍처 심층 분석" (youngju.dev).
//
// Each expert scores all tokens with a softmax over its logit column and keeps
// the C best tokens, C = floor(T * capacity_factor / E), in descending score
// order with ties to the lower token.  The logits come from the router kernel
// run in logits-only mode, which also writes them transposed into pos ([E, T],
// as fp32 bits); the select below reads each expert's row there once,
// coalesced, and then overwrites it with the position map.
#pragma once

#include <float.h>

#include "common.cuh"

namespace moe {


// Block-wide (max m, sum of exp(v - m)) of one value per thread (valid ones
// only; blockDim a multiple of 32, at most 1024): each warp reduces its max and
// its sum about that max with butterflies, then warp 0 merges the warps' pairs,
// rescaling each warp's sum by exp(m_w - m).  The order of the operations is
// fixed, and every thread returns the same pair.  scratch holds 66 floats.
__device__ __forceinline__ float2 block_max_sumexp(float v, bool valid, float* scratch) {
  float m = valid ? v : -FLT_MAX;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(kFullMask, m, off));
  float sum = valid ? expf(v - m) : 0.f;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(kFullMask, sum, off);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) {
    scratch[warp] = m;
    scratch[33 + warp] = sum;
  }
  __syncthreads();
  if (warp == 0) {
    const bool have = lane < (int)(blockDim.x >> 5);
    const float mw = have ? scratch[lane] : -FLT_MAX;
    float M = mw;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(kFullMask, M, off));
    float x = have ? scratch[33 + lane] * expf(mw - M) : 0.f;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(kFullMask, x, off);
    __syncwarp();
    if (lane == 0) {
      scratch[32] = M;
      scratch[65] = x;
    }
  }
  __syncthreads();
  return make_float2(scratch[32], scratch[65]);
}

// Order-preserving map of a float to uint32 (ascending float -> ascending key).
__device__ __forceinline__ uint32_t float_order_key(float v) {
  const uint32_t u = __float_as_uint(v + 0.0f);  // -0 -> +0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Inverse of float_order_key (exact; -0 comes back as +0).
__device__ __forceinline__ float order_key_float(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}



// ------------------------------------------------------------ two-stage select
// Expert e's logit column is cut into S = ceil(T / kEcSlice) slices; stage 1
// runs one CTA per (slice, expert), stage 2 likewise, so E * S CTAs share the
// work instead of E.
//   stage 1 (ec_slice_kernel): the slice's max and sum of exponentials (about
//     its own max), its pos entries set to -1, and its tokens sorted by
//     descending logit then ascending token (32-bit keys, ascending; a bitonic
//     sort within warps, then stable merge rounds in shared memory); the first
//     L = min(C, kEcSlice) are the slice's candidates, keys and tokens in two
//     arrays (past the slice end: sentinel keys above every real key).
//   stage 2 (ec_rank_kernel): every candidate's rank among all candidates of
//     its expert is its index in its own list plus, for every other list, the
//     number of entries ahead of it (binary search on the keys, one thread per
//     candidate and list): equal keys count as ahead in the lists of earlier
//     slices (lower tokens) and as behind in later ones.  A token of the
//     expert's top C has every token ahead of it within the first C of each
//     slice, so those ranks are exact; any other candidate gets a rank of at
//     least C.  Ranks grow along a sorted list, so the candidates are taken
//     in chunks from the front and the phase stops at the first chunk that
//     reaches rank C.  Ranks below C place the token: ec_idx / ec_score at the
//     rank, pos[e, t] = e * C + rank.  The column's max and sum come from the
//     slices' pairs, merged by one warp in a fixed order.
constexpr int kEcSlice = 1024;            // tokens per stage-1 CTA (one per thread)
constexpr int kEcRankThreads = 1024;
constexpr size_t kEcRankSmemMax = 160 * 1024;  // dynamic shared memory of the rank phase, at most
// The lists are staged in shared memory up to this many keys in all (80 KB): a
// larger staging copy costs more than the few search chunks it speeds up
// (T = 32768, E = 16, 32 lists of 1024: the whole route took 92 us with the
// lists staged, 80 us with the searches in L2).
constexpr size_t kEcStageKeysMax = 20480;

inline int ec_slices(int T) { return T <= 0 ? 0 : ceil_div(T, kEcSlice); }
inline int ec_list_len(int C) { return C < kEcSlice ? C : kEcSlice; }

// Scratch of the select, bytes: candidate keys [E, S, L] (u32) and tokens
// [E, S, L] (int32), the slices' (max, sum) pairs [E, S] (float2) and the
// per-expert arrival counts [E] of the one-launch form, each region 256-byte
// aligned.
inline size_t ec_align256(size_t b) { return (b + 255) / 256 * 256; }
inline size_t ec_scratch_bytes(int T, int E, int C) {
  const size_t S = (size_t)ec_slices(T), L = (size_t)ec_list_len(C > 0 ? C : 1);
  return 2 * ec_align256((size_t)E * S * L * 4) + ec_align256((size_t)E * S * 8) +
         (size_t)E * sizeof(int);
}

// MOE_EC_TWO_LAUNCHES=1 in the environment keeps the two stages as two
// launches (tests, A/B timing).
inline bool ec_two_launches() {
  const char* v = getenv("MOE_EC_TWO_LAUNCHES");
  return v && v[0] == '1';
}

// Number of entries of the ascending list a[0..n) below key (LE: at most key).
template <bool LE>
__device__ __forceinline__ int count_ahead(const uint32_t* a, int n, uint32_t key) {
  int lo = 0, hi = n;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (LE ? a[mid] <= key : a[mid] < key) lo = mid + 1;
    else hi = mid;
  }
  return lo;
}

// Key of a logit: ascending key = descending logit.  Past the slice end the
// key is kEcSentinel, above every finite or infinite logit's key (at most
// 0xFF800000).
__device__ __forceinline__ uint32_t ec_key(float v) { return ~float_order_key(v); }
constexpr uint32_t kEcSentinel = 0xFFFFFFFFu;

// Sort of the CTA's kEcSlice (key, token) pairs, one per thread, thread i
// holding the slice's i-th token: ascending key, ties by ascending token.  A
// bitonic sort of each warp's 32 pairs in registers (packed into 64 bits, so
// ties resolve by token), then five rounds that merge pairs of sorted runs,
// each pair moving to its index in its own run plus the number of pairs of the
// partner run ahead of it.  A run holds the tokens of one contiguous range, so
// the left run's tokens are the lower ones: a left pair counts the right run's
// keys below its own, a right pair the left run's keys at or below its own.
// The searches read 32-bit keys only.  Returns the buffer index (0 or 1)
// holding the result.
__device__ __forceinline__ int slice_sort(uint32_t key, int32_t tok, uint32_t (*sk)[kEcSlice],
                                          int32_t (*st)[kEcSlice]) {
  const int tid = threadIdx.x, lane = tid & 31;
  unsigned long long kt = ((unsigned long long)key << 32) | (uint32_t)tok;
#pragma unroll
  for (int kk = 2; kk <= 32; kk <<= 1) {
#pragma unroll
    for (int j = kk >> 1; j > 0; j >>= 1) {
      const unsigned long long other = __shfl_xor_sync(kFullMask, kt, j);
      const bool take_min = ((lane & j) == 0) == ((lane & kk) == 0);
      kt = take_min ? (other < kt ? other : kt) : (other > kt ? other : kt);
    }
  }
  int src = 0;
  sk[0][tid] = (uint32_t)(kt >> 32);
  st[0][tid] = (int32_t)(uint32_t)kt;
  __syncthreads();
#pragma unroll 1
  for (int len = 32; len < kEcSlice; len <<= 1) {
    const uint32_t k = sk[src][tid];  // the pair now at this thread's position
    const int32_t t = st[src][tid];
    const int run = tid / len, idx = tid - run * len;
    const uint32_t* part = sk[src] + (run ^ 1) * len;
    const int ahead = (run & 1) ? count_ahead<true>(part, len, k) : count_ahead<false>(part, len, k);
    const int at = (run & ~1) * len + idx + ahead;
    sk[src ^ 1][at] = k;
    st[src ^ 1][at] = t;
    __syncthreads();
    src ^= 1;
  }
  return src;
}

// Stage 1 for (slice sl, expert e): the slice's (max, sum) pair, its pos
// entries set to -1 after they were read, and (C > 0) its first L sorted keys.
__device__ __forceinline__ void ec_slice_phase(int T, int C, int L, int S, int e, int sl,
                                               int32_t* __restrict__ pos,
                                               uint32_t* __restrict__ ckey,
                                               int32_t* __restrict__ ctok,
                                               float2* __restrict__ stats,
                                               uint32_t (*sk)[kEcSlice], int32_t (*st)[kEcSlice],
                                               float* scratch) {
  const int t0 = sl * kEcSlice;
  const int n = min(kEcSlice, T - t0);
  const int tid = threadIdx.x;
  int32_t* prow = pos + (size_t)e * T + t0;  // on entry: this expert's logits (fp32 bits)
  float v = -FLT_MAX;
  uint32_t key = kEcSentinel;
  if (tid < n) {
    v = __int_as_float(prow[tid]);
    key = ec_key(v);
  }
  const float2 ms = block_max_sumexp(v, tid < n, scratch);  // the slice is read past here
  if (tid < n) prow[tid] = -1;
  if (threadIdx.x == 0) stats[(size_t)e * S + sl] = ms;
  if (C <= 0) return;
  const int b = slice_sort(key, t0 + tid, sk, st);
  const size_t o = ((size_t)e * S + sl) * L;
  for (int i = tid; i < L; i += blockDim.x) {
    ckey[o + i] = sk[b][i];
    ctok[o + i] = st[b][i];
  }
}

// Stage 2 for (slice sl, expert e): ranks of the slice's candidates among all
// of the expert's; ranks below C place the token.  Reads other CTAs' lists and
// pairs through L2 (ld.global.cg), so the fused kernel may run it right after
// its wait.  stage_smem: the lists are first copied to s_lists in shared
// memory; the searches then read shared memory, else the lists in global
// memory (two separate pointers, so that each path keeps its own address space).
__device__ __forceinline__ void ec_rank_phase(int T, int C, int L, int S, int e, int sl,
                                              const uint32_t* __restrict__ ckey,
                                              const int32_t* __restrict__ ctok,
                                              const float2* __restrict__ stats, int stage_smem,
                                              uint32_t* s_lists,
                                              int32_t* __restrict__ ec_idx,
                                              float* __restrict__ ec_score,
                                              int32_t* __restrict__ pos, float* s_mi, int* s_cnt) {
  const uint32_t* lists = ckey + (size_t)e * S * L;
  const int32_t* toks = ctok + (size_t)e * S * L;
  if (stage_smem) {  // all S key lists of this expert, staged once
    const int n = S * L;
    const int nt = blockDim.x;
    if ((((size_t)e * S * L) & 3) == 0 && (n & 3) == 0) {  // 16-byte pieces, 4 in flight
      const uint4* g4 = reinterpret_cast<const uint4*>(lists);
      uint4* s4 = reinterpret_cast<uint4*>(s_lists);
      const int n4 = n >> 2;
      int i = threadIdx.x;
      for (; i + 3 * nt < n4; i += 4 * nt) {
        const uint4 a = __ldcg(g4 + i), b = __ldcg(g4 + i + nt), c = __ldcg(g4 + i + 2 * nt),
                    d = __ldcg(g4 + i + 3 * nt);
        s4[i] = a;
        s4[i + nt] = b;
        s4[i + 2 * nt] = c;
        s4[i + 3 * nt] = d;
      }
      for (; i < n4; i += nt) s4[i] = __ldcg(g4 + i);
    } else {
      for (int j = threadIdx.x; j < n; j += nt) s_lists[j] = __ldcg(lists + j);
    }
  }
  if (threadIdx.x < 32) {  // the column's softmax denominator: lane l merges slices l, l + 32, ...
    const float2* stp = stats + (size_t)e * S;
    const int lane = threadIdx.x;
    float m = -FLT_MAX, sum = 0.f;
    for (int i = lane; i < S; i += 32) {
      const float2 p = __ldcg(stp + i);
      const float mm = fmaxf(m, p.x);
      sum = sum * expf(m - mm) + p.y * expf(p.x - mm);
      m = mm;
    }
    float M = m;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(kFullMask, M, off));
    float x = sum * expf(m - M);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(kFullMask, x, off);
    if (lane == 0) {
      s_mi[0] = M;
      s_mi[1] = 1.0f / x;
    }
  }
  __syncthreads();
  const float m = s_mi[0], inv = s_mi[1];
  const int P = S - 1;  // the other lists
  // Chunks of B keys, one thread per (key, list slot): slot jj searches the
  // other lists jj, jj + J, ... (one list each unless there are more lists
  // than threads).  Ranks grow along the sorted list, so the chunks stop after
  // the first whose last key ranks at or beyond C (or runs past the list).
  const int B = P > 0 ? max(1, (int)blockDim.x / P) : (int)blockDim.x;
  const int J = (int)blockDim.x / B;  // list slots
  const int kc = (int)threadIdx.x % B, jj = (int)threadIdx.x / B;
#pragma unroll 1
  for (int c0 = 0; c0 < L; c0 += B) {
    const int c = c0 + kc;
    const bool key_thread = jj == 0 && c < L;
    uint32_t key = 0u;
    bool real = false;
    if (c < L && jj < J) {
      const size_t at = (size_t)sl * L + c;
      key = stage_smem ? s_lists[at] : __ldcg(lists + at);
      real = key != kEcSentinel;  // else past the slice end
      int cnt = 0;
      if (real)
        for (int q = jj; q < P; q += J) {
          const bool before = q < sl;  // an earlier slice: its equal keys are lower tokens
          const size_t o = (size_t)(before ? q : q + 1) * L;
          const uint32_t* a = stage_smem ? nullptr : lists + o;
          if (stage_smem)
            cnt += before ? count_ahead<true>(s_lists + o, L, key) : count_ahead<false>(s_lists + o, L, key);
          else
            cnt += before ? count_ahead<true>(a, L, key) : count_ahead<false>(a, L, key);
        }
      s_cnt[jj * B + kc] = cnt;
    }
    __syncthreads();
    bool more = false;
    if (key_thread) {
      int rank = c;
      for (int q = 0; q < J; ++q) rank += s_cnt[q * B + kc];
      if (real && rank < C) {
        const int t = __ldcg(toks + (size_t)sl * L + c);
        const float v = order_key_float(key ^ 0xffffffffu);
        ec_idx[(size_t)e * C + rank] = t;
        ec_score[(size_t)e * C + rank] = expf(v - m) * inv;
        pos[(size_t)e * T + t] = e * C + rank;
      }
      more = (kc == B - 1) && real && rank < C;  // the chunk's last key still places a token
    }
    if (!__syncthreads_or(more)) break;  // also keeps s_cnt until every key thread read it
  }
}

__global__ void __launch_bounds__(kEcSlice)
    ec_slice_kernel(int T, int E, int C, int L, int32_t* __restrict__ pos,
                    uint32_t* __restrict__ ckey, int32_t* __restrict__ ctok,
                    float2* __restrict__ stats) {
  pdl_begin();
  __shared__ uint32_t s_key[2][kEcSlice];
  __shared__ int32_t s_tok[2][kEcSlice];
  __shared__ float scratch[66];
  ec_slice_phase(T, C, L, gridDim.x, blockIdx.y, blockIdx.x, pos, ckey, ctok, stats, s_key, s_tok,
                 scratch);
}

__global__ void __launch_bounds__(kEcRankThreads)
    ec_rank_kernel(int T, int E, int C, int L, const uint32_t* __restrict__ ckey,
                   const int32_t* __restrict__ ctok, const float2* __restrict__ stats,
                   int stage_smem, int32_t* __restrict__ ec_idx, float* __restrict__ ec_score,
                   int32_t* __restrict__ pos) {
  pdl_begin();
  extern __shared__ __align__(16) unsigned char ec_smem[];
  __shared__ float s_mi[2];
  __shared__ int s_cnt[kEcRankThreads];
  ec_rank_phase(T, C, L, gridDim.x, blockIdx.y, blockIdx.x, ckey, ctok, stats, stage_smem,
                reinterpret_cast<uint32_t*>(ec_smem), ec_idx, ec_score, pos, s_mi, s_cnt);
}

// Both stages in one cooperative launch (every CTA resident): after its stage 1
// a CTA counts itself in arrive[e] and waits, bounded, until all S slices of its
// expert have posted, then runs stage 2.  arrive must be zero on entry.  A wait
// that gives up records kErrEcWait and skips stage 2.
constexpr uint32_t kErrEcWait = 16u;
constexpr uint64_t kEcWaitTimeoutNs = 1000000000ull;

__global__ void __launch_bounds__(kEcSlice)
    ec_select_kernel(int T, int E, int C, int L, int32_t* __restrict__ pos,
                     uint32_t* __restrict__ ckey, int32_t* __restrict__ ctok,
                     float2* __restrict__ stats, int stage_smem, int32_t* __restrict__ ec_idx,
                     float* __restrict__ ec_score, int* __restrict__ arrive) {
  pdl_begin();
  extern __shared__ __align__(16) unsigned char ec_smem[];
  __shared__ uint32_t s_key[2][kEcSlice];
  __shared__ int32_t s_tok[2][kEcSlice];
  __shared__ float scratch[66];
  __shared__ float s_mi[2];
  __shared__ int s_ok;
  __shared__ int s_cnt[kEcSlice];
  const int e = blockIdx.y, sl = blockIdx.x, S = gridDim.x;
  ec_slice_phase(T, C, L, S, e, sl, pos, ckey, ctok, stats, s_key, s_tok, scratch);
  if (C <= 0) return;
  __threadfence();  // this CTA's list, pair and pos entries before its arrival
  __syncthreads();
  if (threadIdx.x == 0) {
    atomicAdd(arrive + e, 1);
    volatile int* a = arrive + e;
    int ok = 1;
    const uint64_t t0 = global_timer_ns();
    while (*a < S) {
      if (global_timer_ns() - t0 > kEcWaitTimeoutNs) {
        record_error(kErrEcWait);
        ok = 0;
        break;
      }
    }
    __threadfence();
    s_ok = ok;
  }
  __syncthreads();
  if (!s_ok) return;
  ec_rank_phase(T, C, L, S, e, sl, ckey, ctok, stats, stage_smem,
                reinterpret_cast<uint32_t*>(ec_smem), ec_idx, ec_score, pos, s_mi, s_cnt);
}

// Stage 1 and stage 2 on the logits already transposed into pos ([E, T], fp32
// bits).  scratch: ec_scratch_bytes(T, E, C) bytes, 256-byte aligned.  One
// cooperative launch when the E * S CTAs fit on the GPU at once, else the two
// stages as two launches.
// arrive_fill: the byte the arrival counts start from (0; the bounded-wait
// self-test starts them far below zero, 0x80 bytes, so that no expert's slices
// ever all arrive).  one_launch_only: return cudaErrorNotSupported instead of
// taking the two-launch form.
inline cudaError_t launch_ec_select(int T, int E, int C, int32_t* ec_idx, float* ec_score,
                                    int32_t* pos, void* scratch, cudaStream_t s,
                                    int arrive_fill = 0, bool one_launch_only = false) {
  const int S = ec_slices(T), L = ec_list_len(C > 0 ? C : 1);
  char* base = static_cast<char*>(scratch);
  const size_t list_region = ec_align256((size_t)E * S * L * 4);
  uint32_t* ckey = reinterpret_cast<uint32_t*>(base);
  int32_t* ctok = reinterpret_cast<int32_t*>(base + list_region);
  float2* stats = reinterpret_cast<float2*>(base + 2 * list_region);
  int* arrive = reinterpret_cast<int*>(base + 2 * list_region + ec_align256((size_t)E * S * 8));
  const size_t lists_bytes = (size_t)S * L * 4;
  const int stage = (size_t)S * L <= kEcStageKeysMax && lists_bytes <= kEcRankSmemMax ? 1 : 0;
  const size_t sm = stage ? lists_bytes : 0;
  if (C > 0 && !ec_two_launches()) {
    cudaError_t err = cudaFuncSetAttribute(ec_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)kEcRankSmemMax);
    if (err != cudaSuccess) return err;
    int per_sm = 0, dev = 0, sms = 0;
    if (cudaGetDevice(&dev) == cudaSuccess &&
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess &&
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, ec_select_kernel, kEcSlice, sm) ==
            cudaSuccess &&
        (long long)per_sm * sms >= (long long)S * E) {
      err = cudaMemsetAsync(arrive, arrive_fill, (size_t)E * sizeof(int), s);
      if (err != cudaSuccess) return err;
      cudaLaunchAttribute coop;
      coop.id = cudaLaunchAttributeCooperative;
      coop.val.cooperative = 1;
      err = launch_k(ec_select_kernel, dim3(S, E), dim3(kEcSlice), sm, s, &coop, 1, T, E, C, L, pos,
                     ckey, ctok, stats, stage, ec_idx, ec_score, arrive);
      if (err == cudaSuccess || one_launch_only) return err;
      (void)cudaGetLastError();  // not launched: take the two-launch form
    }
  }
  if (one_launch_only) return cudaErrorNotSupported;
  cudaError_t err = launch_k(ec_slice_kernel, dim3(S, E), dim3(kEcSlice), 0, s, nullptr, 0, T, E, C,
                             L, pos, ckey, ctok, stats);
  if (err != cudaSuccess || C <= 0) return err;
  err = cudaFuncSetAttribute(ec_rank_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kEcRankSmemMax);
  if (err != cudaSuccess) return err;
  return launch_k(ec_rank_kernel, dim3(S, E), dim3(kEcRankThreads), sm, s, nullptr, 0, T, E, C, L,
                  (const uint32_t*)ckey, (const int32_t*)ctok, (const float2*)stats, stage, ec_idx,
                  ec_score, pos);
}

}  // namespace moe
