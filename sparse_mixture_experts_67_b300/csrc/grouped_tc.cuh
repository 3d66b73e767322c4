// Grouped bf16 expert GEMMs on the 5th-generation tensor cores (sm_103a).
//
// The SwiGLU expert of "Mixture of Experts（MoE）の理論と実装" (Expert.forward)
// and "Sparse Mixture of Experts(MoE) 아키텍처 심층 분석" (SwiGLUExpert):
//   gate/up:  H = silu(X_e W_gate,e^T) * (X_e W_up,e^T)   (bf16 out)
//   down:     Y = H_e W_down,e^T                          (fp32 out)
// over the variable-size expert segments [offsets[e], offsets[e+1]) of the
// dispatched rows.  The segment sizes stay on the device.
//
// One persistent CTA per SM, 6 warps:
//   warp 0     TMA producer (one thread): A tile [128 x 64] of the rows and the
//              B tile [256 x 64] of the weights per k-block into a 4-stage
//              ring (128-byte swizzle), completion on mbarriers;
//   warp 1     allocates all 512 TMEM columns; one thread issues
//              tcgen05.mma kind::f16 (M=128, N=256, K=16, fp32 accumulate)
//              into one of two TMEM accumulators and commits to mbarriers;
//   warps 2-5  epilogue: tcgen05.ld of the accumulator (thread = row), SwiGLU
//              or plain fp32, transposed through shared memory and stored as
//              whole row segments, masked at the segment end.
// For gate/up the B tile stacks 128 rows of W_gate over the same 128 rows of
// W_up, so one N=256 instruction produces both halves of the SwiGLU.
// Tiles are (expert, n-block, 128-row block), enumerated on the device from
// the offsets with the row block fastest; CTAs stride over them.  Every barrier wait is bounded in time:
// on expiry the kernel records a code in the device error word, drains its
// in-flight copies and MMAs, frees TMEM and returns.
#pragma once

#include <cuda.h>

#include <stdlib.h>

#include <algorithm>

#include "common.cuh"

namespace moe {
namespace tc {

constexpr int BM = 128, BK = 64;
constexpr int kThreads = 192;
constexpr int A_BYTES = BM * BK * 2;  // 16 KiB
constexpr uint64_t kWaitTimeoutNs = 1000000000ull;
// error-word codes
constexpr uint32_t kErrProducer = 1u, kErrMma = 2u, kErrEpilogue = 4u, kErrDrain = 8u;

// Per-width constants: BN is the MMA N (output columns for down; gate + up
// halves for gate/up).  Narrow tiles leave room for more stages in flight.
// PAIR: 2-CTA MMA, where each CTA holds only its half (BN / 2 rows) of the B tile.
template <int BN, bool PAIR = false>
struct Cfg {
  static constexpr int B_BYTES = (PAIR ? BN / 2 : BN) * BK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int STAGES = (192 * 1024) / STAGE_BYTES > 8 ? 8 : (192 * 1024) / STAGE_BYTES;
  static constexpr uint32_t TMEM_COLS = 2 * BN < 32 ? 32 : 2 * BN;  // two accumulators
};

constexpr int kStagePitch = 36;  // floats per row of an epilogue warp's 32 x 32 staging tile

template <int STAGES>
struct Smem {  // lives after the 1024-aligned stage ring
  // per epilogue warp: a 32-row chunk of the accumulator, transposed through
  // shared memory so that global stores cover whole row segments
  alignas(16) float stage_out[4][32 * kStagePitch];
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
  uint64_t tmem_full[2];
  uint64_t tmem_empty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
  int cum[MOE_MAX_EXPERTS + 1];  // prefix of 128-row blocks per expert
  int off[MOE_MAX_EXPERTS + 1];  // segment offsets
};

template <int BN, bool PAIR = false>
constexpr size_t smem_bytes() {
  using C = Cfg<BN, PAIR>;
  return (size_t)C::STAGES * C::STAGE_BYTES + sizeof(Smem<C::STAGES>) + 1024;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

// The waits pass a suspend-time hint of 1 ms: a waiting thread sleeps until
// the phase completes (or the hint expires) instead of re-polling the barrier.
// Polling at the default limit cost shared-memory bandwidth that the tensor
// cores' operand reads need (gate/up GEMM 168 -> 157 us on top2_d1024).
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, 1000000;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Without the hint: the wait returns at the hardware's default limit, for
// latency-critical chains of short waits.
__device__ __forceinline__ bool mbar_try_wait_short(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// As mbar_try_wait, acquiring at cluster scope (arrivals made by the peer CTA).
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, "
      "1000000;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Waits for the phase of `parity` to complete.  Gives up (false) when the
// CTA's abort flag is raised or after kWaitTimeoutNs, recording `code`.
template <bool CLUSTER_SCOPE = false, bool SHORT = false>
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                          uint32_t code) {
  const uint32_t a = smem_u32(bar);
  auto ready = [&]() {
    return CLUSTER_SCOPE ? mbar_try_wait_cluster(a, parity)
                         : (SHORT ? mbar_try_wait_short(a, parity) : mbar_try_wait(a, parity));
  };
  if (ready()) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (ready()) return true;
    if (*abort_flag) return false;
    if (global_timer_ns() - t0 > kWaitTimeoutNs) {
      record_error(code);
      *abort_flag = 1;
      return false;
    }
  }
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Address, in the cluster's shared window, of this CTA's variable `saddr`
// as placed in the CTA of cluster rank `rank`.
__device__ __forceinline__ uint32_t cluster_addr(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}

// Arrive on an mbarrier of another CTA of the cluster (release at cluster scope).
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_bar) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_bar)
               : "memory");
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar, int x,
                                            int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, "
      "%3}], [%4];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

// Four rows r0..r3 (64 columns from x) of a 2-D tensor whose map has a
// one-row box, written as four consecutive 128-byte rows at dst.
__device__ __forceinline__ void tma_gather4(void* dst, const CUtensorMap* map, uint64_t* bar, int x,
                                            int r0, int r1, int r2, int r3) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(r0), "r"(r1), "r"(r2), "r"(r3),
      "r"(smem_u32(bar))
      : "memory");
}

// 2-CTA form: the completion is signalled on `cluster_bar`, which may be the
// mbarrier of either CTA of the pair (here always the pair's rank-0 CTA).
__device__ __forceinline__ void tma_load_2d_pair(void* dst, const CUtensorMap* map, uint32_t cluster_bar,
                                                 int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.cta_group::2 "
      "[%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(cluster_bar)
      : "memory");
}

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void tc_mma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                           uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Pair forms (cta_group::2), issued by the pair's rank-0 CTA.  One MMA of
// M = 256 reads A rows 0-127 from this CTA's shared memory and rows 128-255
// from the peer's (same offset), the first and second halves of B's N rows
// likewise, and writes each CTA's 128 rows of D into that CTA's TMEM.
__device__ __forceinline__ void tc_mma_f16_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                                uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive on the mbarrier at this offset in each CTA of cta_mask once the
// pair's issued MMAs complete (a completion signal; it moves no data).
__device__ __forceinline__ void tc_commit_pair(uint64_t* bar, uint16_t cta_mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 "
      "[%0], %1;" ::"r"(smem_u32(bar)),
      "h"(cta_mask)
      : "memory");
}

// Shared-memory matrix descriptor: K-major tile with 128-byte rows in the
// 128-byte swizzle (8-row atoms of 1024 bytes, stride byte offset 1024).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFFu);  // start address
  d |= (uint64_t)1u << 16;                  // leading byte offset (unused for this layout)
  d |= (uint64_t)(1024u >> 4) << 32;        // stride byte offset: next 8-row group
  d |= (uint64_t)1u << 46;                  // descriptor version
  d |= (uint64_t)2u << 61;                  // 128-byte swizzle
  return d;
}

// Instruction descriptor, kind::f16: fp32 accumulator, bf16 A and B, both K-major.
__host__ __device__ constexpr uint32_t make_idesc_bf16(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

#define MOE_TMEM_LD32(taddr, r)                                                                   \
  asm volatile(                                                                                   \
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14," \
      "%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"              \
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),       \
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),   \
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),            \
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),            \
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])             \
      : "r"(taddr))

// 16 TMEM lanes x 8 repetitions of 256 bits: thread i gets, for repetition j
// (columns 8j .. 8j+7), r[4j], r[4j+1] = lane i/4, columns 8j + 2(i%4) + {0,1}
// and r[4j+2], r[4j+3] = lane i/4 + 8, the same columns (the layout of an
// m16n8 accumulator fragment, repeated along the columns).
#define MOE_TMEM_LD16x256_X8(taddr, r)                                                             \
  asm volatile(                                                                                   \
      "tcgen05.ld.sync.aligned.16x256b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14," \
      "%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"              \
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),       \
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),   \
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),            \
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),            \
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])             \
      : "r"(taddr))

__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

struct TileCoord {
  int e, row0, row_end, nt;
};

// Tiles are enumerated expert by expert.  Inside an expert the row blocks go
// in groups of `group` (0: one group of all of them); inside a group the row
// block varies fastest and the n-block slowest, so the CTAs of one wave share
// each weight tile (read from HBM once) while the group's rows stay in L2.
template <class SmemT>
__device__ __forceinline__ TileCoord map_tile(const SmemT& S, int E, int n_tiles, int tile,
                                              int unit_rows = BM, int group = 0) {
  TileCoord c;
  int lo = 0, hi = E;  // S.cum[lo] * n_tiles <= tile < S.cum[hi] * n_tiles
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (S.cum[mid] * n_tiles <= tile) lo = mid;
    else hi = mid;
  }
  const int m_tiles = S.cum[lo + 1] - S.cum[lo];
  const int local = tile - S.cum[lo] * n_tiles;
  int g0 = 0, gs = m_tiles;  // the group's first row block and its row blocks
  if (group > 0 && m_tiles > group) {
    g0 = min(local / (group * n_tiles), (m_tiles - 1) / group) * group;
    gs = min(group, m_tiles - g0);
  }
  const int in = local - g0 * n_tiles;
  const int nt = in / gs;
  c.e = lo;
  c.nt = nt;
  c.row0 = S.off[lo] + (g0 + in - nt * gs) * unit_rows;
  c.row_end = S.off[lo + 1];
  return c;
}

__device__ __forceinline__ float silu_fast(float a) { return __fdividef(a, 1.0f + __expf(-a)); }

// y[addr..addr+3] += v (a relaxed float4 reduction, as atomicAdd on float4),
// with an L2 policy: evict_last keeps y's lines in L2 between the additions of
// a token's two slots, which come from units of different experts.
__device__ __forceinline__ uint64_t l2_evict_last_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
__device__ __forceinline__ void red_add_f4_hint(float* addr, float4 v, uint64_t pol) {
  asm volatile("red.global.add.L2::cache_hint.v4.f32 [%0], {%1, %2, %3, %4}, %5;" ::"l"(addr),
               "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w), "l"(pol)
               : "memory");
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// GATEUP: out = bf16 H [R, N] (N = F), B rows from two maps (gate, up), BN/2 each.
// !GATEUP: out = fp32 Y [R, N] (N = d), B rows from one map, BN per tile.
// COMBINE (down only): instead of Y, row r adds topk_w[a] * Y[r,:] into
// out = y [T, N] (zeroed beforehand) at token a / kslots, a = perm[r], with
// float4 atomics.  With kslots <= 2 every element of y receives at most two
// additions onto zero, so the sum is the same in either order: deterministic.
// GATHER (gate/up only): row r of A is row gsrc[r] / gdiv of the tensor behind
// tmA (x itself, mapped with a one-row box) instead of row r; each producer
// lane brings 4 of the tile's 128 rows per k-block with one TMA gather4.
// PAIR: launched in clusters of 2 as one 2-CTA MMA unit (tcgen05 cta_group::2)
// over 256-row blocks.  Each CTA loads its own 128 A rows and its half of the
// B tile (gate/up: rank 0 the gate rows, rank 1 the up rows), signalling the
// full barrier of the rank-0 CTA, whose single thread issues M = 256 MMAs and
// commits to the empty / accumulator-full barriers of both CTAs.  Each CTA's
// epilogue drains its own TMEM rows and arrives on rank 0's accumulator-empty
// barrier (4 warps x 2 CTAs).  Per SM this moves 32 KiB instead of 48 KiB of
// operands into shared memory per k-block for the same 128 x 256 outputs.
// PAIRING: 0 single CTA, 2 PAIR.
template <bool GATEUP, int BN, bool COMBINE = false, bool GATHER = false, int PAIRING = 0>
__global__ void __launch_bounds__(kThreads, 1)
    grouped_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB0,
                      const __grid_constant__ CUtensorMap tmB1, const int32_t* __restrict__ offsets,
                      int R, int E, int N, int K, void* __restrict__ out,
                      const int32_t* __restrict__ perm = nullptr,
                      const float* __restrict__ topk_w = nullptr, int kslots = 1,
                      const __nv_bfloat16* __restrict__ gx = nullptr,
                      const int32_t* __restrict__ gsrc = nullptr, int gdiv = 1,
                      int frag_store = 0, int y_keep = 0) {
  static_assert(PAIRING == 0 || PAIRING == 2, "single CTA or 2-CTA pair");
  constexpr bool PAIR = PAIRING == 2, CL = PAIR;
  static_assert(!(PAIR && (GATHER || BN != 256)), "2-CTA MMA: 256-wide tiles without gather");
  using C = Cfg<BN, PAIR>;
  constexpr int STAGES = C::STAGES;
  constexpr int STAGE_BYTES = C::STAGE_BYTES;
  constexpr int B_BYTES = C::B_BYTES;
  constexpr uint32_t TMEM_COLS = C::TMEM_COLS;
  using SmemT = Smem<STAGES>;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* ring = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  SmemT& S = *reinterpret_cast<SmemT*>(ring + (size_t)STAGES * STAGE_BYTES);
  volatile int* abort_flag = &S.abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr int kTileN = GATEUP ? BN / 2 : BN;  // output columns per tile
  constexpr int kUnitRows = CL ? 2 * BM : BM;  // rows of one work unit (a cluster's)
  constexpr int kGroup = GATEUP ? 0 : 8;  // row blocks per raster group (down: 8)
  const uint32_t crank = CL ? cluster_ctarank() : 0u;
  const int unit0 = CL ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
  const int ustride = CL ? (int)(gridDim.x >> 1) : (int)gridDim.x;
  constexpr uint16_t kPair = 0x3;
  const int n_tiles = (N + kTileN - 1) / kTileN;
  const int num_kb = K / BK;

  // --- setup (barriers and TMEM first: this part may overlap the previous kernel)
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&S.full[s], 1);
      mbar_init(&S.empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&S.tmem_full[b], 1);
      mbar_init(&S.tmem_empty[b], PAIR ? 8 : 128);  // PAIR: one arrival per epilogue warp of both CTAs
    }
    mbar_init(&S.drain, 1);
    S.abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    prefetch_tensormap(&tmA);
    prefetch_tensormap(&tmB0);
    if (GATEUP) prefetch_tensormap(&tmB1);
  }
  if (warp == 1) {
    if (PAIR) {  // collective with the peer CTA's warp 1
      asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                       smem_u32(&S.tmem_base)),
                   "r"(TMEM_COLS)
                   : "memory");
      asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    } else {
      asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                       smem_u32(&S.tmem_base)),
                   "r"(TMEM_COLS)
                   : "memory");
      asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
  }
  pdl_begin();  // the segment offsets come from the previous kernel
  for (int i = threadIdx.x; i <= E; i += blockDim.x) S.off[i] = min(max(offsets[i], 0), R);
  __syncthreads();
  if (threadIdx.x == 0) {
    int cum = 0;
    for (int e = 0; e < E; ++e) {
      S.cum[e] = cum;
      const int cnt = max(S.off[e + 1] - S.off[e], 0);
      cum += (cnt + kUnitRows - 1) / kUnitRows;
    }
    S.cum[E] = cum;
  }
  tc_fence_before();
  __syncthreads();
  if (CL) cluster_sync_all();  // the peer's barriers are initialised before any remote signal
  tc_fence_after();
  const uint32_t tmem_base = S.tmem_base;
  // Work units.  A down launch whose last wave would be partly empty splits each
  // tile of that wave into two 128-column halves (N = 128 MMAs on the first half
  // of the loaded B tile), so the wave takes half as long.
  const int total_tiles = S.cum[E] * n_tiles;
  int full_units = total_tiles, split_tiles = 0;
  if (!GATEUP && BN == 256) {
    const int rem = total_tiles % ustride;
    if (rem > 0 && 2 * rem <= ustride) {
      full_units = total_tiles - rem;
      split_tiles = rem;
    }
  }
  const int total = full_units + 2 * split_tiles;
  // unit -> tile coordinates, first output column inside the tile, column count
  auto unit_at = [&](int u, TileCoord& c, int& col_off, int& width) {
    if (u < full_units) {
      // down: the last experts first, whose H rows the gate/up kernel wrote last
      // (still in L2 when this kernel starts)
      c = map_tile(S, E, n_tiles, GATEUP ? u : full_units - 1 - u, kUnitRows, kGroup);
      c.row0 += (int)crank * BM;  // this CTA's half of the cluster's rows
      col_off = 0;
      width = kTileN;
    } else {
      const int v = u - full_units;
      c = map_tile(S, E, n_tiles, full_units + (v >> 1), kUnitRows, kGroup);
      c.row0 += (int)crank * BM;
      col_off = (v & 1) * (kTileN / 2);
      width = kTileN / 2;
    }
  };

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (GATHER || lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued = 0, issued_phase = 0;  // per-stage bits: loads issued, their parity
      for (int tile = unit0; tile < total && !*abort_flag; tile += ustride) {
        TileCoord c;
        int col_off, width;
        unit_at(tile, c, col_off, width);
        const int brow = c.e * N + c.nt * kTileN + col_off;
        int tok[4] = {0, 0, 0, 0};  // GATHER: source rows of tile rows 4 * lane + i
        if (GATHER) {               // (rows past the segment read row 0; never stored)
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int r = c.row0 + 4 * lane + i;
            tok[i] = r < c.row_end ? gsrc[r] / gdiv : 0;
          }
        }
        bool ok = true;
        for (int kb = 0; kb < num_kb; ++kb) {
          int go = 1;
          if (lane == 0) go = mbar_wait(&S.empty[stage], phase ^ 1u, abort_flag, kErrProducer);
          if (GATHER) go = __shfl_sync(kFullMask, go, 0);
          if (!go) {
            ok = false;
            break;
          }
          unsigned char* sA = ring + (size_t)stage * STAGE_BYTES;
          unsigned char* sB = sA + A_BYTES;
          // a half unit of the down GEMM loads only the 128 B rows it uses (tmB1)
          const bool half_unit = !GATEUP && tile >= full_units;
          if (PAIR) {
            // both CTAs' loads land on rank 0's full barrier, which expects them all
            if (lane == 0) {
              const uint32_t fb = cluster_addr(smem_u32(&S.full[stage]), 0);
              if (crank == 0)
                mbar_arrive_expect_tx(&S.full[stage],
                                      2 * (half_unit ? STAGE_BYTES - B_BYTES / 2 : STAGE_BYTES));
              tma_load_2d_pair(sA, &tmA, fb, kb * BK, c.row0);
              if (half_unit)  // down, 128-column half: 64 B rows per CTA (tmB0 has a 64-row box)
                tma_load_2d_pair(sB, &tmB0, fb, kb * BK, brow + (int)crank * (BN / 4));
              else
                tma_load_2d_pair(sB, GATEUP && crank == 0 ? &tmB0 : &tmB1, fb, kb * BK,
                                 GATEUP ? brow : brow + (int)crank * (BN / 2));
            }
          } else if (lane == 0) {
            mbar_arrive_expect_tx(&S.full[stage], half_unit ? STAGE_BYTES - B_BYTES / 2 : STAGE_BYTES);
          }
          if (GATHER) {
            __syncwarp();  // the expected byte count is set before any gather lands
            tma_gather4(sA + lane * 4 * 128, &tmA, &S.full[stage], kb * BK, tok[0], tok[1], tok[2],
                        tok[3]);
          }
          if (lane == 0 && !PAIR) {
            if (!GATHER) tma_load_2d(sA, &tmA, &S.full[stage], kb * BK, c.row0);
            if (GATEUP) {
              tma_load_2d(sB, &tmB0, &S.full[stage], kb * BK, brow);
              tma_load_2d(sB + B_BYTES / 2, &tmB1, &S.full[stage], kb * BK, brow);
            } else {
              tma_load_2d(sB, half_unit ? &tmB1 : &tmB0, &S.full[stage], kb * BK, brow);
            }
          }
          issued |= 1u << stage;
          issued_phase = (issued_phase & ~(1u << stage)) | (phase << stage);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
      }
      // drain: every issued load must have landed before the CTA may exit.
      // PAIR, rank 1: its loads complete on rank 0's barriers, which it cannot
      // poll; on the normal path rank 0's MMAs consumed them all before the
      // closing cluster barrier.  After an abort it leaves them time to land.
      if (PAIR && crank != 0) {
        if (lane == 0 && *abort_flag) {
          const uint64_t t0 = global_timer_ns();
          while (global_timer_ns() - t0 < 200000ull) {
          }
        }
      } else if (lane == 0) {
        for (int s = 0; s < STAGES; ++s) {
          if (!((issued >> s) & 1u)) continue;
          const uint32_t a = smem_u32(&S.full[s]);
          const uint32_t par = (issued_phase >> s) & 1u;
          const uint64_t t0 = global_timer_ns();
          while (!mbar_try_wait(a, par)) {
            if (global_timer_ns() - t0 > kWaitTimeoutNs) {
              record_error(kErrDrain);
              break;
            }
          }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // (PAIR: rank 0 only; rank 1's warp 1 just holds its TMEM allocation)
    if (lane == 0 && (!PAIR || crank == 0)) {
      constexpr uint32_t idesc_full = make_idesc_bf16(PAIR ? 2 * BM : BM, BN);
      constexpr uint32_t idesc_half = make_idesc_bf16(PAIR ? 2 * BM : BM, BN / 2);
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      for (int tile = unit0; tile < total && !*abort_flag; tile += ustride) {
        const uint32_t idesc = tile < full_units ? idesc_full : idesc_half;
        if (!mbar_wait<PAIR>(&S.tmem_empty[acc], acc_phase ^ 1u, abort_flag, kErrMma)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
        bool ok = true;
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!mbar_wait(&S.full[stage], phase, abort_flag, kErrMma)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = smem_u32(ring + (size_t)stage * STAGE_BYTES);
          const uint32_t b0 = a0 + A_BYTES;
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            if (PAIR)
              tc_mma_f16_pair(d_tmem, sw128_desc(a0 + kk * 32), sw128_desc(b0 + kk * 32), idesc,
                              (kb | kk) != 0 ? 1u : 0u);
            else
              tc_mma_f16(d_tmem, sw128_desc(a0 + kk * 32), sw128_desc(b0 + kk * 32), idesc,
                         (kb | kk) != 0 ? 1u : 0u);
          }
          // frees the smem stage once these MMAs finish (in both CTAs when paired)
          if (PAIR) tc_commit_pair(&S.empty[stage], kPair);
          else tc_commit(&S.empty[stage]);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        if (PAIR) tc_commit_pair(&S.tmem_full[acc], kPair);
        else tc_commit(&S.tmem_full[acc]);
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      // drain: all issued MMAs complete before TMEM is released
      if (PAIR) tc_commit_pair(&S.drain, 0x1);
      else tc_commit(&S.drain);
      const uint32_t a = smem_u32(&S.drain);
      const uint64_t t0 = global_timer_ns();
      while (!mbar_try_wait(a, 0)) {
        if (global_timer_ns() - t0 > kWaitTimeoutNs) {
          record_error(kErrDrain);
          break;
        }
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    // Each warp owns TMEM lane quarter q (tile rows 32q .. 32q+31, thread = row
    // when reading TMEM).  A chunk of columns goes through the warp's staging
    // tile in shared memory and leaves as whole row segments (4-8 rows per store
    // instruction instead of 32 scattered 16-byte pieces): 64 bf16 columns
    // (128-byte rows, 16-byte pieces XOR-swizzled by row) for H, 32 fp32 columns
    // (rows padded to 144 bytes) for Y.  Both staging patterns are free of bank
    // conflicts.
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    float* stg = S.stage_out[q];
    uint32_t* stg_w = reinterpret_cast<uint32_t*>(stg);
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int tile = unit0; tile < total; tile += ustride) {
      TileCoord c;
      int col_off, width;
      unit_at(tile, c, col_off, width);
      if (!mbar_wait(&S.tmem_full[acc], acc_phase, abort_flag, kErrEpilogue)) break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + (uint32_t)(acc * BN) + ((uint32_t)(q * 32) << 16);
      const int rbase = c.row0 + q * 32;  // row of lane 0
      const int row = rbase + lane;
      const bool valid = row < c.row_end;
      const int n0 = c.nt * kTileN + col_off;
      if (GATEUP) {
        __nv_bfloat16* H = static_cast<__nv_bfloat16*>(out);
        constexpr int kCh = kTileN >= 64 ? 64 : 32;  // columns per staged chunk
        uint4* stg16 = reinterpret_cast<uint4*>(stg_w);  // 32 rows x 8 pieces of 16 bytes
#pragma unroll 1
        for (int c0 = 0; c0 < kTileN; c0 += kCh) {
#pragma unroll 1
          for (int cc = c0; cc < c0 + kCh; cc += 32) {
            uint32_t g[32], u[32];
            MOE_TMEM_LD32(taddr + cc, g);
            MOE_TMEM_LD32(taddr + kTileN + cc, u);
            tmem_ld_wait();
            uint32_t p[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const float h0 = silu_fast(__uint_as_float(g[2 * i])) * __uint_as_float(u[2 * i]);
              const float h1 = silu_fast(__uint_as_float(g[2 * i + 1])) * __uint_as_float(u[2 * i + 1]);
              p[i] = pack_bf16x2(h0, h1);
            }
            // row `lane`, pieces (cc - c0) / 8 + i, stored at piece ^ (row & 7)
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int piece = ((cc - c0) >> 3) + i;
              stg16[lane * 8 + (piece ^ (lane & 7))] =
                  make_uint4(p[4 * i], p[4 * i + 1], p[4 * i + 2], p[4 * i + 3]);
            }
          }
          __syncwarp();
          if (n0 + c0 < N) {
            constexpr int kLanesPerRow = kCh / 8, kRowsPerStore = 32 / kLanesPerRow;
#pragma unroll
            for (int j = 0; j < 32 / kRowsPerStore; ++j) {
              const int r = j * kRowsPerStore + lane / kLanesPerRow, part = lane % kLanesPerRow;
              const int grow = rbase + r;
              if (grow < c.row_end)
                *reinterpret_cast<uint4*>(H + (size_t)grow * N + n0 + c0 + part * 8) =
                    stg16[r * 8 + (part ^ (r & 7))];
            }
          }
          __syncwarp();
        }
      } else {
        // COMBINE: this row's token and routing weight, shuffled to the storing lanes
        const int a = (COMBINE && valid) ? perm[row] : 0;
        const float wgt = (COMBINE && valid) ? topk_w[a] : 0.f;
        const int tok = a / kslots;
        float* Y = static_cast<float*>(out);
        const uint64_t ypol = (COMBINE && y_keep) ? l2_evict_last_policy() : 0ull;
        // plain stores go straight from the fragments, the combine's atomics through
        // the staging (float4 additions covering four rows each measured faster)
        const bool use_frag = frag_store == 2 ? !COMBINE : frag_store == 1;
        if (use_frag) {
          // straight from the 16x256b fragments: four lanes store one row's 32
          // contiguous bytes per instruction (whole sectors), no shared memory
#pragma unroll 1
          for (int hh = 0; hh < 2; ++hh) {  // the warp's two 16-row halves
            const int rl0 = hh * 16 + (lane >> 2), rl1 = rl0 + 8;  // rows within the warp's 32
            const int g0 = rbase + rl0, g1 = rbase + rl1;
            const int t0 = __shfl_sync(kFullMask, tok, rl0), t1 = __shfl_sync(kFullMask, tok, rl1);
            const float w0 = __shfl_sync(kFullMask, wgt, rl0), w1 = __shfl_sync(kFullMask, wgt, rl1);
            const bool v0 = g0 < c.row_end, v1 = g1 < c.row_end;
            const uint32_t tq = taddr + ((uint32_t)(hh * 16) << 16);
#pragma unroll 1
            for (int cc = 0; cc < width; cc += 64) {
              uint32_t v[32];
              MOE_TMEM_LD16x256_X8(tq + cc, v);
              tmem_ld_wait();
              if (n0 + cc < N) {
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                  const int col = n0 + cc + 8 * j + 2 * (lane & 3);
                  const float2 a0 = make_float2(__uint_as_float(v[4 * j]), __uint_as_float(v[4 * j + 1]));
                  const float2 a1 = make_float2(__uint_as_float(v[4 * j + 2]), __uint_as_float(v[4 * j + 3]));
                  if (COMBINE) {
                    if (v0) atomicAdd(reinterpret_cast<float2*>(Y + (size_t)t0 * N + col),
                                      make_float2(w0 * a0.x, w0 * a0.y));
                    if (v1) atomicAdd(reinterpret_cast<float2*>(Y + (size_t)t1 * N + col),
                                      make_float2(w1 * a1.x, w1 * a1.y));
                  } else {
                    if (v0) *reinterpret_cast<float2*>(Y + (size_t)g0 * N + col) = a0;
                    if (v1) *reinterpret_cast<float2*>(Y + (size_t)g1 * N + col) = a1;
                  }
                }
              }
            }
          }
        } else
#pragma unroll 1
        for (int cc = 0; cc < width; cc += 32) {
          uint32_t v[32];
          MOE_TMEM_LD32(taddr + cc, v);
          tmem_ld_wait();
          float4* srow = reinterpret_cast<float4*>(stg + lane * kStagePitch);
#pragma unroll
          for (int i = 0; i < 8; ++i)
            srow[i] = make_float4(__uint_as_float(v[4 * i]), __uint_as_float(v[4 * i + 1]),
                                  __uint_as_float(v[4 * i + 2]), __uint_as_float(v[4 * i + 3]));
          __syncwarp();
          if (n0 + cc < N) {  // 8 lanes per row, 4 rows per store
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const int r = j * 4 + (lane >> 3), part = lane & 7;
              const int grow = rbase + r;
              const float4 val = *reinterpret_cast<const float4*>(stg + r * kStagePitch + part * 4);
              if (COMBINE) {
                const int rt = __shfl_sync(kFullMask, tok, r);
                const float rw = __shfl_sync(kFullMask, wgt, r);
                if (grow < c.row_end) {
                  float* ya = Y + (size_t)rt * N + n0 + cc + part * 4;
                  const float4 add = make_float4(rw * val.x, rw * val.y, rw * val.z, rw * val.w);
                  if (y_keep) red_add_f4_hint(ya, add, ypol);
                  else atomicAdd(reinterpret_cast<float4*>(ya), add);
                }
              } else if (grow < c.row_end) {
                *reinterpret_cast<float4*>(Y + (size_t)grow * N + n0 + cc + part * 4) = val;
              }
            }
          }
          __syncwarp();
        }
      }
      tc_fence_before();
      if (PAIR) {  // one arrival per warp, on rank 0's barrier
        __syncwarp();
        if (lane == 0) {
          if (crank == 0) mbar_arrive(&S.tmem_empty[acc]);
          else mbar_arrive_cluster(cluster_addr(smem_u32(&S.tmem_empty[acc]), 0));
        }
      } else {
        mbar_arrive(&S.tmem_empty[acc]);
      }
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (CL) cluster_sync_all();  // the peer no longer writes here or arrives on our barriers
  if (warp == 1) {
    tc_fence_after();
    if (PAIR)
      asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                   "r"(TMEM_COLS)
                   : "memory");
    else
      asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                   "r"(TMEM_COLS)
                   : "memory");
  }
}

// ------------------------------------------------------------------ host side

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// Row-major bf16 matrix [rows, cols] read in boxes of [box_rows, 64] with the
// 128-byte swizzle; out-of-range rows read as zero.
inline bool make_map(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 2};
  const cuuint32_t box[2] = {(cuuint32_t)BK, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// How the down GEMM's epilogue writes: 1 = straight from 16x256b TMEM fragments,
// 0 = through a shared-memory transpose into whole row segments, 2 = the first
// for plain stores of Y and the second for the fused combine's atomics
// (measured, whole layers alternating A/B: fine_e64 1001 against 1011 us;
// top2_d1024 297 against 293 us, large_d4096 at T=4096 2023 against 2014 us).
// MOE_DOWN_EPILOGUE in the environment ("frag", "staged") forces one.
inline int down_frag_store() {
  const char* v = getenv("MOE_DOWN_EPILOGUE");
  if (v && v[0] == 'f') return 1;
  if (v && v[0] == 's') return 0;
  return 2;
}

inline int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    return 148;
  return n;
}

template <bool GATEUP, int BN, bool COMBINE = false, bool GATHER = false>
cudaError_t launch_bn(const CUtensorMap& a, const CUtensorMap& b0, const CUtensorMap& b1,
                      const int32_t* offsets, int R, int E, int N, int K, void* out, int sms,
                      cudaStream_t s, const int32_t* perm = nullptr, const float* topk_w = nullptr,
                      int kslots = 1, const __nv_bfloat16* gx = nullptr,
                      const int32_t* gsrc = nullptr, int gdiv = 1) {
  constexpr size_t sm = smem_bytes<BN>();
  cudaError_t e = cudaFuncSetAttribute(grouped_tc_kernel<GATEUP, BN, COMBINE, GATHER>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
  if (e != cudaSuccess) return e;
  constexpr int tile_n = GATEUP ? BN / 2 : BN;
  const long long max_tiles = (long long)((R + BM - 1) / BM + E) * ((N + tile_n - 1) / tile_n);
  const int grid = (int)std::min<long long>(sms, max_tiles);
  return launch_k(grouped_tc_kernel<GATEUP, BN, COMBINE, GATHER>, dim3(grid), dim3(kThreads), sm, s,
                  nullptr, 0, a, b0, b1, offsets, R, E, N, K, out, perm, topk_w, kslots, gx, gsrc,
                  gdiv, down_frag_store(), 0);
}

// How 256-wide launches pair CTAs: 2 = 2-CTA MMA (PAIR, the default), 0 =
// single CTAs.  MOE_GROUPED_CLUSTER in the environment ("pair", "none")
// selects one (tests, A/B timing).
inline int cluster_mode() {
  const char* v = getenv("MOE_GROUPED_CLUSTER");
  if (!v || !*v) return 2;
  if (v[0] == 'n' || v[0] == '0') return 0;
  return 2;
}

// Cluster-of-2 launch of a 256-wide kernel as one 2-CTA MMA unit (PAIRING 2).  The grid is the
// number of clusters that fit at once (queried once per device and mode),
// capped by the work, times two.
template <bool GATEUP, bool COMBINE, int PAIRING>
cudaError_t launch_cluster(const CUtensorMap& a, const CUtensorMap& b0, const CUtensorMap& b1,
                           const int32_t* offsets, int R, int E, int N, int K, void* out,
                           cudaStream_t s, const int32_t* perm = nullptr,
                           const float* topk_w = nullptr, int kslots = 1, int y_keep = 0) {
  constexpr int BN = 256;
  constexpr size_t sm = smem_bytes<BN, PAIRING == 2>();
  auto kern = grouped_tc_kernel<GATEUP, BN, COMBINE, false, PAIRING>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = 2;
  attr.val.clusterDim.y = 1;
  attr.val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = sm;
  cfg.stream = s;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  static int max_clusters[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (max_clusters[dev] == 0) {
    cfg.gridDim = dim3(2 * 74, 1, 1);
    int n = 0;
    e = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
    if (e != cudaSuccess) return e;
    max_clusters[dev] = n > 0 ? n : 1;
  }
  constexpr int tile_n = GATEUP ? BN / 2 : BN;
  const long long units = (long long)((R + 2 * BM - 1) / (2 * BM) + E) * ((N + tile_n - 1) / tile_n);
  const int clusters = (int)std::min<long long>(max_clusters[dev], units);
  return launch_k(kern, dim3(2 * clusters), dim3(kThreads), sm, s, &attr, 1, a, b0, b1, offsets, R,
                  E, N, K, out, perm, topk_w, kslots, (const __nv_bfloat16*)nullptr,
                  (const int32_t*)nullptr, 1, down_frag_store(), y_keep);
}

template <bool GATEUP, bool COMBINE>
cudaError_t launch_paired(const CUtensorMap& a, const CUtensorMap& b0, const CUtensorMap& b1,
                          const int32_t* offsets, int R, int E, int N, int K, void* out,
                          cudaStream_t s, const int32_t* perm = nullptr,
                          const float* topk_w = nullptr, int kslots = 1, int y_keep = 0) {
  return launch_cluster<GATEUP, COMBINE, 2>(a, b0, b1, offsets, R, E, N, K, out, s, perm, topk_w, kslots,
                                            y_keep);
}

// MMA width for a launch.  256 everywhere it was measured best (both GEMMs
// when compute-bound, down always); gate/up with fewer than 256 rows per
// expert on average is weight-bandwidth-bound and uses 128-wide tiles, twice
// as many as 256-wide ones, for a better-filled last wave.
// MOE_GROUPED_TILE_N in the environment forces a width (used by the tests).
inline int choose_bn(int R, int E, int N, bool gateup, int sms) {
  if (const char* force = getenv("MOE_GROUPED_TILE_N")) {  // testing override: 64, 128 or 256
    const int v = atoi(force);
    if (v == 64 || v == 128 || v == 256) return v;
  }
  (void)N;
  (void)sms;
  if (gateup && (long long)R < 2LL * BM * E) return 128;
  return 256;
}

template <bool GATEUP>
cudaError_t launch(const CUtensorMap* maps_by_bn, int bn, const int32_t* offsets, int R, int E, int N,
                   int K, void* out, int sms, cudaStream_t s) {
  // maps_by_bn: {A, B0, B1} for the chosen width
  switch (bn) {
    case 64: return launch_bn<GATEUP, 64>(maps_by_bn[0], maps_by_bn[1], maps_by_bn[2], offsets, R, E, N, K, out, sms, s);
    case 128: return launch_bn<GATEUP, 128>(maps_by_bn[0], maps_by_bn[1], maps_by_bn[2], offsets, R, E, N, K, out, sms, s);
    default: return launch_bn<GATEUP, 256>(maps_by_bn[0], maps_by_bn[1], maps_by_bn[2], offsets, R, E, N, K, out, sms, s);
  }
}

}  // namespace tc

inline cudaError_t launch_gateup_tc(const __nv_bfloat16* x_perm, const int32_t* offsets,
                                    const __nv_bfloat16* w_gate, const __nv_bfloat16* w_up, int R,
                                    int d, int F, int E, __nv_bfloat16* h, cudaStream_t s) {
  const int sms = tc::sm_count();
  const int bn = tc::choose_bn(R, E, F, true, sms);
  CUtensorMap m[3];
  if (!tc::make_map(&m[0], x_perm, (uint64_t)R, (uint64_t)d, tc::BM) ||
      !tc::make_map(&m[1], w_gate, (uint64_t)E * F, (uint64_t)d, bn / 2) ||
      !tc::make_map(&m[2], w_up, (uint64_t)E * F, (uint64_t)d, bn / 2))
    return cudaErrorInvalidValue;
  if (bn == 256 && tc::cluster_mode() != 0)
    return tc::launch_paired<true, false>(m[0], m[1], m[2], offsets, R, E, F, d, h, s);
  return tc::launch<true>(m, bn, offsets, R, E, F, d, h, sms, s);
}

// Gate/up with the dispatch gather fused into the A load: row r of the
// segment-ordered A is x[src[r] / div] (src = perm with div = k for top-k,
// the expert-choice token ids with div = 1); x_perm is never materialised.
inline cudaError_t launch_gateup_gather_tc(const __nv_bfloat16* x, int T, const int32_t* src,
                                           int div, const int32_t* offsets, const __nv_bfloat16* w_gate,
                                           const __nv_bfloat16* w_up, int R, int d, int F, int E,
                                           __nv_bfloat16* h, cudaStream_t s) {
  const int sms = tc::sm_count();
  const int bn = tc::choose_bn(R, E, F, true, sms);
  CUtensorMap m[3];
  if (!tc::make_map(&m[0], x, (uint64_t)T, (uint64_t)d, 1) ||  // one-row box for gather4
      !tc::make_map(&m[1], w_gate, (uint64_t)E * F, (uint64_t)d, bn / 2) ||
      !tc::make_map(&m[2], w_up, (uint64_t)E * F, (uint64_t)d, bn / 2))
    return cudaErrorInvalidValue;
  switch (bn) {
    case 64:
      return tc::launch_bn<true, 64, false, true>(m[0], m[1], m[2], offsets, R, E, F, d, h, sms, s,
                                                  nullptr, nullptr, 1, x, src, div);
    case 128:
      return tc::launch_bn<true, 128, false, true>(m[0], m[1], m[2], offsets, R, E, F, d, h, sms, s,
                                                   nullptr, nullptr, 1, x, src, div);
    default:
      return tc::launch_bn<true, 256, false, true>(m[0], m[1], m[2], offsets, R, E, F, d, h, sms, s,
                                                   nullptr, nullptr, 1, x, src, div);
  }
}

inline cudaError_t launch_down_tc(const __nv_bfloat16* h, const int32_t* offsets,
                                  const __nv_bfloat16* w_down, int R, int d, int F, int E,
                                  float* y_perm, cudaStream_t s) {
  const int sms = tc::sm_count();
  const int bn = tc::choose_bn(R, E, d, false, sms);
  const int mode = bn == 256 ? tc::cluster_mode() : 0;
  // A, and B with a full-tile box and a half-height box (single CTA: tiles and
  // tail halves; PAIR: quarter box for tail halves, half box for tiles)
  CUtensorMap m[3];
  if (!tc::make_map(&m[0], h, (uint64_t)R, (uint64_t)F, tc::BM) ||
      !tc::make_map(&m[1], w_down, (uint64_t)E * d, (uint64_t)F, mode == 2 ? bn / 4 : bn) ||
      !tc::make_map(&m[2], w_down, (uint64_t)E * d, (uint64_t)F, bn / 2))
    return cudaErrorInvalidValue;
  if (mode != 0)
    return tc::launch_paired<false, false>(m[0], m[1], m[2], offsets, R, E, d, F, y_perm, s);
  return tc::launch<false>(m, bn, offsets, R, E, d, F, y_perm, sms, s);
}

// Down projection fused with the combine for k <= 2 (deterministic, see the
// kernel): y [T, d] must be zero on entry; row r adds topk_w[perm[r]] * (h_r
// W_down^T) into y[perm[r] / k].
inline cudaError_t launch_down_combine_tc(const __nv_bfloat16* h, const int32_t* offsets,
                                          const __nv_bfloat16* w_down, int R, int d, int F, int E,
                                          const int32_t* perm, const float* topk_w, int k, float* y,
                                          cudaStream_t s) {
  const int sms = tc::sm_count();
  const int mode = tc::cluster_mode();
  CUtensorMap m[3];  // A, and B boxes as in launch_down_tc (256 wide)
  if (!tc::make_map(&m[0], h, (uint64_t)R, (uint64_t)F, tc::BM) ||
      !tc::make_map(&m[1], w_down, (uint64_t)E * d, (uint64_t)F, mode == 2 ? 64 : 256) ||
      !tc::make_map(&m[2], w_down, (uint64_t)E * d, (uint64_t)F, 128))
    return cudaErrorInvalidValue;
  // y's lines stay in L2 between a token's two additions when y takes at most a
  // quarter of L2 (32 MiB: T = 8192, d = 1024 exactly); a larger y would push
  // out H and W_down
  const size_t y_bytes = (size_t)((R + k - 1) / k) * d * sizeof(float);
  const int y_keep = y_bytes <= (size_t)32 << 20 ? 1 : 0;
  if (mode != 0)
    return tc::launch_paired<false, true>(m[0], m[1], m[2], offsets, R, E, d, F, y, s, perm,
                                          topk_w, k, y_keep);
  return tc::launch_bn<false, 256, true>(m[0], m[1], m[2], offsets, R, E, d, F, y, sms, s, perm,
                                         topk_w, k);
}

}  // namespace moe
