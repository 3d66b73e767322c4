/*
 * moe.h — C ABI of the sparse Mixture-of-Experts SwiGLU layer forward (B300, sm_103a).
 *
 * Pages the operations follow (title, site, section):
 *   [moe-theory]  "Mixture of Experts（MoE）の理論と実装 — 条件付き計算でLLMを効率化する",
 *                 disassemble-channel.com: Expert, MoELayer.route / forward / load_balancing_loss
 *   [moe-intro]   Qiita MoE explainer (hiyoko1729), "ゲート / ルーターって何者？" equations
 *   [sparse-moe]  "Sparse Mixture of Experts(MoE) 아키텍처 심층 분석", youngju.dev:
 *                 SwiGLUExpert, TopKGating, ExpertChoiceGating, compute_load_balancing_loss,
 *                 MoELayerWithAuxLoss, ExpertParallelRouter.dispatch
 *   [zh-moe]      "机器学习基础系列——混合专家模型", sshipanoo.com: GatingNetwork (bias)
 *
 * Conventions shared by every call
 *   - Every tensor pointer is a DEVICE pointer owned by the caller, row-major,
 *     and must stay valid until the work enqueued on `stream` has finished.
 *     The library never allocates device memory; scratch comes from the caller.
 *   - Every call only enqueues work on `stream` (a cudaStream_t; NULL is the
 *     legacy default stream) and never waits for the device.
 *   - moe_dtype applies to x and to every weight tensor; routing outputs are
 *     always fp32 / int32; the layer output y is always fp32.
 *   - Weights use the nn.Linear layout: W_g [E,d]; W_gate, W_up [E,F,d]
 *     (K-major rows); W_down [E,d,F].
 *   - T == 0 (or R == 0) is a valid no-op.
 *   - Index tensors are device data the host never reads, so they are not
 *     checked: topk_idx values must lie in [0, E), offsets must be
 *     non-decreasing with offsets[E] <= R, gather sources in [0, T*div),
 *     inv_perm values in [0, R) or -1, pos values in [0, E*C) or -1.  Values
 *     outside these ranges are undefined behaviour (out-of-bounds accesses).
 *     The layer call produces all of them itself and is not exposed to this.
 *   - Errors are reported by the return value.  Arguments are checked before
 *     the first launch, so on MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED and
 *     MOE_ERR_WORKSPACE nothing is enqueued; after MOE_ERR_CUDA earlier stages
 *     of the same call may have been enqueued and the outputs are undefined.
 *       MOE_ERR_INVALID_ARG  null required pointer, negative size, k < 1,
 *                            k > E, E > 256, capacity C > T, capacity_factor <= 0
 *       MOE_ERR_UNSUPPORTED  dtype/shape/alignment outside what the kernels take
 *                            (bf16 needs d and F multiples of 64, pointers 16-byte
 *                            aligned; fp32 needs d and F multiples of 4)
 *       MOE_ERR_WORKSPACE    ws_bytes smaller than the matching *_workspace_size
 *       MOE_ERR_CUDA         a CUDA launch/attribute call failed (cudaGetLastError)
 *   - Kernels that wait on barriers give up after a bounded time and record a
 *     non-zero code in the library's device error word (moe_device_error);
 *     their outputs are then undefined, and the CUDA context stays usable.
 */
#ifndef MOE_H_
#define MOE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* moe_stream_t; /* identical to cudaStream_t */

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,
  MOE_ERR_UNSUPPORTED = 2,
  MOE_ERR_WORKSPACE = 3,
  MOE_ERR_CUDA = 4
} moe_status;

typedef enum { MOE_F32 = 0, MOE_BF16 = 1 } moe_dtype;

typedef enum { MOE_ROUTING_TOPK = 0, MOE_ROUTING_EXPERT_CHOICE = 1 } moe_routing;

/* Largest expert count any call accepts. */
#define MOE_MAX_EXPERTS 256

/* Routing flags (moe_route flags, moe_layer_desc.flags).
 * MOE_ROUTE_NO_RENORM: the combine weights are the selected probabilities
 * g[t,idx] as they are, the gate of the equations in [moe-intro] ("ゲート /
 * ルーターって何者？", y = sum over TopK of g_i E_i(x)) and [sparse-moe] (top-k
 * gating formula); without it they are renormalised to sum to 1, as the code
 * on every page does. */
#define MOE_ROUTE_NO_RENORM 1
/* MOE_ROUTE_CAPACITY (moe_layer_desc.flags, top-k): capacity-limited token
 * choice of [zh-moe] expert_capacity_routing.  Each expert takes at most
 * capacity = int(T / E * capacity_factor * k) assignments (computed in double,
 * in this order), the first ones in token order; the others are dropped (no
 * dispatch row, inv_perm -1) and each token's kept weights are renormalised
 * over its kept slots (all 0 when none is kept).  Needs capacity_factor > 0;
 * not combinable with MOE_ROUTE_NO_RENORM.  counts, f and p describe the
 * routing before the drops; offsets the kept segments. */
#define MOE_ROUTE_CAPACITY 2

/* Human-readable name of a status code (static string, never NULL). */
const char* moe_status_string(moe_status status);

/* Reads (and if clear != 0, resets) the device error word on the current
 * device.  0 means no kernel gave up on a barrier wait.  This call
 * synchronises the device; it is a diagnostic, not part of the hot path. */
moe_status moe_device_error(uint32_t* word, int clear);

/* Self-test of the bounded waits.  Runs the expert-choice selection that
 * moe_expert_choice_route runs (T tokens, E experts, C picks per expert; pos
 * holds the logits transposed, [E,T] fp32 bits) as its one cooperative launch,
 * with every expert's count of arrived slices started far below zero, so that
 * the wait of each CTA for its expert's other slices is never satisfied.  Each
 * such wait gives up after its limit (1 s), records code 16 in the device error
 * word and returns, writing no picks: the launch ends and the context stays
 * usable.  ec_idx [E,C], ec_score [E,C] and pos are left undefined; ws as for
 * moe_expert_choice_route (at least moe_expert_choice_workspace_size for the
 * same T, E and C).  Errors: MOE_ERR_INVALID_ARG for T < 1, E outside 1..256,
 * C outside 1..T or a NULL array; MOE_ERR_WORKSPACE; MOE_ERR_UNSUPPORTED when the
 * E * ceil(T / 1024) CTAs cannot all be resident at once (the two-launch form
 * has no such wait).  A diagnostic that takes about a second, not part of the
 * hot path. */
moe_status moe_selftest_wait_expiry(int T, int E, int C, int32_t* ec_idx, float* ec_score,
                                    int32_t* pos, void* ws, size_t ws_bytes, moe_stream_t stream);

/* ------------------------------------------------------------------ router
 * Token-choice router ([moe-theory] MoELayer.route; [moe-intro] s = W_g x,
 * g = softmax(s), TopK; [sparse-moe] TopKGating; bias as in [zh-moe]
 * GatingNetwork):
 *   s[t,e]  = sum_i x[t,i] * w_g[e,i] + bias[e]            (fp32 accumulate)
 *   g[t,:]  = softmax(s[t,:])                               (max-subtracted)
 *   topk_idx[t,j], j < k: the k largest s[t,:], slot 0 largest, ties to the
 *             lower expert index (selection on the logits: the softmax is
 *             monotone in a row, so this is the same set)
 *   topk_w[t,j] = g[t,idx] / sum_{j'} g[t,idx_j']            (sums to 1),
 *             or g[t,idx] itself with flags & MOE_ROUTE_NO_RENORM
 * Arguments
 *   x [T,d] (dt), w_g [E,d] (dt), bias [E] fp32 or NULL
 *   topk_idx [T,k] int32, topk_w [T,k] fp32             (required outputs)
 *   logits [T,E] fp32, probs [T,E] fp32                 (optional, NULL to skip)
 *   aux_partials: optional fp32 [moe_route_aux_rows(T), E]; when given, row r
 *             holds sum of g[t,e] over the r-th block of tokens (32 tokens
 *             for E <= 16, 64 above; moe_route_aux_rows(T) covers both),
 *             consumed by moe_aux_loss.
 *   z_partials: optional fp32 [moe_route_aux_rows(T)]; entry r holds the sum
 *             over the r-th block of tokens of (log sum_e exp s[t,e])^2, the
 *             router z-loss of [sparse-moe] router_z_loss before its mean
 *             (consumed by moe_aux_loss).
 * Limits: 1 <= k <= E <= 256.                                               */
size_t moe_route_aux_rows(int T);
moe_status moe_route(const void* x, const void* w_g, const float* bias, int T, int d, int E,
                     int k, moe_dtype dt, int32_t* topk_idx, float* topk_w, float* logits,
                     float* probs, float* aux_partials, float* z_partials, int flags,
                     moe_stream_t stream);

/* -------------------------------------------------- expert-choice router
 * [sparse-moe] ExpertChoiceGating.forward:
 *   s = x w_g^T + bias;  score[e,t] = softmax over t of s[:,e]
 *   C = floor(T * capacity_factor / E)            (moe_expert_choice_capacity)
 *   expert e keeps its C highest-scoring tokens, in descending score order,
 *   ties to the lower token index (selection on the logit column).
 * Outputs
 *   ec_idx [E,C] int32 token ids, ec_score [E,C] fp32 scores,
 *   pos [E,T] int32: e*C + c where token t is expert e's c-th pick, else -1
 *     (the non-zero pattern of the page's dispatch mask; dispatch row of a pick),
 *   logits [T,E] fp32: required.
 * pos doubles as scratch: the router stores the logits there transposed
 * ([E,T] fp32 bits) and the selection reads each row once, coalesced, before
 * writing the position map over it.
 * ws: device scratch of moe_expert_choice_workspace_size(T, E, capacity_factor)
 *   bytes (caller-owned; contents on entry do not matter), holding each
 *   1024-token slice's sorted candidates and softmax partial sums.
 * Errors: MOE_ERR_INVALID_ARG for T < 0, E outside 1..256, a capacity factor
 *   that is not positive or C > T, a required pointer NULL; MOE_ERR_WORKSPACE
 *   when ws is NULL or smaller than the size above (C > 0).
 * Limits: C <= T, E <= 256.                                                  */
int moe_expert_choice_capacity(int T, int E, float capacity_factor);
size_t moe_expert_choice_workspace_size(int T, int E, float capacity_factor);
moe_status moe_expert_choice_route(const void* x, const void* w_g, const float* bias, int T,
                                   int d, int E, float capacity_factor, moe_dtype dt,
                                   int32_t* ec_idx, float* ec_score, int32_t* pos,
                                   float* logits, void* ws, size_t ws_bytes, moe_stream_t stream);

/* ------------------------------------------------------------- dispatch
 * Groups the T*k assignments by expert ([sparse-moe] MoELayerWithAuxLoss
 * masks; stable form of ExpertParallelRouter.dispatch's argsort):
 *   assignment a = t*k + j goes to expert topk_idx[t,j];
 *   counts[e]   = number of assignments of expert e;
 *   offsets     = exclusive scan of counts, offsets[E] = T*k;
 *   perm[row]   = a for row in [offsets[e], offsets[e+1]), ascending a;
 *   inv_perm[a] = row;  x_perm[row,:] = x[perm[row] / k, :].
 * Bit-exact and deterministic.  ws: moe_permute_workspace_size(T,E,k) bytes,
 * 16-byte aligned, contents need not be initialised.                       */
size_t moe_permute_workspace_size(int T, int E, int k);
moe_status moe_permute(const void* x, const int32_t* topk_idx, int T, int d, int E, int k,
                       moe_dtype dt, void* x_perm, int32_t* counts, int32_t* offsets,
                       int32_t* perm, int32_t* inv_perm, void* ws, size_t ws_bytes,
                       moe_stream_t stream);

/* Allocation-free variant of moe_permute: same arguments, outputs and
 * results (bit-exact), but no workspace argument.  The pages have no
 * counterpart; this exists for callers that cannot provide device scratch:
 * plugin hosts that give a kernel only its input and output buffers, and
 * deployments whose device memory is reserved up front by another allocator,
 * so that nothing may call cudaMalloc while they run.  The scratch (per-tile
 * expert counts and their scanned bases) lives in a fixed array of
 * MOE_PERMUTE_NOALLOC_SCRATCH_BYTES inside the library's device memory, held
 * by every GPU that loads the library until the process exits.
 *   Limit: ceil(T*k / 2048) * E <= MOE_PERMUTE_NOALLOC_SCRATCH_BYTES / 8
 *          (32768 for 256 KiB: e.g. T*k up to 262144 at E = 256, 1048576 at
 *          E = 64); larger sizes return MOE_ERR_WORKSPACE without any work.
 *   The first call on each device looks up the array's device address (with
 *   that device current) and caches it; make that first call before any
 *   stream capture.  The call itself never allocates (no cudaMalloc or
 *   cudaFree).
 *   All calls share the one array and it keeps the last call's contents
 *   (every entry a call reads it first writes); calls whose work overlaps on
 *   the GPU race on it, so the caller must serialise them.                  */
#define MOE_PERMUTE_NOALLOC_SCRATCH_BYTES (256u * 1024u)
moe_status moe_permute_noalloc(const void* x, const int32_t* topk_idx, int T, int d, int E, int k,
                               moe_dtype dt, void* x_perm, int32_t* counts, int32_t* offsets,
                               int32_t* perm, int32_t* inv_perm, moe_stream_t stream);

/* Row gather used by both routings: x_perm[r,:] = x[src[r] / div, :] for
 * r < R (div = k for top-k perm arrays, 1 for expert-choice token ids).    */
moe_status moe_gather_rows(const void* x, const int32_t* src, int R, int div, int T, int d,
                           moe_dtype dt, void* x_perm, moe_stream_t stream);

/* ------------------------------------------------------ grouped experts
 * SwiGLU expert FFN ([moe-theory] Expert.forward; [sparse-moe] SwiGLUExpert)
 * over variable-size expert segments: rows [offsets[e], offsets[e+1]) of
 * x_perm belong to expert e.  offsets is a DEVICE array [E+1] (read on the
 * device; the host never waits for it), non-decreasing, offsets[E] <= R.
 *   h[r,:]      = silu(x_perm[r,:] W_gate[e]^T) * (x_perm[r,:] W_up[e]^T)
 *                 (fp32 accumulate; stored in dt, i.e. bf16 for bf16 inputs)
 *   y_perm[r,:] = h[r,:] W_down[e]^T                            (fp32)
 * h is caller scratch [R,F] of dtype dt.  Rows >= offsets[E] are not written.
 * bf16 runs on tcgen05 tensor cores (TMA-fed, TMEM accumulators); fp32 runs
 * on FFMA (exact-fp32 parity path).                                         */
moe_status moe_grouped_gateup_swiglu(const void* x_perm, const int32_t* offsets,
                                     const void* w_gate, const void* w_up, int R, int d, int F,
                                     int E, moe_dtype dt, void* h, moe_stream_t stream);
/* Gate/up with the dispatch gather fused into the operand load: row r of the
 * grouped input is x[src[r] / div, :] of x [T,d], so x_perm is never written.
 * src = perm from moe_permute (div = k), or the expert-choice ec_idx (div = 1).
 * Bit-identical to moe_permute / moe_gather_rows followed by
 * moe_grouped_gateup_swiglu.  bf16 only (MOE_ERR_UNSUPPORTED otherwise);
 * src values must lie in [0, T*div).  It saves the R x d x_perm buffer but is
 * slower when the GEMM is compute-bound: each 128-row block is re-gathered
 * (TMA gather4, 128-byte rows) for every n-block, where the contiguous path
 * loads 16 KiB boxes; moe_layer_forward therefore materialises x_perm.      */
moe_status moe_grouped_gateup_swiglu_gather(const void* x, const int32_t* src, int div, int T,
                                            const int32_t* offsets, const void* w_gate,
                                            const void* w_up, int R, int d, int F, int E,
                                            moe_dtype dt, void* h, moe_stream_t stream);
moe_status moe_grouped_down(const void* h, const int32_t* offsets, const void* w_down, int R,
                            int d, int F, int E, moe_dtype dt, float* y_perm,
                            moe_stream_t stream);
/* Both of the above in sequence. */
moe_status moe_experts_swiglu(const void* x_perm, const int32_t* offsets, const void* w_gate,
                              const void* w_up, const void* w_down, int R, int d, int F, int E,
                              moe_dtype dt, void* h, float* y_perm, moe_stream_t stream);

/* -------------------------------------------------------------- combine
 * [moe-theory] MoELayer.forward / [sparse-moe] MoELayerWithAuxLoss:
 *   y[t,:] = sum_{j=0..k-1} topk_w[t,j] * y_perm[inv_perm[t*k+j], :]
 * summed in slot order in fp32 (deterministic).  y [T,d] fp32.            */
moe_status moe_combine(const float* y_perm, const int32_t* inv_perm, const float* topk_w, int T,
                       int d, int k, float* y, moe_stream_t stream);

/* Expert-choice combine (dispatch mask of [sparse-moe] ExpertChoiceGating):
 *   y[t,:] = sum over e ascending with pos[e,t] >= 0 of
 *            ec_score_flat[pos[e,t]] * y_perm[pos[e,t], :]
 * A token no expert chose gets y = 0.                                      */
moe_status moe_ec_combine(const float* y_perm, const int32_t* pos, const float* ec_score, int T,
                          int d, int E, int C, float* y, moe_stream_t stream);

/* ------------------------------------------------------------ aux stats
 * [moe-theory] MoELayer.load_balancing_loss:
 *   f[e] = counts[e] / T (sum f = k);  p[e] = mean_t g[t,e];
 *   loss = E * sum_e f[e] p[e]     (unweighted; balanced routing gives k)
 * [sparse-moe] compute_load_balancing_loss convention (optional outputs):
 *   f_frac[e] = counts[e] / (T k) (sum 1);  loss_frac = E * sum_e f_frac[e] p[e]
 *   (= loss / k; balanced routing gives 1)
 * p comes from probs [T,E] when probs != NULL, else from aux_partials
 * ([moe_route_aux_rows(T), E], written by moe_route); one must be given.
 * Router z-loss ([sparse-moe] router_z_loss), optional: z_loss = mean over
 *   tokens of (log sum_e exp s)^2 from z_partials (written by moe_route).
 * f, p, loss, f_frac, loss_frac, z_loss: each may be NULL.
 * Fixed-order reductions: deterministic.                                    */
moe_status moe_aux_loss(const float* probs, const float* aux_partials, const int32_t* counts,
                        int T, int E, int k, float* f, float* p, float* loss, float* f_frac,
                        float* loss_frac, const float* z_partials, float* z_loss,
                        moe_stream_t stream);

/* ---------------------------------------------------------- whole layer */
typedef struct {
  int T, d, F, E, k;       /* k ignored for expert choice */
  moe_routing routing;
  float capacity_factor;   /* expert choice; top-k with MOE_ROUTE_CAPACITY */
  moe_dtype dtype;         /* x and weights */
  int flags;               /* routing flags (MOE_ROUTE_NO_RENORM, MOE_ROUTE_CAPACITY), top-k */
} moe_layer_desc;

typedef struct {
  const void* w_g;         /* [E,d] */
  const float* bias;       /* [E] or NULL */
  const void* w_gate;      /* [E,F,d] */
  const void* w_up;        /* [E,F,d] */
  const void* w_down;      /* [E,d,F] */
} moe_layer_weights;

/* Optional outputs of moe_layer_forward; any field may be NULL. */
typedef struct {
  int32_t* topk_idx;       /* [T,k]  top-k only */
  float* topk_w;           /* [T,k]  top-k only */
  float* logits;           /* [T,E] */
  int32_t* counts;         /* [E]    top-k only */
  int32_t* offsets;        /* [E+1]  top-k only */
  float* f;                /* [E]    top-k only */
  float* p;                /* [E]    top-k only */
  float* loss;             /* [1]    top-k only */
  int32_t* ec_idx;         /* [E,C]  expert choice only */
  float* ec_score;         /* [E,C]  expert choice only */
  int32_t* pos;            /* [E,T]  expert choice only */
  float* f_frac;           /* [E]    top-k only: counts / (T k) */
  float* loss_frac;        /* [1]    top-k only: loss / k */
  int32_t* dropped;        /* [1]    top-k with MOE_ROUTE_CAPACITY: dropped assignments */
  float* z_loss;           /* [1]    top-k only: router z-loss */
} moe_layer_outputs;

/* Bytes of scratch moe_layer_forward needs for `desc` (0 on invalid desc). */
size_t moe_layer_workspace_size(const moe_layer_desc* desc);

/* Whole forward pass, one stream, no host synchronisation:
 *   top-k:  route (+aux partials) -> histogram/scan -> stable permute -> gather
 *           -> gate/up GEMM + SwiGLU -> down GEMM -> combine -> aux stats
 *   expert choice: EC route -> gather -> gate/up -> down -> EC combine
 * y [T,d] fp32.  ws: moe_layer_workspace_size(desc) bytes, 256-byte aligned. */
moe_status moe_layer_forward(const moe_layer_desc* desc, const moe_layer_weights* w,
                             const void* x, float* y, const moe_layer_outputs* out, void* ws,
                             size_t ws_bytes, moe_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_H_ */
