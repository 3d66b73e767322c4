"""Plain fp64 CPU oracle of the sparse MoE SwiGLU layer forward.

TEST INFRASTRUCTURE.  Only the test-suite, the package smoke check and the
CPU-baseline leg of the benchmark may import this module.  It shares no code
with the CUDA path; it is a direct restatement of the pages' equations in
numpy, slow on purpose, written so a reader can check it against the pages.

Pages cited (title, site):
  [moe-theory]  "Mixture of Experts（MoE）の理論と実装 — 条件付き計算でLLMを効率化する",
                disassemble-channel.com
  [moe-intro]   Qiita MoE explainer (hiyoko1729), section "ゲート / ルーターって何者？"
  [sparse-moe]  "Sparse Mixture of Experts(MoE) 아키텍처 심층 분석: 설계 원리부터
                DeepSeek-V3·Qwen3까지", youngju.dev
  [zh-moe]      "机器学习基础系列——混合专家模型", sshipanoo.com

Readings of points the pages leave open (each also listed in the design notes):
  * selection is made on the logits (softmax is monotone within a row), ties go
    to the lower expert index; slot 0 holds the largest weight;
  * the selected weights are renormalised to sum to 1 (code on every page);
    without renormalisation (the equations of [moe-intro] and [sparse-moe]) they
    are the selected softmax probabilities as they are;
  * f_i = count_i / T, so sum(f) = k, loss = E * sum(f * p) (unweighted); in the
    convention of [sparse-moe] f_i = count_i / (T k), so sum(f) = 1;
  * the router bias, when present, is added to the logits before the softmax;
  * expert choice selects per expert on the logit column (same order as the
    softmax over tokens), ties to the lower token index, output in descending
    score order; the combine weight is the raw score (no renormalisation);
  * dispatch order inside an expert segment is ascending assignment id t*k+j;
  * capacity-limited token choice keeps, per expert, its first `capacity`
    assignments in token order (the greedy loop of [zh-moe]).

Every function here is pinned by ``tests/test_oracle_pins.py`` against
closed forms, invariants, brute force and library special cases.
"""

from __future__ import annotations

import math
from typing import Optional, Sequence, Tuple

import numpy as np

Array = np.ndarray


def router_logits(x: Array, w_g: Array, bias: Optional[Array] = None) -> Array:
    """s[t, e] = sum_i x[t, i] * W_g[e, i] (+ b[e]).

    [moe-theory] MoELayer.route (gate logits); [moe-intro] equation s = W_g x;
    [sparse-moe] TopKGating (nn.Linear without bias, weight [E, d]);
    [zh-moe] GatingNetwork.forward (adds the bias b).
    """
    s = np.asarray(x, np.float64) @ np.asarray(w_g, np.float64).T
    if bias is not None:
        s = s + np.asarray(bias, np.float64)[None, :]
    return s


def softmax(s: Array, axis: int = -1) -> Array:
    """Max-subtracted softmax.  [moe-theory] MoELayer.route (softmax block)."""
    m = np.max(s, axis=axis, keepdims=True)
    z = np.exp(s - m)
    return z / np.sum(z, axis=axis, keepdims=True)


def topk_select(s: Array, k: int) -> Array:
    """Indices of the k largest logits per row, largest first, ties to the lower index.

    [moe-theory] MoELayer.route uses argsort(-g)[:, :k]; a stable sort on -s
    makes the tie order explicit (lower expert index first).
    """
    return np.argsort(-s, axis=1, kind="stable")[:, :k].astype(np.int64)


def topk_route(s: Array, k: int, renormalize: bool = True) -> Tuple[Array, Array, Array]:
    """(idx [T,k], w [T,k], g [T,E]) with w the renormalised selected probabilities.

    [moe-theory] MoELayer.route: g = softmax(s); select top-k; w_j = g_{i_j} / sum_sel g.
    [sparse-moe] TopKGating.forward does the same with torch.topk.
    renormalize=False: w_j = g_{i_j} as it is, the gate of the equations in
    [moe-intro] "ゲート / ルーターって何者？" (y = sum over TopK of g_i E_i(x)) and of the
    top-k gating formula in [sparse-moe].
    """
    g = softmax(s, axis=1)
    idx = topk_select(s, k)
    w = np.zeros(idx.shape, np.float64)
    for t in range(s.shape[0]):
        sel = g[t, idx[t]]
        w[t] = sel / np.sum(sel) if renormalize else sel
    return idx, w, g


def aux_stats(g: Array, idx: Array, E: int) -> Tuple[Array, Array, Array, float]:
    """(counts [E], f [E], p [E], loss): load-balancing statistics.

    [moe-theory] MoELayer.load_balancing_loss: f_i counts the selections of
    expert i divided by the number of tokens (so sum f = k), p_i is the mean
    routing probability, loss = E * sum_i f_i p_i (balanced routing gives k).
    """
    T, k = idx.shape
    counts = np.zeros(E, np.int64)
    for t in range(T):
        for j in range(k):
            counts[idx[t, j]] += 1
    f = counts.astype(np.float64) / T
    p = np.mean(g, axis=0)
    loss = float(E * np.sum(f * p))
    return counts, f, p, loss


def aux_stats_fraction(g: Array, idx: Array, E: int) -> Tuple[Array, float]:
    """(f [E], loss) in the convention of [sparse-moe] compute_load_balancing_loss:
    f_i is the fraction of the T*k assignments routed to expert i (sum f = 1),
    p_i the mean routing probability, loss = E * sum_i f_i p_i (balanced routing
    gives 1).
    """
    T, k = idx.shape
    counts = np.zeros(E, np.int64)
    for t in range(T):
        for j in range(k):
            counts[idx[t, j]] += 1
    f = counts.astype(np.float64) / (T * k)
    p = np.mean(g, axis=0)
    return f, float(E * np.sum(f * p))


def router_z_loss(s: Array) -> float:
    """mean_t (log sum_e exp s[t, e])^2, the ST-MoE style router z-loss of
    [sparse-moe] router_z_loss (logsumexp over the experts, squared, averaged
    over the tokens); the log-sum-exp is taken with the row max subtracted."""
    s = np.asarray(s, np.float64)
    m = np.max(s, axis=1)
    log_z = m + np.log(np.sum(np.exp(s - m[:, None]), axis=1))
    return float(np.mean(log_z ** 2))


def dispatch(idx: Array, E: int) -> Tuple[Array, Array, Array, Array]:
    """(counts [E], offsets [E+1], perm [T*k], inv_perm [T*k]).

    Assignment a = t*k + j goes to expert idx[t, j].  Rows are grouped by
    expert in ascending expert order and, inside an expert, by ascending a:
    the stable form of the argsort over expert indices in [sparse-moe]
    ExpertParallelRouter.dispatch.  perm[row] = a, inv_perm[a] = row.
    """
    flat = idx.reshape(-1)
    perm = np.argsort(flat, kind="stable").astype(np.int64)
    counts = np.bincount(flat, minlength=E).astype(np.int64)
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
    inv_perm = np.empty_like(perm)
    inv_perm[perm] = np.arange(perm.size, dtype=np.int64)
    return counts, offsets, perm, inv_perm


def silu(a: Array) -> Array:
    """a * sigmoid(a) = a / (1 + exp(-a)).  [moe-theory] Expert.forward."""
    return a / (1.0 + np.exp(-a))


def swiglu_expert(x_rows: Array, w_gate: Array, w_up: Array, w_down: Array,
                  round_h=None) -> Array:
    """E(x) = W_down (silu(W_gate x) * (W_up x)) for each row of x_rows.

    [moe-theory] Expert.forward (W1 is the up projection, W2 the down one);
    [sparse-moe] SwiGLUExpert.forward (nn.Linear layout, no bias, dropout off).
    ``round_h`` optionally maps the hidden activation through a rounding
    function (used only to model a low-precision hidden tensor).
    """
    gate = x_rows @ np.asarray(w_gate, np.float64).T
    up = x_rows @ np.asarray(w_up, np.float64).T
    h = silu(gate) * up
    if round_h is not None:
        h = round_h(h)
    return h @ np.asarray(w_down, np.float64).T


def moe_forward(x: Array, idx: Array, w: Array, experts: Sequence, round_h=None) -> Array:
    """y_t = sum_{j<k} w[t,j] * E_{idx[t,j]}(x_t), summed in slot order j = 0..k-1.

    Loop structure of [sparse-moe] MoELayerWithAuxLoss.forward: for each slot,
    for each expert, run the expert on the tokens whose slot selects it and
    add the weighted output.  [moe-theory] MoELayer.forward is the same sum
    written per token.  x: [T, d] fp64, experts[e] -> (W_gate, W_up, W_down).
    """
    T, k = idx.shape
    contrib = np.zeros((k, T, x.shape[1]), np.float64)
    for e in range(len(experts)):
        rows_any = np.any(idx == e, axis=1)
        if not rows_any.any():
            continue
        wg, wu, wd = experts[e]
        for j in range(k):
            mask = idx[:, j] == e
            if mask.any():
                out = swiglu_expert(x[mask], wg, wu, wd, round_h)
                contrib[j, mask] = w[mask, j][:, None] * out
    y = np.zeros((T, x.shape[1]), np.float64)
    for j in range(k):
        y += contrib[j]
    return y


def dense_mixture(x: Array, g: Array, experts: Sequence) -> Array:
    """y = sum over all experts of g_i * E_i(x).  [zh-moe] MixtureOfExperts.forward."""
    y = np.zeros((x.shape[0], x.shape[1]), np.float64)
    for e in range(len(experts)):
        y += g[:, e:e + 1] * swiglu_expert(x, *experts[e])
    return y


def token_capacity(T: int, E: int, capacity_factor: float, k: int) -> int:
    """Assignments one expert may take: int((T / E) * capacity_factor * k).
    [zh-moe] expert_capacity_routing (capacity = tokens per expert x factor x top_k)."""
    return int(math.floor((T / E) * capacity_factor * k))


def capacity_route(s: Array, k: int, capacity_factor: float):
    """Token choice with a per-expert capacity, [zh-moe] expert_capacity_routing:
    tokens in ascending order take their top-k experts while the expert still has
    room (its load below the capacity), the others are dropped; the kept
    probabilities of a token are renormalised over its kept slots (a token with
    none kept gets zero weights).

    The k experts of one token are distinct, so the order of its slots does not
    change which assignments are kept; the selection itself is topk_route's.
    Returns (idx [T,k], w [T,k] with 0 on dropped slots, kept [T,k] bool,
    dropped count, load [E], capacity).
    """
    T, E = s.shape
    cap = token_capacity(T, E, capacity_factor, k)
    idx, _, g = topk_route(s, k)
    load = np.zeros(E, np.int64)
    kept = np.zeros(idx.shape, bool)
    for t in range(T):
        for j in range(k):
            e = idx[t, j]
            if load[e] < cap:
                kept[t, j] = True
                load[e] += 1
    w = np.zeros(idx.shape, np.float64)
    for t in range(T):
        sel = np.where(kept[t], g[t, idx[t]], 0.0)
        total = np.sum(sel)
        if total > 0:
            w[t] = sel / total
    return idx, w, kept, int(np.sum(~kept)), load, cap


def expert_choice_capacity(T: int, E: int, capacity_factor: float) -> int:
    """C = int(T * capacity_factor / E).  [sparse-moe] ExpertChoiceGating.forward."""
    return int(math.floor(T * capacity_factor / E))


def expert_choice_route(s: Array, capacity_factor: float) -> Tuple[int, Array, Array, Array]:
    """(C, ec_idx [E,C], ec_score [E,C], pos [E,T]).

    [sparse-moe] ExpertChoiceGating.forward: scores = softmax over tokens of
    each expert's logit column; every expert keeps its C highest-scoring
    tokens (descending score, ties to the lower token index); the dispatch
    mask holds the score at the chosen tokens.  pos[e, t] is the dispatch row
    e*C + c of token t in expert e's segment, or -1.
    """
    T, E = s.shape
    C = expert_choice_capacity(T, E, capacity_factor)
    scores = softmax(s.T, axis=1)  # [E, T]
    ec_idx = np.zeros((E, C), np.int64)
    ec_score = np.zeros((E, C), np.float64)
    pos = np.full((E, T), -1, np.int64)
    for e in range(E):
        order = np.argsort(-s[:, e], kind="stable")[:C]
        ec_idx[e] = order
        ec_score[e] = scores[e, order]
        pos[e, order] = e * C + np.arange(C)
    return C, ec_idx, ec_score, pos


def expert_choice_forward(x: Array, ec_idx: Array, ec_score: Array, experts: Sequence,
                          round_h=None) -> Array:
    """y_t = sum over experts e (ascending) that chose t of score[e,t] * E_e(x_t).

    The combine of [sparse-moe] ExpertChoiceGating's dispatch mask: a token
    chosen by no expert gets 0 from the layer (the residual is outside it).
    """
    E, C = ec_idx.shape
    y = np.zeros((x.shape[0], x.shape[1]), np.float64)
    for e in range(E):
        if C == 0:
            continue
        out = swiglu_expert(x[ec_idx[e]], *experts[e], round_h=round_h)
        y[ec_idx[e]] += ec_score[e][:, None] * out
    return y


def bf16_round(a: Array) -> Array:
    """Round fp64 values to the nearest bf16 value (ties to even), returned as fp64.

    bf16 keeps 8 significant bits: with a = m * 2**ex, 0.5 <= |m| < 1, the
    representable neighbours are multiples of 2**(ex - 8).  Models a tensor
    stored in bf16; used only when a test asks for it.  Normal range only.
    """
    m, ex = np.frexp(np.asarray(a, np.float64))
    return np.ldexp(np.rint(np.ldexp(m, 8)), ex - 8)
