"""Pins of the fp64 oracle against what the pages and the mathematics fix.

Nothing here compares the oracle with itself: each pin checks a hand-derived
closed form (tests/golden/hand_cases.json), an invariant the pages state, a
brute-force enumeration on tiny inputs, or a special case that reduces to a
library routine (torch float64 on the CPU, scipy).  The planted-mistake test
at the end applies plausible mistakes to the oracle, on the CPU, and checks
that at least one pin catches each.
"""

import itertools
import json
import math
import os
import types
from fractions import Fraction

import numpy as np
import pytest

import oracle
from sparse_mixture_experts_67_b300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_cases.json")


def _golden():
    with open(GOLDEN) as fh:
        return json.load(fh)


def _log_entry(v):
    return 0.0 if v == 0 else math.log(v)


def _frac(a):
    return np.vectorize(lambda s: float(Fraction(s)))(np.asarray(a, dtype=object)).astype(np.float64)


def _rand_experts(rng, E, d, F, scale=0.3):
    return [(rng.normal(0, scale, (F, d)), rng.normal(0, scale, (F, d)), rng.normal(0, scale, (d, F)))
            for _ in range(E)]


# --------------------------------------------------------------------------- pins


def pin_golden_route(orc):
    g = _golden()
    for name in ("route_two_tokens", "route_three_experts_top2"):
        case = g[name]
        x = np.asarray(case["x"], np.float64)
        w_g = np.vectorize(_log_entry)(np.asarray(case["w_g_log"], np.float64))
        s = orc.router_logits(x, w_g)
        idx, w, probs = orc.topk_route(s, case["k"])
        assert idx.tolist() == case["idx"], name
        np.testing.assert_allclose(w, _frac(case["w"]), rtol=0, atol=1e-15)
        np.testing.assert_allclose(probs, _frac(case["g"]), rtol=0, atol=1e-15)
        counts, f, p, loss = orc.aux_stats(probs, idx, w_g.shape[0])
        assert counts.tolist() == case["counts"], name
        np.testing.assert_allclose(f, _frac(case["f"]), rtol=0, atol=1e-15)
        np.testing.assert_allclose(p, _frac(case["p"]), rtol=0, atol=1e-15)
        assert abs(loss - float(Fraction(case["loss"]))) < 1e-14, name


def pin_golden_dispatch(orc):
    case = _golden()["dispatch_three_tokens"]
    counts, offsets, perm, inv_perm = orc.dispatch(np.asarray(case["idx"]), case["E"])
    assert counts.tolist() == case["counts"]
    assert offsets.tolist() == case["offsets"]
    assert perm.tolist() == case["perm"]
    assert inv_perm.tolist() == case["inv_perm"]


def pin_golden_expert_choice(orc):
    case = _golden()["expert_choice_four_tokens"]
    s = np.vectorize(_log_entry)(np.asarray(case["s_log"], np.float64))
    C, ec_idx, ec_score, pos = orc.expert_choice_route(s, case["capacity_factor"])
    assert C == case["C"]
    assert ec_idx.tolist() == case["ec_idx"]
    np.testing.assert_allclose(ec_score, _frac(case["ec_score"]), rtol=0, atol=1e-15)
    assert pos.tolist() == case["pos"]


def pin_golden_silu(orc):
    case = _golden()["silu_values"]
    np.testing.assert_allclose(orc.silu(np.asarray(case["a"])), case["silu"], rtol=1e-15, atol=0)
    scalar = _golden()["swiglu_scalar"]
    y = orc.swiglu_expert(np.array([[scalar["x"]]]), np.array([[scalar["w_gate"]]]),
                          np.array([[scalar["w_up"]]]), np.array([[scalar["w_down"]]]))
    assert abs(y[0, 0] - scalar["y"]) < 1e-14


def pin_silu_vs_scipy(orc):
    from scipy.special import expit

    a = np.linspace(-30, 30, 1001)
    np.testing.assert_allclose(orc.silu(a), a * expit(a), rtol=1e-13, atol=1e-300)


def pin_weights_sum_to_one(orc):
    rng = np.random.default_rng(1)
    for E in (2, 5, 8, 64):
        s = rng.normal(0, 2.0, (37, E))
        for k in sorted({1, 2, min(4, E), E}):
            idx, w, _ = orc.topk_route(s, k)
            np.testing.assert_allclose(w.sum(axis=1), 1.0, rtol=0, atol=1e-14)
            if k == 1:
                assert np.all(w == 1.0)


def pin_topk_on_logits_form(orc):
    """[zh-moe] torch MoELayer: top-k of the logits, then softmax over those k logits."""
    rng = np.random.default_rng(2)
    s = rng.normal(0, 1.5, (50, 8))
    idx, w, _ = orc.topk_route(s, 3)
    top = np.take_along_axis(s, idx, axis=1)
    z = np.exp(top - top.max(axis=1, keepdims=True))
    np.testing.assert_allclose(w, z / z.sum(axis=1, keepdims=True), rtol=0, atol=1e-15)


def pin_topk_brute_force(orc):
    rng = np.random.default_rng(3)
    for E in (3, 5, 8):
        for k in range(1, E + 1):
            s = rng.normal(0, 1.0, (6, E))
            idx, w, g = orc.topk_route(s, k)
            for t in range(s.shape[0]):
                best = max(itertools.combinations(range(E), k), key=lambda c: sum(g[t, list(c)]))
                assert sorted(idx[t].tolist()) == sorted(best)
                assert all(g[t, idx[t, j]] > g[t, idx[t, j + 1]] for j in range(k - 1))


def pin_all_ties(orc):
    """W_g = 0: every logit ties, so the lower-index rule fixes everything in closed form."""
    T, d = 10, 6
    x = np.random.default_rng(4).normal(size=(T, d))
    for E, k in ((8, 2), (5, 5), (64, 4)):
        s = orc.router_logits(x, np.zeros((E, d)))
        idx, w, g = orc.topk_route(s, k)
        assert np.all(idx == np.arange(k)[None, :])
        np.testing.assert_allclose(w, 1.0 / k, rtol=0, atol=1e-15)
        counts, f, p, loss = orc.aux_stats(g, idx, E)
        assert counts.tolist() == [T] * k + [0] * (E - k)
        np.testing.assert_allclose(f, [1.0] * k + [0.0] * (E - k), rtol=0, atol=0)
        np.testing.assert_allclose(p, 1.0 / E, rtol=0, atol=1e-15)
        assert abs(loss - k) < 1e-12


def pin_unrenormalised_route(orc):
    """Without renormalisation the weights are the selected softmax probabilities of the
    equations ([moe-intro], [sparse-moe]): hand values, the same selection, the same
    ratios, and all of g back when k = E."""
    g = _golden()
    case = g["route_three_experts_top2"]
    x = np.asarray(case["x"], np.float64)
    w_g = np.vectorize(_log_entry)(np.asarray(case["w_g_log"], np.float64))
    s = orc.router_logits(x, w_g)
    idx, w, probs = orc.topk_route(s, case["k"], renormalize=False)
    assert idx.tolist() == case["idx"]
    g_hand = _frac(case["g"])
    np.testing.assert_allclose(w, np.take_along_axis(g_hand, np.asarray(case["idx"]), axis=1),
                               rtol=0, atol=1e-15)
    # W_g = 0, E = 8, k = 2: every probability is 1/8
    s0 = orc.router_logits(np.ones((3, 4)), np.zeros((8, 4)))
    _, w0, _ = orc.topk_route(s0, 2, renormalize=False)
    np.testing.assert_allclose(w0, 1.0 / 8, rtol=0, atol=1e-16)
    rng = np.random.default_rng(21)
    s = rng.normal(0, 2.0, (40, 7))
    for k in (1, 3, 7):
        idx_n, w_n, g_n = orc.topk_route(s, k, renormalize=False)
        idx_r, w_r, _ = orc.topk_route(s, k)
        np.testing.assert_array_equal(idx_n, idx_r)
        assert np.all(w_n.sum(axis=1) <= 1.0 + 1e-15)
        np.testing.assert_allclose(w_n / w_n.sum(axis=1, keepdims=True), w_r, rtol=1e-14, atol=0)
        if k == 7:  # every expert selected: the weights are the whole softmax row
            np.testing.assert_allclose(w_n.sum(axis=1), 1.0, rtol=0, atol=1e-15)
            np.testing.assert_allclose(np.sort(w_n, axis=1), np.sort(g_n, axis=1), rtol=0, atol=0)


def pin_aux_fraction_convention(orc):
    """[sparse-moe] compute_load_balancing_loss: f sums to 1 and balanced routing gives 1;
    the hand case's counts give f = counts / (T k)."""
    case = _golden()["route_two_tokens"]
    x = np.asarray(case["x"], np.float64)
    w_g = np.vectorize(_log_entry)(np.asarray(case["w_g_log"], np.float64))
    idx, _, probs = orc.topk_route(orc.router_logits(x, w_g), case["k"])
    f, loss = orc.aux_stats_fraction(probs, idx, 2)
    T, k = idx.shape
    np.testing.assert_allclose(f, np.asarray(case["counts"], np.float64) / (T * k), rtol=0, atol=0)
    assert abs(loss - float(Fraction(case["loss"])) / k) < 1e-15
    # W_g = 0: the first k experts each take 1/k of the assignments, p = 1/E, loss = 1
    for E, k in ((8, 2), (6, 6), (64, 4)):
        s = orc.router_logits(np.ones((5, 3)), np.zeros((E, 3)))
        idx, _, g = orc.topk_route(s, k)
        f, loss = orc.aux_stats_fraction(g, idx, E)
        np.testing.assert_allclose(f, [1.0 / k] * k + [0.0] * (E - k), rtol=0, atol=1e-16)
        assert abs(loss - 1.0) < 1e-12
    rng = np.random.default_rng(22)
    s = rng.normal(0, 1.0, (50, 9))
    idx, _, g = orc.topk_route(s, 3)
    f, _ = orc.aux_stats_fraction(g, idx, 9)
    assert abs(f.sum() - 1.0) < 1e-15


def pin_capacity_route(orc):
    """[zh-moe] expert_capacity_routing: the hand case, then on random logits the greedy
    rule in closed form (each expert keeps its first `capacity` tokens in order), the
    drop count, per-token renormalisation of the kept weights, and no drops at all
    when the capacity covers every assignment."""
    case = _golden()["capacity_three_tokens_top2"]
    x = np.asarray(case["x"], np.float64)
    w_g = np.vectorize(_log_entry)(np.asarray(case["w_g_log"], np.float64))
    s = orc.router_logits(x, w_g)
    idx, w, kept, dropped, load, cap = orc.capacity_route(s, case["k"], case["capacity_factor"])
    assert cap == case["capacity"] and dropped == case["dropped"]
    assert idx.tolist() == case["idx"] and kept.tolist() == case["kept"]
    assert load.tolist() == case["load"]
    np.testing.assert_allclose(w, _frac(case["w"]), rtol=0, atol=1e-15)
    rng = np.random.default_rng(23)
    T, E = 60, 6
    s = rng.normal(0, 1.5, (T, E))
    s[:, 2] += 2.0  # one popular expert, so its capacity binds
    for k, cf in ((1, 1.0), (2, 0.7), (3, 1.25)):
        idx, w, kept, dropped, load, cap = orc.capacity_route(s, k, cf)
        assert cap == int(math.floor(T / E * cf * k))
        idx_r, w_r, _ = orc.topk_route(s, k)
        np.testing.assert_array_equal(idx, idx_r)
        counts = np.bincount(idx.ravel(), minlength=E)
        np.testing.assert_array_equal(load, np.minimum(counts, cap))
        assert dropped == int(np.sum(np.maximum(counts - cap, 0)))
        for e in range(E):
            tok = [t for t in range(T) for j in range(k) if idx[t, j] == e]  # ascending t
            kept_tok = [t for t in range(T) for j in range(k) if idx[t, j] == e and kept[t, j]]
            assert kept_tok == tok[:cap]
        for t in range(T):
            if kept[t].any():
                assert abs(w[t].sum() - 1.0) < 1e-15
                np.testing.assert_array_equal(w[t][~kept[t]], 0.0)
                ratio = w[t][kept[t]] / w_r[t][kept[t]]
                np.testing.assert_allclose(ratio, ratio[0], rtol=1e-14)
            else:
                np.testing.assert_array_equal(w[t], 0.0)
    idx, w, kept, dropped, load, cap = orc.capacity_route(s, 2, float(E))  # capacity 2T
    assert dropped == 0 and kept.all()
    np.testing.assert_allclose(w, orc.topk_route(s, 2)[1], rtol=0, atol=0)


def pin_router_z_loss(orc):
    """[sparse-moe] router_z_loss: closed forms (equal logits c over E experts give
    (c + ln E)^2; one expert gives mean s^2) and scipy's logsumexp on random logits."""
    from scipy.special import logsumexp

    for E, c in ((8, 0.0), (5, 1.5), (64, -3.0)):
        s = np.full((7, E), c)
        assert abs(orc.router_z_loss(s) - (c + math.log(E)) ** 2) < 1e-12
    s1 = np.array([[0.5], [-2.0], [3.0]])
    assert abs(orc.router_z_loss(s1) - np.mean(s1[:, 0] ** 2)) < 1e-15
    rng = np.random.default_rng(24)
    s = rng.normal(0, 4.0, (50, 16)) + 30.0  # large logits: needs the max subtraction
    ref = float(np.mean(logsumexp(s, axis=1) ** 2))
    assert abs(orc.router_z_loss(s) - ref) <= 1e-12 * ref


def pin_softmax_large_logits(orc):
    """Softmax is unchanged by adding a constant to a row, also where exp alone would
    overflow or underflow in fp64: [a, a-1, a-10] gives [1, e^-1, e^-10] / (1 + e^-1 + e^-10)
    for every a (the max-subtracted form; router and expert-choice scores alike)."""
    ref = np.array([1.0, math.exp(-1.0), math.exp(-10.0)])
    ref /= ref.sum()
    for a in (0.0, 1000.0, -1000.0):
        s = np.array([[a, a - 1.0, a - 10.0]])
        np.testing.assert_allclose(orc.softmax(s, axis=1)[0], ref, rtol=1e-14, atol=0)
        _, w, g = orc.topk_route(s, 3)
        np.testing.assert_allclose(g[0], ref, rtol=1e-14, atol=0)
        _, _, sc, _ = orc.expert_choice_route(s.T.copy(), 1.0)  # 3 tokens, one expert, C = 3
        np.testing.assert_allclose(sc[0], ref, rtol=1e-14, atol=0)


def pin_capacity_rounding(orc):
    """Both capacities truncate as Python int() does on the pages ([sparse-moe]
    ExpertChoiceGating: int(T * capacity_factor / E); [zh-moe] expert_capacity_routing:
    int(T / E * capacity_factor * top_k)).  Values worked by hand where the quotient is
    not an integer: 10*1/4 = 2.5 -> 2, 7*0.5/2 = 1.75 -> 1, 10*0.3/4 = 0.75 -> 0,
    10/3*1.25*2 = 8.33 -> 8, 7/2*1*1 = 3.5 -> 3, 9/4*1.5*2 = 6.75 -> 6."""
    assert orc.expert_choice_capacity(10, 4, 1.0) == 2
    assert orc.expert_choice_capacity(7, 2, 0.5) == 1
    assert orc.expert_choice_capacity(10, 4, 0.3) == 0
    assert orc.expert_choice_capacity(8192, 16, 2.0) == 1024
    assert orc.token_capacity(10, 3, 1.25, 2) == 8
    assert orc.token_capacity(7, 2, 1.0, 1) == 3
    assert orc.token_capacity(9, 4, 1.5, 2) == 6
    s = np.zeros((10, 4))  # all ties: the route takes C tokens per expert
    C, ec_idx, _, _ = orc.expert_choice_route(s, 1.0)
    assert C == 2 and ec_idx.shape == (4, 2)
    assert orc.capacity_route(np.zeros((7, 2)), 1, 1.0)[5] == 3


def pin_bias_only(orc):
    """x = 0: the logits are the bias ([zh-moe] GatingNetwork adds b)."""
    b = np.array([1.5 * math.log(1.0 / (e + 1)) for e in range(6)])
    s = orc.router_logits(np.zeros((3, 4)), np.ones((6, 4)), b)
    np.testing.assert_array_equal(s, np.broadcast_to(b, (3, 6)))
    idx, w, _ = orc.topk_route(s, 2)
    assert idx.tolist() == [[0, 1]] * 3
    # b_0 = 0, b_1 = 1.5 ln(1/2): weights 1 : 2^-1.5
    r = 2.0 ** -1.5
    np.testing.assert_allclose(w[0], [1 / (1 + r), r / (1 + r)], rtol=1e-15)


def pin_aux_invariants(orc):
    rng = np.random.default_rng(5)
    for E, k in ((8, 2), (64, 4), (16, 1)):
        s = rng.normal(0, 1.0, (200, E))
        idx, w, g = orc.topk_route(s, k)
        counts, f, p, loss = orc.aux_stats(g, idx, E)
        assert counts.sum() == 200 * k
        assert abs(f.sum() - k) < 1e-12
        assert abs(p.sum() - 1) < 1e-12
        assert loss > 0


def pin_uniform_loss_is_k(orc):
    """Perfectly balanced routing with uniform probabilities gives loss = k ([moe-theory] demo's ideal)."""
    E, k = 8, 2
    T = 8 * 5
    idx = np.array([[(t + j) % E for j in range(k)] for t in range(T)])
    g = np.full((T, E), 1.0 / E)
    counts, f, p, loss = orc.aux_stats(g, idx, E)
    assert counts.tolist() == [T * k // E] * E
    assert abs(loss - k) < 1e-12


def pin_dispatch_brute_force(orc):
    rng = np.random.default_rng(6)
    for T, E, k in ((1, 1, 1), (13, 5, 2), (40, 8, 3), (7, 64, 4)):
        idx = np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)])
        counts, offsets, perm, inv_perm = orc.dispatch(idx, E)
        rows = []
        for e in range(E):
            for t in range(T):
                for j in range(k):
                    if idx[t, j] == e:
                        rows.append(t * k + j)
        assert perm.tolist() == rows
        assert sorted(perm.tolist()) == list(range(T * k))
        assert np.all(inv_perm[perm] == np.arange(T * k))
        assert offsets[0] == 0 and np.all(np.diff(offsets) == counts)
        for e in range(E):
            seg = perm[offsets[e]:offsets[e + 1]]
            assert np.all(np.diff(seg) > 0)
            assert np.all(idx.reshape(-1)[seg] == e)


def pin_swiglu_vs_torch(orc):
    torch = pytest.importorskip("torch")
    import torch.nn.functional as tf

    rng = np.random.default_rng(7)
    n, d, F = 9, 6, 11
    x = rng.normal(size=(n, d))
    wg, wu, wd = rng.normal(size=(F, d)), rng.normal(size=(F, d)), rng.normal(size=(d, F))
    tx = torch.from_numpy(x)
    ref = (tf.silu(tf.linear(tx, torch.from_numpy(wg))) * tf.linear(tx, torch.from_numpy(wu)))
    ref = tf.linear(ref, torch.from_numpy(wd)).numpy()
    np.testing.assert_allclose(orc.swiglu_expert(x, wg, wu, wd), ref, rtol=1e-12, atol=1e-12)


def pin_zero_input(orc):
    rng = np.random.default_rng(8)
    experts = _rand_experts(rng, 4, 5, 7)
    idx = np.array([[0, 3], [2, 1]])
    w = np.array([[0.6, 0.4], [0.3, 0.7]])
    y = orc.moe_forward(np.zeros((2, 5)), idx, w, experts)
    assert np.all(y == 0)


def pin_dense_limit(orc):
    """k = E: the renormalised weights are the full softmax, so the layer is the dense mixture."""
    rng = np.random.default_rng(9)
    T, d, F, E = 12, 5, 7, 4
    x = rng.normal(size=(T, d))
    experts = _rand_experts(rng, E, d, F)
    s = orc.router_logits(x, rng.normal(0, 0.5, (E, d)))
    idx, w, g = orc.topk_route(s, E)
    np.testing.assert_allclose(orc.moe_forward(x, idx, w, experts), orc.dense_mixture(x, g, experts),
                               rtol=1e-12, atol=1e-12)
    # the dense mixture itself against a direct torch evaluation
    torch = pytest.importorskip("torch")
    import torch.nn.functional as tf

    tx = torch.from_numpy(x)
    ref = torch.zeros_like(tx)
    for e, (wg, wu, wd) in enumerate(experts):
        h = tf.silu(tf.linear(tx, torch.from_numpy(wg))) * tf.linear(tx, torch.from_numpy(wu))
        ref += torch.from_numpy(g[:, e:e + 1]) * tf.linear(h, torch.from_numpy(wd))
    np.testing.assert_allclose(orc.dense_mixture(x, g, experts), ref.numpy(), rtol=1e-12, atol=1e-12)


def pin_identical_experts(orc):
    """All experts equal: weights sum to 1, so y = E_0(x) for any k."""
    rng = np.random.default_rng(10)
    T, d, F, E = 15, 6, 9, 8
    x = rng.normal(size=(T, d))
    one = _rand_experts(rng, 1, d, F)[0]
    s = orc.router_logits(x, rng.normal(0, 1.0, (E, d)))
    for k in (1, 2, 5):
        idx, w, _ = orc.topk_route(s, k)
        np.testing.assert_allclose(orc.moe_forward(x, idx, w, [one] * E), orc.swiglu_expert(x, *one),
                                   rtol=1e-12, atol=1e-12)


def pin_single_slot_selects_expert(orc):
    """k = 1: y_t is exactly the output of the selected expert on x_t."""
    rng = np.random.default_rng(11)
    T, d, F, E = 10, 4, 6, 3
    x = rng.normal(size=(T, d))
    experts = _rand_experts(rng, E, d, F)
    s = orc.router_logits(x, rng.normal(0, 1.0, (E, d)))
    idx, w, _ = orc.topk_route(s, 1)
    y = orc.moe_forward(x, idx, w, experts)
    for t in range(T):
        np.testing.assert_allclose(y[t], orc.swiglu_expert(x[t:t + 1], *experts[idx[t, 0]])[0],
                                   rtol=1e-13, atol=1e-13)


def pin_forward_takes_weights_as_given(orc):
    """The combine uses the weights it is handed, unrenormalised ([moe-intro] y = sum of
    g_i E_i(x) over the top k): one-hot slot weights return that slot's expert, weights
    summing to 0.3 or 2.5 give the per-token weighted sum of the slots' experts, and the
    output is linear in the weights."""
    rng = np.random.default_rng(12)
    T, d, F, E, k = 9, 4, 6, 4, 3
    x = rng.normal(size=(T, d))
    experts = _rand_experts(rng, E, d, F)
    idx = np.stack([rng.permutation(E)[:k] for _ in range(T)])
    outs = [[orc.swiglu_expert(x[t:t + 1], *experts[idx[t, j]])[0] for j in range(k)]
            for t in range(T)]
    for j in range(k):
        one_hot = np.zeros((T, k))
        one_hot[:, j] = 1.0
        y = orc.moe_forward(x, idx, one_hot, experts)
        for t in range(T):
            np.testing.assert_allclose(y[t], outs[t][j], rtol=1e-13, atol=1e-13)
    for total in (0.3, 2.5):
        w = rng.uniform(0.1, 1.0, (T, k))
        w *= total / w.sum(axis=1, keepdims=True)
        y = orc.moe_forward(x, idx, w, experts)
        for t in range(T):
            ref = sum(w[t, j] * outs[t][j] for j in range(k))
            np.testing.assert_allclose(y[t], ref, rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(orc.moe_forward(x, idx, 3.0 * w, experts), 3.0 * y,
                                   rtol=1e-12, atol=1e-13)


def pin_expert_choice_invariants(orc):
    rng = np.random.default_rng(12)
    for T, E, cf in ((30, 4, 1.0), (64, 16, 2.0), (9, 3, 0.25), (16, 4, 4.0)):
        s = rng.normal(0, 1.0, (T, E))
        C, ec_idx, ec_score, pos = orc.expert_choice_route(s, cf)
        assert C == int(T * cf // E)
        assert ec_idx.shape == (E, C)
        for e in range(E):
            assert len(set(ec_idx[e].tolist())) == C
            col = np.exp(s[:, e] - s[:, e].max())
            col /= col.sum()
            assert abs(col.sum() - 1) < 1e-12
            np.testing.assert_allclose(ec_score[e], col[ec_idx[e]], rtol=1e-14)
            assert np.all(np.diff(ec_score[e]) <= 0)
        assert int((pos >= 0).sum()) == E * C
        for e in range(E):
            for c in range(C):
                assert pos[e, ec_idx[e, c]] == e * C + c


def pin_expert_choice_brute_force(orc):
    rng = np.random.default_rng(13)
    for T, E, cf in ((8, 2, 1.0), (12, 3, 1.0), (10, 5, 2.0)):
        s = rng.normal(0, 1.0, (T, E))
        C, ec_idx, ec_score, _ = orc.expert_choice_route(s, cf)
        for e in range(E):
            best = max(itertools.combinations(range(T), C), key=lambda c: sum(np.exp(s[list(c), e])))
            assert sorted(ec_idx[e].tolist()) == sorted(best)


def pin_expert_choice_ties_and_empty(orc):
    s = np.zeros((10, 4))
    C, ec_idx, ec_score, pos = orc.expert_choice_route(s, 2.0)
    assert C == 5
    assert np.all(ec_idx == np.arange(5)[None, :])
    np.testing.assert_allclose(ec_score, 0.1, rtol=0, atol=1e-16)
    C0, idx0, sc0, pos0 = orc.expert_choice_route(s, 0.3)
    assert C0 == 0 and idx0.shape == (4, 0) and np.all(pos0 == -1)
    y = orc.expert_choice_forward(np.ones((10, 3)), idx0, sc0, _rand_experts(np.random.default_rng(0), 4, 3, 2))
    assert np.all(y == 0)


def pin_expert_choice_forward(orc):
    """Only tokens chosen by an expert receive its output, weighted by the raw score."""
    rng = np.random.default_rng(14)
    T, d, F, E = 12, 4, 5, 3
    x = rng.normal(size=(T, d))
    experts = _rand_experts(rng, E, d, F)
    s = rng.normal(size=(T, E))
    C, ec_idx, ec_score, pos = orc.expert_choice_route(s, 1.0)
    y = orc.expert_choice_forward(x, ec_idx, ec_score, experts)
    for t in range(T):
        ref = np.zeros(d)
        for e in range(E):
            if pos[e, t] >= 0:
                c = pos[e, t] - e * C
                ref += ec_score[e, c] * orc.swiglu_expert(x[t:t + 1], *experts[e])[0]
        np.testing.assert_allclose(y[t], ref, rtol=1e-13, atol=1e-15)


def pin_bf16_round(orc):
    rng = np.random.default_rng(15)
    a = (rng.normal(0, 3.0, 100000) * np.exp(rng.uniform(-20, 20, 100000))).astype(np.float32)
    # exact halfway cases between bf16 neighbours exercise the ties-to-even rule
    halfway = np.array([1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -(2.0 + 2.0 ** -7)], np.float32)
    a = np.concatenate([a, halfway])
    np.testing.assert_array_equal(orc.bf16_round(a.astype(np.float64)),
                                  synth.to_f64(synth.round_to_bf16_bits(a)))


PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_oracle_pin(pin):
    pin(oracle)


# ------------------------------------------------------------- planted mistakes


def _mutant(**overrides):
    ns = types.SimpleNamespace(**{k: getattr(oracle, k) for k in dir(oracle) if not k.startswith("__")})
    for k, v in overrides.items():
        setattr(ns, k, v)
    return ns


def _no_renorm(s, k, renormalize=True):
    g = oracle.softmax(s, axis=1)
    idx = oracle.topk_select(s, k)
    return idx, np.take_along_axis(g, idx, axis=1), g


def _smallest(s, k, renormalize=True):
    g = oracle.softmax(s, axis=1)
    idx = np.argsort(s, axis=1, kind="stable")[:, :k]
    sel = np.take_along_axis(g, idx, axis=1)
    return idx, sel / sel.sum(axis=1, keepdims=True), g


def _ties_high(s, k, renormalize=True):
    g = oracle.softmax(s, axis=1)
    idx = (s.shape[1] - 1 - np.argsort(-s[:, ::-1], axis=1, kind="stable"))[:, :k]
    sel = np.take_along_axis(g, idx, axis=1)
    return idx, sel / sel.sum(axis=1, keepdims=True), g


def _swap_gate_up(x, wg, wu, wd, round_h=None):
    return oracle.swiglu_expert(x, wu, wg, wd, round_h)


def _down_transposed(x, wg, wu, wd, round_h=None):
    h = oracle.silu(x @ wg.T) * (x @ wu.T)
    return h @ wd


def _f_over_tk(g, idx, E):
    counts, f, p, loss = oracle.aux_stats(g, idx, E)
    f2 = f / idx.shape[1]
    return counts, f2, p, float(E * np.sum(f2 * p))


def _loss_no_E(g, idx, E):
    counts, f, p, loss = oracle.aux_stats(g, idx, E)
    return counts, f, p, loss / E


def _dispatch_desc(idx, E):
    counts, offsets, perm, inv_perm = oracle.dispatch(idx, E)
    perm = perm.copy()
    for e in range(E):
        perm[offsets[e]:offsets[e + 1]] = perm[offsets[e]:offsets[e + 1]][::-1]
    inv = np.empty_like(perm)
    inv[perm] = np.arange(perm.size)
    return counts, offsets, perm, inv


def _ec_softmax_over_experts(s, cf):
    T, E = s.shape
    C, ec_idx, _, pos = oracle.expert_choice_route(s, cf)
    g = oracle.softmax(s, axis=1)
    return C, ec_idx, np.stack([g[ec_idx[e], e] for e in range(E)]), pos


def _forward_unweighted(x, idx, w, experts, round_h=None):
    return oracle.moe_forward(x, idx, np.ones_like(w), experts, round_h)


def _always_renormalise(s, k, renormalize=True):
    return oracle.topk_route(s, k)


def _fraction_over_T(g, idx, E):
    counts, f, p, loss = oracle.aux_stats(g, idx, E)
    return f, loss


def _capacity_without_k(s, k, cf):
    T, E = s.shape
    cap = int(math.floor(T / E * cf))
    return _greedy(s, k, cap, order=range(T))


def _greedy(s, k, cap, order, renorm=True):
    T, E = s.shape
    idx, _, g = oracle.topk_route(s, k)
    load = np.zeros(E, np.int64)
    kept = np.zeros(idx.shape, bool)
    for t in order:
        for j in range(k):
            if load[idx[t, j]] < cap:
                kept[t, j] = True
                load[idx[t, j]] += 1
    w = np.where(kept, np.take_along_axis(g, idx, axis=1), 0.0)
    if renorm:
        tot = w.sum(axis=1, keepdims=True)
        w = np.divide(w, tot, out=np.zeros_like(w), where=tot > 0)
    return idx, w, kept, int(np.sum(~kept)), load, cap


def _capacity_last_tokens_first(s, k, cf):
    T, E = s.shape
    return _greedy(s, k, oracle.token_capacity(T, E, cf, k), order=range(T - 1, -1, -1))


def _capacity_no_renorm(s, k, cf):
    T, E = s.shape
    return _greedy(s, k, oracle.token_capacity(T, E, cf, k), order=range(T), renorm=False)


def _z_loss_unsquared(s):
    m = np.max(s, axis=1)
    return float(np.mean(m + np.log(np.sum(np.exp(s - m[:, None]), axis=1))))


def _z_loss_max_only(s):
    return float(np.mean(np.max(s, axis=1) ** 2))


def _softmax_no_max(s, axis=-1):
    with np.errstate(over="ignore", invalid="ignore", under="ignore"):
        z = np.exp(s)
        return z / np.sum(z, axis=axis, keepdims=True)


def _ec_capacity_ceil(T, E, cf):
    return int(math.ceil(T * cf / E))


def _token_capacity_ceil(T, E, cf, k):
    return int(math.ceil(T / E * cf * k))


def _ec_ties_to_higher_token(s, cf):
    T, E = s.shape
    C = oracle.expert_choice_capacity(T, E, cf)
    scores = oracle.softmax(s.T, axis=1)
    ec_idx = np.zeros((E, C), np.int64)
    ec_score = np.zeros((E, C))
    pos = np.full((E, T), -1, np.int64)
    for e in range(E):
        order = (T - 1 - np.argsort(-s[::-1, e], kind="stable"))[:C]
        ec_idx[e], ec_score[e] = order, scores[e, order]
        pos[e, order] = e * C + np.arange(C)
    return C, ec_idx, ec_score, pos


def _ec_combine_renormalised(x, ec_idx, ec_score, experts, round_h=None):
    E, C = ec_idx.shape
    tot = np.zeros(x.shape[0])
    for e in range(E):
        tot[ec_idx[e]] += ec_score[e]
    y = np.zeros((x.shape[0], x.shape[1]))
    for e in range(E):
        if C:
            out = oracle.swiglu_expert(x[ec_idx[e]], *experts[e], round_h=round_h)
            y[ec_idx[e]] += (ec_score[e] / tot[ec_idx[e]])[:, None] * out
    return y


def _ec_combine_unweighted(x, ec_idx, ec_score, experts, round_h=None):
    return oracle.expert_choice_forward(x, ec_idx, np.ones_like(ec_score), experts, round_h)


def _dispatch_offsets_inclusive(idx, E):
    counts, _, perm, inv = oracle.dispatch(idx, E)
    return counts, np.concatenate([np.cumsum(counts), [counts.sum()]]), perm, inv


def _bf16_truncates(a):
    m, ex = np.frexp(np.asarray(a, np.float64))
    return np.ldexp(np.trunc(m * 256.0) / 256.0, ex)


def _dense_uniform(x, g, experts):
    return oracle.dense_mixture(x, np.full_like(g, 1.0 / g.shape[1]), experts)


def _p_from_combine_weights(g, idx, E):
    T, k = idx.shape
    counts, f, _, _ = oracle.aux_stats(g, idx, E)
    p = np.zeros(E)
    for t in range(T):
        sel = g[t, idx[t]]
        for j in range(k):
            p[idx[t, j]] += sel[j] / sel.sum() / T
    return counts, f, p, float(E * np.sum(f * p))


def _forward_last_slot_only(x, idx, w, experts, round_h=None):
    w2 = np.zeros_like(w)
    w2[:, -1] = w[:, -1]
    return oracle.moe_forward(x, idx, w2, experts, round_h)


def _experts_reversed(x, w_g, bias=None):
    s = (np.asarray(x, np.float64) @ np.asarray(w_g, np.float64).T)[:, ::-1].copy()
    return s if bias is None else s + np.asarray(bias, np.float64)[None, :]


def _z_loss_summed(s):
    m = np.max(s, axis=1)
    return float(np.sum((m + np.log(np.sum(np.exp(s - m[:, None]), axis=1))) ** 2))


def _z_loss_without_max_back(s):
    m = np.max(s, axis=1)
    return float(np.mean(np.log(np.sum(np.exp(s - m[:, None]), axis=1)) ** 2))


def _fraction_loss_without_E(g, idx, E):
    f, loss = oracle.aux_stats_fraction(g, idx, E)
    return f, loss / E


def _topk_slots_ascending(s, k, renormalize=True):
    idx, w, g = oracle.topk_route(s, k, renormalize)
    return idx[:, ::-1].copy(), w[:, ::-1].copy(), g


def _dispatch_perm_inv_swapped(idx, E):
    counts, offsets, perm, inv = oracle.dispatch(idx, E)
    return counts, offsets, inv, perm


def _ec_pos_local(s, cf):
    C, ec_idx, ec_score, pos = oracle.expert_choice_route(s, cf)
    pos = pos.copy()
    for e in range(s.shape[1]):
        pos[e, pos[e] >= 0] -= e * C
    return C, ec_idx, ec_score, pos


def _ec_picks_ascending(s, cf):
    C, ec_idx, ec_score, pos = oracle.expert_choice_route(s, cf)
    ec_idx, ec_score = ec_idx[:, ::-1].copy(), ec_score[:, ::-1].copy()
    pos = np.full_like(pos, -1)
    for e in range(s.shape[1]):
        pos[e, ec_idx[e]] = e * C + np.arange(C)
    return C, ec_idx, ec_score, pos


def _glu_without_silu(x, wg, wu, wd, round_h=None):
    h = (x @ np.asarray(wg, np.float64).T) * (x @ np.asarray(wu, np.float64).T)
    h = h if round_h is None else round_h(h)
    return h @ np.asarray(wd, np.float64).T


def _capacity_load_counts_drops(s, k, cf):
    idx, w, kept, dropped, _, cap = oracle.capacity_route(s, k, cf)
    return idx, w, kept, dropped, np.bincount(idx.ravel(), minlength=s.shape[1]), cap


def _capacity_weights_of_all_slots(s, k, cf):
    idx, _, kept, dropped, load, cap = oracle.capacity_route(s, k, cf)
    return idx, np.where(kept, oracle.topk_route(s, k)[1], 0.0), kept, dropped, load, cap


def _p_over_k(g, idx, E):
    counts, f, p, _ = oracle.aux_stats(g, idx, E)
    p = p / idx.shape[1]
    return counts, f, p, float(E * np.sum(f * p))


def _bias_subtracted(x, w_g, bias=None):
    s = np.asarray(x, np.float64) @ np.asarray(w_g, np.float64).T
    return s if bias is None else s - np.asarray(bias, np.float64)[None, :]


def _silu_is_sigmoid(a):
    return 1.0 / (1.0 + np.exp(-a))


def _forward_renormalises(x, idx, w, experts, round_h=None):
    return oracle.moe_forward(x, idx, w / w.sum(axis=1, keepdims=True), experts, round_h)


def _silu_sign(a):
    return a / (1.0 + np.exp(a))


def _no_bias(x, w_g, bias=None):
    return oracle.router_logits(x, w_g, None)


MUTANTS = {
    "no_renormalisation": dict(topk_route=_no_renorm),
    "select_smallest": dict(topk_route=_smallest),
    "ties_to_higher_index": dict(topk_route=_ties_high),
    "gate_up_swapped": dict(swiglu_expert=_swap_gate_up),
    "down_transposed": dict(swiglu_expert=_down_transposed),
    "f_over_T_times_k": dict(aux_stats=_f_over_tk),
    "loss_without_E": dict(aux_stats=_loss_no_E),
    "dispatch_unstable": dict(dispatch=_dispatch_desc),
    "ec_softmax_over_experts": dict(expert_choice_route=_ec_softmax_over_experts),
    "forward_ignores_weights": dict(moe_forward=_forward_unweighted),
    "silu_sign": dict(silu=_silu_sign),
    "bias_dropped": dict(router_logits=_no_bias),
    "unrenormalised_flag_ignored": dict(topk_route=_always_renormalise),
    "fraction_convention_over_T": dict(aux_stats_fraction=_fraction_over_T),
    "capacity_without_k": dict(capacity_route=_capacity_without_k),
    "capacity_last_tokens_first": dict(capacity_route=_capacity_last_tokens_first),
    "capacity_kept_not_renormalised": dict(capacity_route=_capacity_no_renorm),
    "z_loss_not_squared": dict(router_z_loss=_z_loss_unsquared),
    "z_loss_max_instead_of_logsumexp": dict(router_z_loss=_z_loss_max_only),
    "softmax_without_max_subtraction": dict(softmax=_softmax_no_max),
    "ec_capacity_rounded_up": dict(expert_choice_capacity=_ec_capacity_ceil),
    "token_capacity_rounded_up": dict(token_capacity=_token_capacity_ceil),
    "ec_ties_to_higher_token": dict(expert_choice_route=_ec_ties_to_higher_token),
    "ec_combine_renormalised": dict(expert_choice_forward=_ec_combine_renormalised),
    "ec_combine_ignores_scores": dict(expert_choice_forward=_ec_combine_unweighted),
    "dispatch_offsets_inclusive": dict(dispatch=_dispatch_offsets_inclusive),
    "bf16_round_truncates": dict(bf16_round=_bf16_truncates),
    "dense_mixture_uniform": dict(dense_mixture=_dense_uniform),
    "p_from_combine_weights": dict(aux_stats=_p_from_combine_weights),
    "forward_last_slot_only": dict(moe_forward=_forward_last_slot_only),
    "router_experts_reversed": dict(router_logits=_experts_reversed),
    "z_loss_summed_not_averaged": dict(router_z_loss=_z_loss_summed),
    "z_loss_without_the_max_added_back": dict(router_z_loss=_z_loss_without_max_back),
    "fraction_loss_without_E": dict(aux_stats_fraction=_fraction_loss_without_E),
    "topk_slots_ascending": dict(topk_route=_topk_slots_ascending),
    "dispatch_perm_and_inverse_swapped": dict(dispatch=_dispatch_perm_inv_swapped),
    "ec_pos_without_segment_start": dict(expert_choice_route=_ec_pos_local),
    "ec_picks_ascending": dict(expert_choice_route=_ec_picks_ascending),
    "glu_without_silu": dict(swiglu_expert=_glu_without_silu),
    "capacity_load_counts_drops": dict(capacity_route=_capacity_load_counts_drops),
    "capacity_weights_of_all_slots": dict(capacity_route=_capacity_weights_of_all_slots),
    "p_divided_by_k": dict(aux_stats=_p_over_k),
    "bias_subtracted": dict(router_logits=_bias_subtracted),
    "silu_is_sigmoid": dict(silu=_silu_is_sigmoid),
    "forward_renormalises_weights": dict(moe_forward=_forward_renormalises),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name):
    orc = _mutant(**MUTANTS[name])
    caught = []
    for pin in PINS:
        try:
            pin(orc)
        except Exception:  # noqa: BLE001 - any failure of a pin counts as caught
            caught.append(pin.__name__)
    assert caught, f"no pin catches the planted mistake {name}"
