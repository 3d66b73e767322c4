"""GPU parity: the CUDA path through the C ABI against the fp64 oracle.

Every case draws seeded inputs from the synthetic generator, runs the library
on the device and compares with the oracle element by element: routing and
dispatch integers bit-exactly (given the device's own logits, so both sides
decide in the same precision), floating outputs within the stated tolerances.
"""

import zlib

import numpy as np
import pytest

import oracle
from sparse_mixture_experts_67_b300 import synth
from helpers import (assert_close_output, cached_inputs, check_routing_agreement, dev_weights,
                     require_gpu, to_dev)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    return require_gpu()


@pytest.fixture(scope="module")
def moe(torch):
    import sparse_mixture_experts_67_b300 as m

    m.moe_device_error(clear=True)
    yield m
    assert m.moe_device_error(clear=True) == 0, "a kernel gave up on a barrier wait"


def _np(t):
    return t.detach().cpu().numpy()


ROUTER_CASES = [
    # name, T, d, E, k, dtype, bias
    ("tiny_fp32", 256, 64, 8, 2, "f32", None),
    ("ragged_bf16_e8", 200, 128, 8, 2, "bf16", None),
    ("zipf_bf16_e64", 130, 256, 64, 4, "bf16", "zipf"),
    ("wide_bf16_e256", 100, 64, 256, 8, "bf16", None),
    ("odd_bf16_e10", 77, 128, 10, 3, "bf16", None),
    ("dense_bf16_e5", 64, 64, 5, 5, "bf16", None),
    ("single_f32_e1", 33, 16, 1, 1, "f32", None),
    ("one_token_f32", 1, 8, 4, 2, "f32", None),
    ("wide_f32_e200", 100, 64, 200, 4, "f32", None),
    # several 128-token CTAs of the tensor-core router, ragged last CTA and dispatch tile
    ("multi_bf16_e16", 1000, 512, 16, 2, "bf16", None),
    ("multi_bf16_e64", 1000, 512, 64, 4, "bf16", "zipf"),
    ("multi_bf16_e128", 333, 256, 128, 6, "bf16", None),
    # more dispatch tiles per CTA than one MMA tile holds (625 tiles over 148 CTAs: 4 or
    # 5 each), not a multiple of it: a CTA's last, shorter MMA tile is loaded as one box
    # per dispatch tile (32 or 64 rows)
    ("rem_bf16_e8", 20000, 128, 8, 2, "bf16", None),
    ("rem_bf16_e64", 40000, 128, 64, 4, "bf16", "zipf"),
    # three MMA tiles per CTA (4 + 4 + 2 or 4 + 4 + 3 dispatch tiles, the last one
    # shorter): up to 16 experts both epilogue warp groups run, each over two accumulator
    # phases
    ("many_bf16_e5", 50000, 64, 5, 2, "bf16", None),
    ("many_bf16_e16", 45000, 128, 16, 4, "bf16", None),
    # more than 8 picks (the kernels hold the first 8 weights in registers and
    # rescale the rest in memory): one-warp rows, two-warp rows, wide rows, fp32
    ("k12_bf16_e16", 300, 64, 16, 12, "bf16", None),
    ("k10_bf16_e64", 500, 128, 64, 10, "bf16", "zipf"),
    ("k12_bf16_e256", 300, 64, 256, 12, "bf16", None),
    ("k9_f32_e12", 200, 32, 12, 9, "f32", None),
    # one token; one expert; long token ranges (126-127 dispatch tiles per CTA: each
    # epilogue warp group cycles its accumulator through 16 MMA tiles)
    # 17-32 experts (8 columns per epilogue warp) and a wide row with padding columns
    ("e24_bf16", 700, 128, 24, 3, "bf16", "zipf"),
    ("e100_bf16", 600, 64, 100, 5, "bf16", None),
    ("one_token_bf16_e8", 1, 64, 8, 2, "bf16", None),
    ("single_bf16_e1", 40, 64, 1, 1, "bf16", None),
    ("long_bf16_e8", 600000, 64, 8, 2, "bf16", None),
    ("long_bf16_e64", 300000, 64, 64, 4, "bf16", "zipf"),
]


@pytest.mark.parametrize("router", ["auto", "warp_mma", "tcgen05"])
@pytest.mark.parametrize("case", ROUTER_CASES, ids=[c[0] for c in ROUTER_CASES])
def test_router_parity(moe, torch, case, router, monkeypatch):
    name, T, d, E, k, dt, bias = case
    if router != "auto":
        if dt != "bf16":
            pytest.skip("the bf16 routers only")
        monkeypatch.setenv("MOE_ROUTER_TC", "1" if router == "tcgen05" else "0")
    cfg = synth.small_config(name, T, d, 64, E, k, dt, seed=zlib.crc32(name.encode()) % 1000, wg_std=0.1,
                             bias="zipf" if bias else "none")
    x, w_g, b = synth.make_x(cfg), synth.make_router_weight(cfg), synth.router_bias(cfg)
    out = moe.moe_route(to_dev(x), to_dev(w_g), None if b is None else to_dev(b), k,
                        want_logits=True, want_probs=True, want_aux=True)
    torch.cuda.synchronize()
    x64, wg64 = synth.to_f64(x), synth.to_f64(w_g)
    s_ref = oracle.router_logits(x64, wg64, b)
    s_gpu = _np(out["logits"]).astype(np.float64)
    bound = 1e-5 * (np.abs(x64) @ np.abs(wg64).T) + 1e-6
    assert np.all(np.abs(s_gpu - s_ref) <= bound), "router logits outside the fp32 accumulation bound"
    # same-precision decision: the oracle's selection on the device's logits
    idx_ref, w_ref, g_ref = oracle.topk_route(s_gpu, k)
    np.testing.assert_array_equal(_np(out["topk_idx"]), idx_ref)
    np.testing.assert_allclose(_np(out["topk_w"]), w_ref, rtol=0, atol=2e-6)
    np.testing.assert_allclose(_np(out["probs"]), g_ref, rtol=0, atol=2e-6)
    np.testing.assert_allclose(_np(out["topk_w"]).sum(axis=1), 1.0, rtol=0, atol=3e-6)
    # end to end against fp64 logits: only near-ties may differ
    idx64, _, g64 = oracle.topk_route(s_ref, k)
    check_routing_agreement(_np(out["topk_idx"]), idx64, g64)
    # aux statistics from the router's partial sums
    counts_ref, f_ref, p_ref, loss_ref = oracle.aux_stats(g_ref, idx_ref, E)
    counts = torch.from_numpy(counts_ref.astype(np.int32)).cuda()
    aux = moe.moe_aux_loss(counts, T, k, aux_partials=out["aux_partials"])
    torch.cuda.synchronize()
    np.testing.assert_allclose(_np(aux["f"]), f_ref, rtol=1e-7, atol=0)
    np.testing.assert_allclose(_np(aux["p"]), p_ref, rtol=0, atol=2e-6)
    assert abs(float(_np(aux["loss"])[0]) - loss_ref) <= 1e-5 * max(1.0, loss_ref)
    f_frac_ref, loss_frac_ref = oracle.aux_stats_fraction(g_ref, idx_ref, E)
    np.testing.assert_allclose(_np(aux["f_frac"]), f_frac_ref, rtol=1e-7, atol=0)
    auxz = moe.moe_aux_loss(counts, T, k, aux_partials=out["aux_partials"],
                            z_partials=out["z_partials"])
    torch.cuda.synchronize()
    z_ref = oracle.router_z_loss(s_gpu)
    assert abs(float(_np(auxz["z_loss"])[0]) - z_ref) <= 1e-5 * max(1.0, z_ref)
    assert abs(float(_np(aux["loss_frac"])[0]) - loss_frac_ref) <= 1e-5 * max(1.0, loss_frac_ref)
    aux2 = moe.moe_aux_loss(counts, T, k, probs=out["probs"])
    torch.cuda.synchronize()
    np.testing.assert_allclose(_np(aux2["p"]), p_ref, rtol=0, atol=2e-6)
    # without renormalisation: same selection, the selected probabilities as weights
    out_n = moe.moe_route(to_dev(x), to_dev(w_g), None if b is None else to_dev(b), k,
                          want_logits=True, renormalize=False)
    torch.cuda.synchronize()
    idx_n, w_n, _ = oracle.topk_route(_np(out_n["logits"]).astype(np.float64), k, renormalize=False)
    np.testing.assert_array_equal(_np(out_n["topk_idx"]), idx_n)
    np.testing.assert_allclose(_np(out_n["topk_w"]), w_n, rtol=0, atol=2e-6)


PERMUTE_CASES = [
    # name, T, d, E, k, dtype, idx pattern
    ("random_e8_bf16", 1000, 64, 8, 2, "bf16", "random"),
    ("random_e64_k4", 3000, 128, 64, 4, "bf16", "random"),
    ("skewed_e64_empty", 2500, 64, 64, 4, "bf16", "skewed"),
    ("all_to_one", 700, 64, 8, 1, "bf16", "one"),
    ("multi_tile_e256", 5000, 64, 256, 2, "bf16", "random"),
    ("fp32_e8", 333, 16, 8, 2, "f32", "random"),
    # tiles^2 * E above the fused scan's bound (a tile holds 32 tokens for E <= 16, else
    # 64), so the one-CTA scan writes the per-tile bases: 1, 2, 4 and 8 experts per lane,
    # packed rows for E <= 16 (5, 8), one row per step for E = 24
    ("separate_scan_e64", 200000, 64, 64, 4, "bf16", "random"),
    ("separate_scan_e8", 300000, 64, 8, 2, "bf16", "skewed"),
    ("separate_scan_e5", 250000, 64, 5, 1, "bf16", "random"),
    ("separate_scan_e24", 60000, 32, 24, 2, "f32", "random"),
    ("separate_scan_e100", 30000, 64, 100, 2, "bf16", "skewed"),
    ("separate_scan_e256", 20000, 64, 256, 2, "bf16", "random"),
]


def _idx_pattern(rng, T, E, k, kind):
    if kind == "one":
        return np.full((T, k), 3 % E, np.int32)
    if kind == "skewed":
        p = 1.0 / (np.arange(E) + 1.0) ** 2
        p[40:] = 0
        p /= p.sum()
        return np.stack([rng.choice(E, size=k, replace=False, p=p) for _ in range(T)]).astype(np.int32)
    return np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)]).astype(np.int32)


@pytest.mark.parametrize("case", PERMUTE_CASES, ids=[c[0] for c in PERMUTE_CASES])
def test_permute_bit_exact(moe, torch, case):
    name, T, d, E, k, dt, kind = case
    rng = np.random.default_rng(zlib.crc32(name.encode()))
    idx = _idx_pattern(rng, T, E, k, kind)
    cfg = synth.small_config(name, T, d, 64, E, k, dt, seed=5)
    x = synth.make_x(cfg)
    out = moe.moe_permute(to_dev(x), torch.from_numpy(idx).cuda(), E)
    torch.cuda.synchronize()
    counts, offsets, perm, inv_perm = oracle.dispatch(idx.astype(np.int64), E)
    np.testing.assert_array_equal(_np(out["counts"]), counts)
    np.testing.assert_array_equal(_np(out["offsets"]), offsets)
    np.testing.assert_array_equal(_np(out["perm"]), perm)
    np.testing.assert_array_equal(_np(out["inv_perm"]), inv_perm)
    xp = _np(out["x_perm"].view(torch.int16) if dt == "bf16" else out["x_perm"])
    ref = x.view(np.int16)[perm // k] if dt == "bf16" else x[perm // k]
    np.testing.assert_array_equal(xp, ref)


EXPERT_CASES = [
    # name, counts per expert, d, F, dtype
    ("bf16_ragged", [130, 0, 1, 257, 64, 500, 3, 0], 128, 256, "bf16"),
    ("bf16_one_expert", [300], 64, 192, "bf16"),
    ("bf16_e64_skew", [400 // (e + 1) for e in range(64)], 128, 128, "bf16"),
    ("f32_ragged", [70, 0, 5, 131], 64, 128, "f32"),
    # 197 row blocks on <= 148 CTAs: the down GEMM splits its last partial wave
    ("bf16_tail_split", [20000, 5000], 256, 128, "bf16"),
]


@pytest.mark.parametrize("tile_n", ["auto", "64", "128", "256"])
@pytest.mark.parametrize("case", EXPERT_CASES, ids=[c[0] for c in EXPERT_CASES])
def test_grouped_experts_parity(moe, torch, case, tile_n, monkeypatch):
    name, cnts, d, F, dt = case
    if tile_n != "auto":
        if dt != "bf16":
            pytest.skip("tile width applies to the tensor-core path")
        monkeypatch.setenv("MOE_GROUPED_TILE_N", tile_n)
    E = len(cnts)
    R = int(sum(cnts))
    cfg = synth.small_config(name, R, d, F, E, 1, dt, seed=11, x_std=1.0, w_std=0.05)
    inp = synth.make_inputs(cfg)
    offsets = np.concatenate([[0], np.cumsum(cnts)]).astype(np.int32)
    w = dev_weights(inp)
    y_perm, h = moe.moe_experts_swiglu(to_dev(inp.x), torch.from_numpy(offsets).cuda(), w["w_gate"],
                                       w["w_up"], w["w_down"])
    torch.cuda.synchronize()
    x64 = synth.to_f64(inp.x)
    experts = synth.ExpertsF64(inp.w_gate, inp.w_up, inp.w_down)
    y_ref = np.zeros((R, d))
    y_ref_h = np.zeros((R, d))
    for e in range(E):
        lo, hi = offsets[e], offsets[e + 1]
        if hi > lo:
            y_ref[lo:hi] = oracle.swiglu_expert(x64[lo:hi], *experts[e])
            y_ref_h[lo:hi] = oracle.swiglu_expert(x64[lo:hi], *experts[e], round_h=oracle.bf16_round)
    assert_close_output(_np(y_perm), y_ref, dt, f"y_perm[{name}]", ref_bf16_h=y_ref_h if dt == "bf16" else None)


def _run_layer(moe, torch, inp, outputs_spec, renormalize=True):
    cfg = inp.cfg
    w = dev_weights(inp)
    x = to_dev(inp.x)
    outs = {}
    for name, (shape, dtype) in outputs_spec.items():
        outs[name] = torch.empty(shape, dtype=dtype, device="cuda")
    if cfg.routing == "expert_choice":
        y = moe.moe_layer_forward(x, w, k=0, routing=1, capacity_factor=cfg.capacity_factor, outputs=outs)
    else:
        y = moe.moe_layer_forward(x, w, k=cfg.k, outputs=outs, renormalize=renormalize)
    torch.cuda.synchronize()
    return y, outs


def _topk_outputs(torch, cfg):
    T, E, k = cfg.T, cfg.E, cfg.k
    return {"topk_idx": ((T, k), torch.int32), "topk_w": ((T, k), torch.float32),
            "logits": ((T, E), torch.float32), "counts": ((E,), torch.int32),
            "offsets": ((E + 1,), torch.int32), "f": ((E,), torch.float32),
            "p": ((E,), torch.float32), "loss": ((1,), torch.float32),
            "f_frac": ((E,), torch.float32), "loss_frac": ((1,), torch.float32),
            "z_loss": ((1,), torch.float32)}


def _check_topk_layer(moe, torch, cfg, sample=None, renormalize=True):
    inp = cached_inputs(cfg)
    y, outs = _run_layer(moe, torch, inp, _topk_outputs(torch, cfg), renormalize=renormalize)
    x64 = synth.to_f64(inp.x)
    s_gpu = _np(outs["logits"]).astype(np.float64)
    # routing, dispatch and aux: full size, same-precision decisions
    idx_g, w_g, g_g = oracle.topk_route(s_gpu, cfg.k, renormalize=renormalize)
    np.testing.assert_array_equal(_np(outs["topk_idx"]), idx_g)
    np.testing.assert_allclose(_np(outs["topk_w"]), w_g, rtol=0, atol=2e-6)
    counts, offsets, _, _ = oracle.dispatch(idx_g, cfg.E)
    np.testing.assert_array_equal(_np(outs["counts"]), counts)
    np.testing.assert_array_equal(_np(outs["offsets"]), offsets)
    _, f_ref, p_ref, loss_ref = oracle.aux_stats(g_g, idx_g, cfg.E)
    np.testing.assert_allclose(_np(outs["f"]), f_ref, rtol=1e-6, atol=0)
    np.testing.assert_allclose(_np(outs["p"]), p_ref, rtol=0, atol=1e-5)
    assert abs(float(_np(outs["loss"])[0]) - loss_ref) <= 1e-4 * max(1.0, loss_ref)
    f_frac_ref, loss_frac_ref = oracle.aux_stats_fraction(g_g, idx_g, cfg.E)
    np.testing.assert_allclose(_np(outs["f_frac"]), f_frac_ref, rtol=1e-6, atol=0)
    assert abs(float(_np(outs["loss_frac"])[0]) - loss_frac_ref) <= 1e-4 * max(1.0, loss_frac_ref)
    z_ref = oracle.router_z_loss(s_gpu)
    assert abs(float(_np(outs["z_loss"])[0]) - z_ref) <= 1e-5 * max(1.0, z_ref)
    # end-to-end routing against fp64 logits
    s64 = oracle.router_logits(x64, synth.to_f64(inp.w_g), inp.bias)
    idx64, w64, g64 = oracle.topk_route(s64, cfg.k, renormalize=renormalize)
    agree = check_routing_agreement(_np(outs["topk_idx"]), idx64, g64)
    # outputs (sampled at full size) against the fp64 oracle with its own routing
    tokens = np.arange(cfg.T) if sample is None else np.sort(
        np.random.default_rng(cfg.seed).choice(cfg.T, size=min(sample, cfg.T), replace=False))
    tokens = tokens[agree[tokens]]
    experts = synth.ExpertsF64(inp.w_gate, inp.w_up, inp.w_down)
    y_ref = oracle.moe_forward(x64[tokens], idx64[tokens], w64[tokens], experts)
    y_ref_h = None
    if cfg.dtype == "bf16":
        y_ref_h = oracle.moe_forward(x64[tokens], idx64[tokens], w64[tokens], experts,
                                     round_h=oracle.bf16_round)
    return assert_close_output(_np(y)[tokens], y_ref, cfg.dtype, what=f"y[{cfg.name}]",
                               ref_bf16_h=y_ref_h)


def test_layer_tiny_fp32(moe, torch):
    _check_topk_layer(moe, torch, synth.CONFIGS["tiny_fp32"])


@pytest.mark.parametrize("router", ["auto", "warp_mma", "tcgen05"])
@pytest.mark.parametrize("E,k", [(8, 2), (40, 4)])
def test_layer_small_bf16_multi_tile(moe, torch, E, k, router, monkeypatch):
    """Several router CTAs and dispatch tiles (32 or 64 tokens per tile, four or two per
    tensor-core router CTA) with a ragged last one, through the whole layer."""
    if router != "auto":
        monkeypatch.setenv("MOE_ROUTER_TC", "1" if router == "tcgen05" else "0")
    cfg = synth.small_config(f"small_bf16_e{E}", 1000, 256, 384, E, k, "bf16", seed=21 + E,
                             x_std=1.0, w_std=0.02, wg_std=0.1)
    _check_topk_layer(moe, torch, cfg)


@pytest.mark.parametrize("E,k,T", [(8, 2, 20000), (64, 4, 40000)])
def test_layer_tensor_core_router_short_last_tiles(moe, torch, E, k, T, monkeypatch):
    """The tensor-core router with four or five dispatch tiles per CTA (MMA tiles of four
    or two, then a shorter one loaded as one box per dispatch tile), through the dispatch
    counts, the aux statistics and the whole layer."""
    monkeypatch.setenv("MOE_ROUTER_TC", "1")
    cfg = synth.small_config(f"short_tiles_e{E}", T, 128, 128, E, k, "bf16", seed=70 + E,
                             x_std=1.0, w_std=0.05, wg_std=0.1, bias="zipf" if E > 16 else "none")
    _check_topk_layer(moe, torch, cfg)


@pytest.mark.parametrize("E,k,router", [(256, 8, "auto"), (64, 10, "auto"), (256, 8, "warp_mma")])
def test_layer_most_experts_and_picks(moe, torch, E, k, router, monkeypatch):
    """The largest expert count the library takes (E = 256, wide router rows read in
    32-column chunks, 256 expert segments) and more than 8 picks per token, through
    the whole layer and the separate combine."""
    if router != "auto":
        monkeypatch.setenv("MOE_ROUTER_TC", "0")
    cfg = synth.small_config(f"most_e{E}_k{k}", 3000, 128, 128, E, k, "bf16", seed=80 + E + k,
                             x_std=1.0, w_std=0.05, wg_std=0.1)
    _check_topk_layer(moe, torch, cfg)


@pytest.mark.parametrize("E,k", [(8, 2), (16, 4), (40, 1)])
def test_layer_without_renormalisation(moe, torch, E, k):
    """MOE_ROUTE_NO_RENORM: the combine weights are the selected probabilities themselves
    (fused down+combine for k <= 2, the separate combine above; both routers)."""
    cfg = synth.small_config(f"norenorm_e{E}", 900, 256, 384, E, k, "bf16", seed=40 + E, x_std=1.0,
                             w_std=0.02, wg_std=0.1)
    _check_topk_layer(moe, torch, cfg, renormalize=False)


@pytest.mark.parametrize("E,k,cf", [(8, 2, 1.0), (16, 4, 0.8), (8, 1, 0.5), (6, 2, 0.001)],
                         ids=["e8_k2_fused", "e16_k4", "e8_k1_heavy", "capacity_zero"])
def test_layer_capacity_limited(moe, torch, E, k, cf):
    """MOE_ROUTE_CAPACITY against the oracle's capacity_route on the device logits: the
    selection, the kept segments, the drop count, the kept-renormalised weights and y
    (the fused down+combine for k <= 2, the separate combine above; all dropped at cf 0.001)."""
    cfg = synth.small_config(f"cap_e{E}_k{k}", 1000, 256, 384, E, k, "bf16", seed=50 + E + k,
                             x_std=1.0, w_std=0.02, wg_std=0.1, bias="zipf")
    inp = cached_inputs(cfg)
    w = dev_weights(inp)
    x = to_dev(inp.x)
    T = cfg.T
    outs = {"topk_idx": torch.empty((T, k), dtype=torch.int32, device="cuda"),
            "topk_w": torch.empty((T, k), dtype=torch.float32, device="cuda"),
            "logits": torch.empty((T, E), dtype=torch.float32, device="cuda"),
            "counts": torch.empty((E,), dtype=torch.int32, device="cuda"),
            "offsets": torch.empty((E + 1,), dtype=torch.int32, device="cuda"),
            "dropped": torch.full((1,), -7, dtype=torch.int32, device="cuda")}
    y = moe.moe_layer_forward(x, w, k=k, capacity_factor=cf, outputs=outs, capacity=True)
    torch.cuda.synchronize()
    s_gpu = _np(outs["logits"]).astype(np.float64)
    cf32 = float(np.float32(cf))
    idx_g, w_cap, kept, dropped, load, cap = oracle.capacity_route(s_gpu, k, cf32)
    np.testing.assert_array_equal(_np(outs["topk_idx"]), idx_g)
    np.testing.assert_array_equal(_np(outs["counts"]), np.bincount(idx_g.ravel(), minlength=E))
    np.testing.assert_array_equal(_np(outs["offsets"]), np.concatenate([[0], np.cumsum(load)]))
    assert int(_np(outs["dropped"])[0]) == dropped
    if cf >= 0.5:
        assert dropped > 0  # the capacity binds on these inputs
    np.testing.assert_allclose(_np(outs["topk_w"]), w_cap, rtol=0, atol=2e-6)
    x64 = synth.to_f64(inp.x)
    experts = synth.ExpertsF64(inp.w_gate, inp.w_up, inp.w_down)
    y_ref = oracle.moe_forward(x64, idx_g, w_cap, experts)
    y_ref_h = oracle.moe_forward(x64, idx_g, w_cap, experts, round_h=oracle.bf16_round)
    if dropped == T * k:
        assert np.all(_np(y) == 0)
    else:
        assert_close_output(_np(y), y_ref, "bf16", what=f"y[{cfg.name}]", ref_bf16_h=y_ref_h)


def test_layer_capacity_separate_scan(moe, torch):
    """Capacity-limited top-2 over 64 experts at T = 20000: 313 router tiles of 128
    assignments, so 313^2 * 64 reads send the counts through the one-CTA scan, which
    applies the capacity to the segment bases.  Routing outputs are checked whole, y
    on every 8th token (the oracle's tokens are independent)."""
    E, k, cf = 64, 2, 0.8
    cfg = synth.small_config("cap_scan_e64", 20000, 256, 384, E, k, "bf16", seed=77, x_std=1.0,
                             w_std=0.02, wg_std=0.1, bias="zipf")
    inp = cached_inputs(cfg)
    w = dev_weights(inp)
    x = to_dev(inp.x)
    T = cfg.T
    outs = {"topk_idx": torch.empty((T, k), dtype=torch.int32, device="cuda"),
            "topk_w": torch.empty((T, k), dtype=torch.float32, device="cuda"),
            "logits": torch.empty((T, E), dtype=torch.float32, device="cuda"),
            "counts": torch.empty((E,), dtype=torch.int32, device="cuda"),
            "offsets": torch.empty((E + 1,), dtype=torch.int32, device="cuda"),
            "dropped": torch.full((1,), -7, dtype=torch.int32, device="cuda")}
    y = moe.moe_layer_forward(x, w, k=k, capacity_factor=cf, outputs=outs, capacity=True)
    torch.cuda.synchronize()
    s_gpu = _np(outs["logits"]).astype(np.float64)
    idx_g, w_cap, kept, dropped, load, cap = oracle.capacity_route(s_gpu, k, float(np.float32(cf)))
    np.testing.assert_array_equal(_np(outs["topk_idx"]), idx_g)
    np.testing.assert_array_equal(_np(outs["counts"]), np.bincount(idx_g.ravel(), minlength=E))
    np.testing.assert_array_equal(_np(outs["offsets"]), np.concatenate([[0], np.cumsum(load)]))
    assert int(_np(outs["dropped"])[0]) == dropped and dropped > 0
    np.testing.assert_allclose(_np(outs["topk_w"]), w_cap, rtol=0, atol=2e-6)
    sub = np.arange(0, T, 8)
    x64 = synth.to_f64(inp.x)[sub]
    experts = synth.ExpertsF64(inp.w_gate, inp.w_up, inp.w_down)
    y_ref = oracle.moe_forward(x64, idx_g[sub], w_cap[sub], experts)
    y_ref_h = oracle.moe_forward(x64, idx_g[sub], w_cap[sub], experts, round_h=oracle.bf16_round)
    assert_close_output(_np(y)[sub], y_ref, "bf16", what="y[cap_scan_e64]", ref_bf16_h=y_ref_h)


@pytest.mark.slow
def test_layer_top2_d1024(moe, torch):
    """Every token's output of the top-2 d=1024 workload against the fp64 oracle."""
    _check_topk_layer(moe, torch, synth.CONFIGS["top2_d1024"])


@pytest.mark.slow
def test_layer_fine_e64(moe, torch):
    """Every token's output of the fine-grained E=64 top-4 workload (Zipf bias)."""
    _check_topk_layer(moe, torch, synth.CONFIGS["fine_e64"])


@pytest.mark.slow
def test_layer_fine_e64_forced_empty(moe, torch):
    """Every token's output with experts 48..63 empty and expert 0 overfull."""
    _check_topk_layer(moe, torch, synth.CONFIGS["fine_e64_forced_empty"])


@pytest.mark.slow
@pytest.mark.parametrize("T", synth.LARGE_T_SWEEP)
def test_layer_large_d4096(moe, torch, T):
    """The large layer: every token up to T=256; above, a fixed seeded sample of 1024
    tokens (routing, counts and offsets still at full size)."""
    cfg = synth.CONFIGS["large_d4096"].with_tokens(T)
    _check_topk_layer(moe, torch, cfg, sample=None if T <= 256 else 1024)


def _check_ec_layer(moe, torch, cfg):
    inp = cached_inputs(cfg)
    C = cfg.C
    spec = {"logits": ((cfg.T, cfg.E), torch.float32), "ec_idx": ((cfg.E, C), torch.int32),
            "ec_score": ((cfg.E, C), torch.float32), "pos": ((cfg.E, cfg.T), torch.int32)}
    y, outs = _run_layer(moe, torch, inp, spec)
    s_gpu = _np(outs["logits"]).astype(np.float64)
    C_ref, idx_g, sc_g, pos_g = oracle.expert_choice_route(s_gpu, cfg.capacity_factor)
    assert C_ref == C
    np.testing.assert_array_equal(_np(outs["ec_idx"]), idx_g)
    np.testing.assert_array_equal(_np(outs["pos"]), pos_g)
    np.testing.assert_allclose(_np(outs["ec_score"]), sc_g, rtol=1e-5, atol=1e-9)
    x64 = synth.to_f64(inp.x)
    s64 = oracle.router_logits(x64, synth.to_f64(inp.w_g), inp.bias)
    _, idx64, sc64, _ = oracle.expert_choice_route(s64, cfg.capacity_factor)
    # selections may differ from fp64 only at near-ties of the per-expert scores
    for e in range(cfg.E):
        a, b = set(_np(outs["ec_idx"])[e].tolist()), set(idx64[e].tolist())
        if a != b:
            col = oracle.softmax(s64[:, e])
            for t1 in a - b:
                for t2 in b - a:
                    assert abs(col[t1] - col[t2]) < 1e-6
    experts = synth.ExpertsF64(inp.w_gate, inp.w_up, inp.w_down)
    y_ref = oracle.expert_choice_forward(x64, idx64, sc64, experts)
    y_ref_h = None
    if cfg.dtype == "bf16":
        y_ref_h = oracle.expert_choice_forward(x64, idx64, sc64, experts, round_h=oracle.bf16_round)
    return assert_close_output(_np(y), y_ref, cfg.dtype, what=f"y[{cfg.name}]", ref_bf16_h=y_ref_h)


@pytest.mark.parametrize("launches", ["one", "two"])
def test_layer_small_expert_choice(moe, torch, launches, monkeypatch):
    """The select as one cooperative launch (slices wait for their expert's other slices)
    and as two launches."""
    monkeypatch.setenv("MOE_EC_TWO_LAUNCHES", "1" if launches == "two" else "0")
    cfg = synth.LayerConfig("small_ec", T=500, d=128, F=256, E=6, k=0, dtype="bf16", x_std=1.0,
                            w_std=0.05, wg_std=0.1, seed=31, routing="expert_choice",
                            capacity_factor=1.5)
    _check_ec_layer(moe, torch, cfg)


def test_layer_expert_choice_fp32(moe, torch):
    cfg = synth.LayerConfig("small_ec32", T=300, d=32, F=64, E=4, k=0, dtype="f32", x_std=0.5,
                            w_std=0.05, wg_std=0.1, seed=32, routing="expert_choice",
                            capacity_factor=1.0)
    _check_ec_layer(moe, torch, cfg)


@pytest.mark.parametrize("T,E,cf", [(6000, 2, 1.0), (40, 4, 2.0), (40, 4, 1.0), (2000, 3, 1.7)],
                         ids=["C3000_several_per_thread", "C20", "C10", "C1133"])
def test_layer_expert_choice_capacities(moe, torch, T, E, cf):
    """Capacities below a warp, between a warp and the CTA, and above the CTA's thread
    count (several sorted picks per thread), through the whole layer."""
    cfg = synth.LayerConfig(f"ec_T{T}_E{E}", T=T, d=64, F=64, E=E, k=0, dtype="bf16", x_std=1.0,
                            w_std=0.05, wg_std=0.1, seed=34, routing="expert_choice",
                            capacity_factor=cf)
    _check_ec_layer(moe, torch, cfg)


@pytest.mark.parametrize("launches", ["one", "two"])
@pytest.mark.parametrize("T,E,cf", [(32768, 16, 2.0), (5000, 8, 1.0)], ids=["T32768_C4096", "T5000_C625"])
def test_layer_expert_choice_many_slices(moe, torch, T, E, cf, launches, monkeypatch):
    """Token counts beyond one 1024-token slice per expert: 32 slices whose candidate
    lists are searched in global memory (too large to stage), and a capacity below the
    slice length with a ragged last slice; one cooperative launch or two."""
    monkeypatch.setenv("MOE_EC_TWO_LAUNCHES", "1" if launches == "two" else "0")
    cfg = synth.LayerConfig(f"ec_T{T}_E{E}", T=T, d=64, F=64, E=E, k=0, dtype="bf16", x_std=1.0,
                            w_std=0.05, wg_std=0.1, seed=36, routing="expert_choice",
                            capacity_factor=cf)
    _check_ec_layer(moe, torch, cfg)


def test_expert_choice_route_exact_ties(moe, torch):
    """Tokens with identical rows tie exactly on every expert's logit: the selection keeps
    the lower token ids and orders equal scores by token, as the oracle does."""
    cfg = synth.small_config("ec_ties", 1200, 64, 64, 5, 1, "bf16", seed=35, wg_std=0.1)
    x = synth.make_x(cfg)
    x = np.ascontiguousarray(np.tile(x[:16], (cfg.T // 16, 1)))  # 16 distinct rows, repeated
    w_g = synth.make_router_weight(cfg)
    cf = 1.25  # exact in fp32: the capacity is floor(T * cf / E) of the fp32 factor
    r = moe.moe_expert_choice_route(to_dev(x), to_dev(w_g), None, cf)
    torch.cuda.synchronize()
    s_gpu = _np(r["logits"]).astype(np.float64)
    C_ref, idx_g, sc_g, pos_g = oracle.expert_choice_route(s_gpu, cf)
    assert C_ref == r["C"]
    np.testing.assert_array_equal(_np(r["ec_idx"]), idx_g)
    np.testing.assert_array_equal(_np(r["pos"]), pos_g)
    np.testing.assert_allclose(_np(r["ec_score"]), sc_g, rtol=1e-5, atol=1e-9)


@pytest.mark.slow
def test_bounded_wait_expiry_reports_and_recovers(moe, torch):
    """A barrier wait that nothing satisfies gives up after its bound: the expert-choice
    selection's cooperative launch, with the arrival counts started far below zero, ends
    within a few seconds with code 16 in the device error word and no picks written, and
    the next call on the same context is correct."""
    import time
    moe.moe_device_error(clear=True)
    t0 = time.time()
    moe.moe_selftest_wait_expiry(8192, 16, 2.0)
    elapsed = time.time() - t0
    assert moe.moe_device_error(clear=True) == 16
    assert 0.9 < elapsed < 30.0, elapsed  # the 1 s limit, then every CTA returned
    # the context is still usable
    cfg = synth.LayerConfig("after_expiry", T=3000, d=128, F=256, E=8, k=0, dtype="bf16", x_std=1.0,
                            w_std=0.05, wg_std=0.1, seed=91, routing="expert_choice",
                            capacity_factor=2.0)
    _check_ec_layer(moe, torch, cfg)
    assert moe.moe_device_error(clear=False) == 0


def test_layer_ec_e16(moe, torch):
    _check_ec_layer(moe, torch, synth.CONFIGS["ec_e16"])


def test_expert_choice_zero_capacity(moe, torch):
    cfg = synth.LayerConfig("ec_zero", T=10, d=64, F=64, E=4, k=0, dtype="bf16", x_std=1.0,
                            w_std=0.05, wg_std=0.1, seed=33, routing="expert_choice",
                            capacity_factor=0.3)
    assert cfg.C == 0
    inp = synth.make_inputs(cfg)
    y, outs = _run_layer(moe, torch, inp, {"pos": ((cfg.E, cfg.T), torch.int32)})
    assert np.all(_np(y) == 0)
    assert np.all(_np(outs["pos"]) == -1)


def test_layer_dense_limit_and_single_expert(moe, torch):
    for E, k in ((4, 4), (1, 1)):
        cfg = synth.small_config(f"dense{E}", 150, 64, 128, E, k, "f32", seed=40 + E, x_std=1.0,
                                 w_std=0.05)
        _check_topk_layer(moe, torch, cfg)


def test_layer_zero_tokens(moe, torch):
    cfg = synth.small_config("zero", 4, 64, 128, 8, 2, "bf16", seed=3)
    inp = synth.make_inputs(cfg)
    w = dev_weights(inp)
    x = to_dev(inp.x)[:0]
    y = torch.full((0, 64), 7.0, device="cuda")
    moe.moe_layer_forward(x, w, k=2, y=y)
    torch.cuda.synchronize()
    assert y.shape == (0, 64)


@pytest.mark.parametrize("k", [1, 2, 4])
def test_layer_deterministic(moe, torch, k):
    """Bit-identical outputs on repeated runs (k <= 2 combines in the down GEMM with atomics)."""
    cfg = synth.small_config("det", 3000, 128, 256, 16, k, "bf16", seed=50, x_std=1.0, w_std=0.05)
    inp = synth.make_inputs(cfg)
    w = dev_weights(inp)
    x = to_dev(inp.x)
    ys = [moe.moe_layer_forward(x, w, k=k).clone() for _ in range(3)]
    torch.cuda.synchronize()
    assert all(torch.equal(ys[0], yi) for yi in ys[1:])


GATHER_CASES = [
    # name, T, d, F, E, k (0: expert-choice style token ids, div 1)
    ("topk_e8_k2", 700, 128, 256, 8, 2),
    ("topk_e64_k4", 1200, 128, 128, 64, 4),
    ("ec_style_e5", 300, 64, 192, 5, 0),
]


@pytest.mark.parametrize("tile_n", ["auto", "64", "128", "256"])
@pytest.mark.parametrize("case", GATHER_CASES, ids=[c[0] for c in GATHER_CASES])
def test_gateup_gather_against_oracle(moe, torch, case, tile_n, monkeypatch):
    """Gate/up with the row gather inside the GEMM's A load, followed by the down GEMM,
    against the oracle's dispatch and SwiGLU experts on the gathered rows (bf16-H
    max-abs, rel-L2 against pure fp64); it also equals materialising x_perm first, bit
    for bit."""
    name, T, d, F, E, k = case
    if tile_n != "auto":
        monkeypatch.setenv("MOE_GROUPED_TILE_N", tile_n)
    rng = np.random.default_rng(zlib.crc32(name.encode()))
    cfg = synth.small_config(name, T, d, F, E, max(k, 1), "bf16", seed=7, w_std=0.05)
    inp = synth.make_inputs(cfg)
    x = to_dev(inp.x)
    w = dev_weights(inp)
    if k > 0:
        idx = np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)]).astype(np.int32)
        p = moe.moe_permute(x, torch.from_numpy(idx).cuda(), E)
        x_perm, offsets, src, div = p["x_perm"], p["offsets"], p["perm"], k
        _, off_ref, perm_ref, _ = oracle.dispatch(idx.astype(np.int64), E)
        src_rows = perm_ref // k  # token of each dispatch row
    else:
        C = T // 3
        src_np = np.concatenate([rng.choice(T, size=C, replace=False) for _ in range(E)]).astype(np.int32)
        src = torch.from_numpy(src_np).cuda()
        offsets = torch.from_numpy((np.arange(E + 1) * C).astype(np.int32)).cuda()
        x_perm, div = moe.moe_gather_rows(x, src, 1), 1
        off_ref, src_rows = np.arange(E + 1) * C, src_np.astype(np.int64)
    h_gat = moe.moe_grouped_gateup_swiglu_gather(x, src, div, offsets, w["w_gate"], w["w_up"])
    y_gat = moe.moe_grouped_down(h_gat, offsets, w["w_down"])
    h_ref = moe.moe_grouped_gateup_swiglu(x_perm, offsets, w["w_gate"], w["w_up"])
    torch.cuda.synchronize()
    np.testing.assert_array_equal(_np(offsets), off_ref)
    x64 = synth.to_f64(inp.x)
    experts = synth.ExpertsF64(inp.w_gate, inp.w_up, inp.w_down)
    R = int(off_ref[-1])
    y_ref, y_ref_h = np.zeros((R, d)), np.zeros((R, d))
    for e in range(E):
        lo, hi = int(off_ref[e]), int(off_ref[e + 1])
        if hi > lo:
            xr = x64[src_rows[lo:hi]]
            y_ref[lo:hi] = oracle.swiglu_expert(xr, *experts[e])
            y_ref_h[lo:hi] = oracle.swiglu_expert(xr, *experts[e], round_h=oracle.bf16_round)
    assert_close_output(_np(y_gat), y_ref, "bf16", f"gathered y_perm[{name}]", ref_bf16_h=y_ref_h)
    assert torch.equal(h_ref.view(torch.int16), h_gat.view(torch.int16))


@pytest.mark.parametrize("k", [2, 4])
def test_cluster_paths_bit_identical(moe, torch, k, monkeypatch):
    """The 2-CTA pair changes only where operand bytes come from and which SM issues the
    MMA (one M = 256 instruction over both CTAs' rows), never the per-element arithmetic:
    outputs equal the single-CTA path bit for bit.  Row counts leave partial 256-row
    blocks and an expert of < 128 rows."""
    mode = "pair"
    cfg = synth.small_config("pair_layer", 4000, 256, 512, 8, k, "bf16", seed=60, x_std=1.0, w_std=0.05)
    inp = synth.make_inputs(cfg)
    w = dev_weights(inp)
    x = to_dev(inp.x)
    # outputs start as NaN so that a row a path fails to write cannot match
    y_cl = torch.full((cfg.T, cfg.d), float("nan"), dtype=torch.float32, device="cuda")
    y_one = y_cl.clone()
    monkeypatch.setenv("MOE_GROUPED_CLUSTER", mode)
    moe.moe_layer_forward(x, w, k=k, y=y_cl)
    monkeypatch.setenv("MOE_GROUPED_CLUSTER", "none")
    moe.moe_layer_forward(x, w, k=k, y=y_one)
    torch.cuda.synchronize()
    assert not torch.isnan(y_cl).any()
    assert torch.equal(y_cl, y_one)


def test_cluster_paths_grouped_ragged(moe, torch, monkeypatch):
    """The 2-CTA pair form of the separate gate/up and down entry points on ragged
    segments (empty experts, one row, a 128-row half block) against the single-CTA path."""
    mode = "pair"
    cnts = [300, 0, 1, 128, 129, 700, 0, 255]
    d, F = 256, 512
    cfg = synth.small_config("pair_ragged", int(sum(cnts)), d, F, len(cnts), 1, "bf16", seed=61,
                             x_std=1.0, w_std=0.05)
    inp = synth.make_inputs(cfg)
    offsets = torch.from_numpy(np.concatenate([[0], np.cumsum(cnts)]).astype(np.int32)).cuda()
    w = dev_weights(inp)
    x = to_dev(inp.x)
    monkeypatch.setenv("MOE_GROUPED_TILE_N", "256")
    R = int(sum(cnts))
    outs = {}
    for m in (mode, "none"):
        monkeypatch.setenv("MOE_GROUPED_CLUSTER", m)
        # outputs start as NaN so that a row a path fails to write cannot match
        h = torch.full((R, F), float("nan"), dtype=torch.bfloat16, device="cuda")
        yp = torch.full((R, d), float("nan"), dtype=torch.float32, device="cuda")
        moe.moe_grouped_gateup_swiglu(x, offsets, w["w_gate"], w["w_up"], h)
        moe.moe_grouped_down(h, offsets, w["w_down"], yp)
        outs[m] = (h, yp)
    torch.cuda.synchronize()
    (h_cl, yp_cl), (h_one, yp_one) = outs[mode], outs["none"]
    assert not torch.isnan(yp_cl).any()
    assert torch.equal(h_cl.view(torch.int16), h_one.view(torch.int16))
    assert torch.equal(yp_cl, yp_one)


@pytest.mark.parametrize("k", [2, 4])
def test_down_epilogue_forms_bit_identical(moe, torch, k, monkeypatch):
    """The down GEMM's epilogue storing straight from TMEM fragments equals the
    shared-memory-staged form bit for bit: the same fp32 values stored, or (k <= 2, the
    fused combine) the same two additions onto zero per element; ragged segments and a
    split last wave (3000 tokens, 256-column tiles) included."""
    cfg = synth.small_config("down_epi", 3000, 256, 512, 8, k, "bf16", seed=64, x_std=1.0, w_std=0.05)
    inp = synth.make_inputs(cfg)
    w = dev_weights(inp)
    x = to_dev(inp.x)
    outs = {}
    for form in ("frag", "staged"):
        monkeypatch.setenv("MOE_DOWN_EPILOGUE", form)
        y = torch.full((cfg.T, cfg.d), float("nan"), dtype=torch.float32, device="cuda")
        moe.moe_layer_forward(x, w, k=k, y=y)
        outs[form] = y
    torch.cuda.synchronize()
    assert not torch.isnan(outs["frag"]).any()
    assert torch.equal(outs["frag"], outs["staged"])


@pytest.mark.parametrize("k", [2, 4])
def test_programmatic_dependent_launch_bit_identical(moe, torch, k, monkeypatch):
    """With programmatic dependent launch each kernel starts under the tail of the previous
    one but waits for its completion before touching memory: outputs equal the plainly
    stream-ordered launches bit for bit, over back-to-back layer calls."""
    cfg = synth.small_config("pdl", 3000, 256, 512, 8, k, "bf16", seed=62, x_std=1.0, w_std=0.05)
    inp = synth.make_inputs(cfg)
    w = dev_weights(inp)
    x = to_dev(inp.x)
    outs = {}
    for flag in ("0", "1"):
        monkeypatch.setenv("MOE_PDL", flag)
        ys = [torch.full((cfg.T, cfg.d), float("nan"), dtype=torch.float32, device="cuda")
              for _ in range(3)]
        for y in ys:  # back to back on one stream: each call reuses the previous call's buffers
            moe.moe_layer_forward(x, w, k=k, y=y)
        outs[flag] = ys
    torch.cuda.synchronize()
    for y in outs["0"] + outs["1"]:
        assert not torch.isnan(y).any()
        assert torch.equal(y, outs["0"][0])


def test_host_pipeline_matches_batchwise(moe, torch):
    """HostPipeline overlaps each batch's copies with its neighbours' forwards; every output
    equals copying in, running and copying back that batch alone, bit for bit."""
    cfg = synth.small_config("pipe", 700, 256, 384, 8, 2, "bf16", seed=63, x_std=1.0, w_std=0.05)
    inp = synth.make_inputs(cfg)
    w = dev_weights(inp)
    layer = moe.MoELayer(w, k=2)
    rng = np.random.default_rng(5)
    xs = []
    for _ in range(5):
        bits = synth.round_to_bf16_bits(rng.standard_normal((cfg.T, cfg.d)))
        xs.append(torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).pin_memory())
    ys = [torch.full((cfg.T, cfg.d), float("nan"), dtype=torch.float32).pin_memory() for _ in xs]
    pipe = moe.HostPipeline(layer, cfg.T, cfg.d, torch.bfloat16)
    pipe.run(xs, ys)
    torch.cuda.synchronize()
    for xh, yh in zip(xs, ys):
        ref = layer(xh.cuda()).cpu()
        assert torch.equal(yh, ref)
