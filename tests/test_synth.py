"""The seeded input generator: reproducible, one stream per tensor (weights do not
depend on T), the value distributions and shapes of the workload table, and exact
storage in bf16 or fp32."""

import math

import numpy as np
import pytest

from sparse_mixture_experts_67_b300 import synth


def test_reproducible_and_seed_dependent():
    cfg = synth.small_config("rep", 40, 64, 32, 4, 2, "bf16", seed=9)
    a, b = synth.make_inputs(cfg), synth.make_inputs(cfg)
    for name in ("x", "w_g", "w_gate", "w_up", "w_down"):
        np.testing.assert_array_equal(getattr(a, name), getattr(b, name))
    other = synth.make_inputs(synth.small_config("rep", 40, 64, 32, 4, 2, "bf16", seed=10))
    assert not np.array_equal(a.x, other.x) and not np.array_equal(a.w_gate, other.w_gate)


def test_weights_do_not_depend_on_tokens():
    """The large-expert sweep changes T with fixed weights; x of a smaller T is the
    leading rows of a larger one."""
    base = synth.small_config("sweep", 64, 64, 32, 4, 2, "bf16", seed=11)
    small, big = synth.make_inputs(base.with_tokens(16)), synth.make_inputs(base.with_tokens(64))
    for name in ("w_g", "w_gate", "w_up", "w_down"):
        np.testing.assert_array_equal(getattr(small, name), getattr(big, name))
    np.testing.assert_array_equal(small.x, big.x[:16])
    assert base.with_tokens(16).with_tokens(32).name == "sweep@T32"


def test_tensors_use_distinct_streams():
    cfg = synth.small_config("streams", 64, 64, 64, 3, 1, "f32", seed=12, x_std=1.0, w_std=1.0,
                             wg_std=1.0)
    inp = synth.make_inputs(cfg)
    blocks = [inp.x[:64], inp.w_g[:3]] + [w[e][:64] for e in range(3)
                                         for w in (inp.w_gate, inp.w_up, inp.w_down)]
    flat = [b.ravel()[:192] for b in blocks]
    for i in range(len(flat)):
        for j in range(i + 1, len(flat)):
            assert not np.array_equal(flat[i], flat[j])


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_value_distribution(dtype):
    cfg = synth.small_config("dist", 512, 256, 128, 4, 2, dtype, seed=13, x_std=0.5, w_std=0.02,
                             wg_std=0.1)
    inp = synth.make_inputs(cfg)
    for arr, std in ((inp.x, 0.5), (inp.w_g, 0.1), (inp.w_gate, 0.02), (inp.w_up, 0.02),
                     (inp.w_down, 0.02)):
        v = synth.to_f64(arr)
        n = v.size
        assert abs(v.mean()) < 5 * std / math.sqrt(n)
        assert abs(v.std() / std - 1.0) < 5 / math.sqrt(2 * n) + (4e-3 if dtype == "bf16" else 0)
    store = np.uint16 if dtype == "bf16" else np.float32
    assert inp.x.dtype == store and inp.w_down.dtype == store


def test_bf16_storage_is_the_rounded_fp32_draw():
    """bf16 tensors are the fp32 draws rounded once to nearest: within half a unit in
    the last place (2^-8 relative) and exactly representable."""
    f = synth.small_config("round", 32, 64, 16, 2, 1, "f32", seed=14)
    b = synth.small_config("round", 32, 64, 16, 2, 1, "bf16", seed=14)
    x32, x16 = synth.make_x(f).astype(np.float64), synth.to_f64(synth.make_x(b))
    assert np.all(np.abs(x16 - x32) <= np.abs(x32) * 2.0 ** -8)
    bits = synth.round_to_bf16_bits(x16.astype(np.float32))
    np.testing.assert_array_equal(synth.to_f64(bits), x16)


def test_workload_table():
    c = synth.CONFIGS
    assert (c["tiny_fp32"].T, c["tiny_fp32"].d, c["tiny_fp32"].F, c["tiny_fp32"].E,
            c["tiny_fp32"].k, c["tiny_fp32"].dtype) == (256, 64, 128, 8, 2, "f32")
    top2 = c["top2_d1024"]
    assert (top2.T, top2.d, top2.F, top2.E, top2.k, top2.dtype) == (8192, 1024, 4096, 8, 2, "bf16")
    assert top2.R == 16384
    assert top2.active_flops() == 6.0 * 16384 * 1024 * 4096 + 2.0 * 8192 * 1024 * 8
    big = c["large_d4096"]
    assert (big.d, big.F, big.E, big.k) == (4096, 14336, 8, 2)
    assert synth.LARGE_T_SWEEP == (16, 256, 4096, 16384)
    fine = c["fine_e64"]
    assert (fine.T, fine.d, fine.F, fine.E, fine.k, fine.bias) == (16384, 2048, 1408, 64, 4, "zipf")
    ec = c["ec_e16"]
    assert ec.routing == "expert_choice" and (ec.T, ec.E, ec.capacity_factor) == (8192, 16, 2.0)
    assert ec.C == 1024 and ec.R == 16384
    seeds = [cfg.seed for cfg in c.values()]
    assert len(set(seeds)) == len(seeds)


def test_router_bias_recipes():
    fine = synth.CONFIGS["fine_e64"]
    b = synth.router_bias(fine)
    assert b.dtype == np.float32 and b.shape == (64,)
    assert b[0] == 0.0
    np.testing.assert_allclose(b.astype(np.float64), -1.5 * np.log(np.arange(1, 65)), rtol=1e-6)
    assert np.all(np.diff(b) < 0)  # strictly decreasing popularity
    forced = synth.router_bias(synth.CONFIGS["fine_e64_forced_empty"])
    assert forced[0] == 3.0 and np.all(forced[1:48] == 0.0) and np.all(forced[48:] == -1.0e4)
    assert synth.router_bias(synth.CONFIGS["top2_d1024"]) is None
