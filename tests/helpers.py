"""Shared helpers for the GPU parity tests: device upload of seeded inputs,
tolerance checks and cached workloads."""

from __future__ import annotations

import functools

import numpy as np
import pytest

from sparse_mixture_experts_67_b300 import synth

# Tolerances of the layer outputs (stated per precision of x and the weights):
#   bf16 inputs, fp32 accumulation: max-abs 2e-2 and relative L2 1e-2;
#   fp32 path: 1e-5 relative (max-abs error over max |ref|, and relative L2).
BF16_MAX_ABS, BF16_REL_L2 = 2e-2, 1e-2
F32_REL = 1e-5
# routing may differ from the fp64 oracle only where the two probabilities tie
# within this margin
NEAR_TIE = 1e-6


def torch_mod():
    return pytest.importorskip("torch")


def require_gpu():
    torch = torch_mod()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sparse_mixture_experts_67_b300 import build_lib

    build_lib.build()
    return torch


def to_dev(a: np.ndarray):
    torch = torch_mod()
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).cuda()
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def dev_weights(inp: synth.LayerInputs):
    return {"w_g": to_dev(inp.w_g), "bias": None if inp.bias is None else to_dev(inp.bias),
            "w_gate": to_dev(inp.w_gate), "w_up": to_dev(inp.w_up), "w_down": to_dev(inp.w_down)}


@functools.lru_cache(maxsize=2)
def cached_inputs(cfg: synth.LayerConfig) -> synth.LayerInputs:
    return synth.make_inputs(cfg)


def assert_close_output(got: np.ndarray, ref: np.ndarray, dtype: str, what: str = "y",
                        ref_bf16_h: np.ndarray = None):
    """Output tolerance check; returns (max-abs vs ref, rel-L2 vs ref).

    ref is the pure fp64 oracle.  For bf16 inputs the hidden activation H is a
    bf16 tensor (the tensor-core input of the down projection), so the
    max-abs bound is taken against ref_bf16_h, the oracle with H rounded to
    bf16, when given; the relative-L2 bound is always against pure fp64.
    """
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    err = np.abs(got - ref)
    den = np.linalg.norm(ref)
    rel_l2 = np.linalg.norm(got - ref) / den if den > 0 else np.linalg.norm(got - ref)
    if dtype == "bf16":
        err_h = err if ref_bf16_h is None else np.abs(got - np.asarray(ref_bf16_h, np.float64))
        assert err_h.max() <= BF16_MAX_ABS, (
            f"{what}: max-abs {err_h.max():.3e} > {BF16_MAX_ABS} (vs fp64 {err.max():.3e})")
        assert rel_l2 <= BF16_REL_L2, f"{what}: rel-L2 {rel_l2:.3e} > {BF16_REL_L2}"
        print(f"PARITY {what}: max-abs vs fp64 {err.max():.3e}, vs bf16-H oracle {err_h.max():.3e}, "
              f"rel-L2 {rel_l2:.3e} over {got.size} values")
    else:
        scale = max(np.abs(ref).max(), 1e-30)
        assert err.max() <= F32_REL * scale, f"{what}: max-abs {err.max():.3e} > {F32_REL} * {scale:.3e}"
        assert rel_l2 <= F32_REL, f"{what}: rel-L2 {rel_l2:.3e} > {F32_REL}"
        print(f"PARITY {what}: max-abs {err.max():.3e} (max |ref| {scale:.3e}), rel-L2 {rel_l2:.3e} "
              f"over {got.size} values")
    return float(err.max()), float(rel_l2)


def check_routing_agreement(gpu_idx: np.ndarray, ref_idx: np.ndarray, ref_probs: np.ndarray):
    """Top-k sets may differ from the fp64 oracle only at near-ties; returns agreeing token mask."""
    agree = np.all(gpu_idx == ref_idx, axis=1)
    for t in np.nonzero(~agree)[0]:
        g = ref_probs[t]
        gs, rs = set(gpu_idx[t].tolist()), set(ref_idx[t].tolist())
        if gs == rs:  # same set, slot order swapped: the two weights tie
            pairs = [(a, b) for a, b in zip(gpu_idx[t], ref_idx[t]) if a != b]
        else:
            pairs = [(a, b) for a in gs - rs for b in rs - gs]
        for a, b in pairs:
            assert abs(g[a] - g[b]) < NEAR_TIE, (
                f"token {t}: routing differs away from a tie: gpu {gpu_idx[t]} oracle {ref_idx[t]} "
                f"probs {g[a]:.9f} vs {g[b]:.9f}")
    return agree
