"""Seeded synthetic inputs for the MoE layer workloads.

This module only draws random numbers and rounds them to the storage dtype.
It holds none of the layer's arithmetic, so the fp64 oracle and the CUDA path
can both be fed from it without sharing any computation.

Every tensor is drawn from its own PCG64 stream keyed by ``(seed, tensor_id)``
so that the weights of a configuration do not depend on how many tokens are
drawn (the large-expert configuration is swept over T with fixed weights).

Storage: fp32 tensors are ``np.float32``; bf16 tensors are ``np.uint16`` bit
patterns obtained from fp32 by round-to-nearest-even.  ``to_f64`` widens
either exactly.
"""

from __future__ import annotations

import dataclasses
import math
import os
from concurrent.futures import ThreadPoolExecutor
from typing import Dict, Optional, Sequence, Tuple

import numpy as np

# tensor ids of the independent streams
_X, _WG, _EXPERT0 = 0, 1, 2


@dataclasses.dataclass(frozen=True)
class LayerConfig:
    """Shape and value distribution of one synthetic MoE layer workload."""

    name: str
    T: int
    d: int
    F: int
    E: int
    k: int  # slots per token (top-k); unused by expert choice
    dtype: str  # "f32" or "bf16": x and all weights
    x_std: float
    w_std: float
    wg_std: float
    seed: int
    routing: str = "topk"  # "topk" or "expert_choice"
    capacity_factor: float = 0.0  # expert choice only
    bias: str = "none"  # "none", "zipf", "forced_empty"

    @property
    def C(self) -> int:
        """Expert-choice capacity: floor(T * cf / E)."""
        return int(math.floor(self.T * self.capacity_factor / self.E))

    @property
    def R(self) -> int:
        """Rows after dispatch."""
        return self.E * self.C if self.routing == "expert_choice" else self.T * self.k

    def with_tokens(self, T: int) -> "LayerConfig":
        return dataclasses.replace(self, T=T, name=f"{self.name.split('@')[0]}@T{T}")

    def active_flops(self) -> float:
        """Expert GEMM flops (3 matmuls of 2*d*F per routed row) + router flops."""
        return 6.0 * self.R * self.d * self.F + 2.0 * self.T * self.d * self.E


# The five workloads: a tiny fp32 layer, a top-2 layer, a large-expert layer
# swept over T, a fine-grained skewed layer and an expert-choice layer.
CONFIGS: Dict[str, LayerConfig] = {
    "tiny_fp32": LayerConfig("tiny_fp32", T=256, d=64, F=128, E=8, k=2, dtype="f32",
                             x_std=0.5, w_std=0.02, wg_std=0.1, seed=1000),
    "top2_d1024": LayerConfig("top2_d1024", T=8192, d=1024, F=4096, E=8, k=2, dtype="bf16",
                              x_std=1.0, w_std=0.02, wg_std=0.1, seed=1001),
    "large_d4096": LayerConfig("large_d4096", T=16384, d=4096, F=14336, E=8, k=2, dtype="bf16",
                               x_std=1.0, w_std=0.02, wg_std=0.1, seed=1002),
    "fine_e64": LayerConfig("fine_e64", T=16384, d=2048, F=1408, E=64, k=4, dtype="bf16",
                            x_std=1.0, w_std=0.02, wg_std=0.1, seed=1003, bias="zipf"),
    "ec_e16": LayerConfig("ec_e16", T=8192, d=1024, F=4096, E=16, k=0, dtype="bf16",
                          x_std=1.0, w_std=0.02, wg_std=0.1, seed=1004,
                          routing="expert_choice", capacity_factor=2.0),
}
LARGE_T_SWEEP: Tuple[int, ...] = (16, 256, 4096, 16384)

# Correctness-only variant of the fine-grained shape whose bias empties
# experts 48..63 and overfills expert 0.
CONFIGS["fine_e64_forced_empty"] = dataclasses.replace(
    CONFIGS["fine_e64"], name="fine_e64_forced_empty", bias="forced_empty", seed=1005)


def _rng(seed: int, tensor_id: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64([seed, tensor_id]))


def round_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns, round to nearest even (finite inputs)."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def to_f64(a: np.ndarray) -> np.ndarray:
    """Exact widening of a stored tensor (fp32 or bf16 bits) to fp64."""
    if a.dtype == np.uint16:
        return (a.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    return a.astype(np.float64)


def _normal(seed: int, tensor_id: int, shape, std: float, dtype: str) -> np.ndarray:
    z = _rng(seed, tensor_id).standard_normal(size=shape, dtype=np.float32)
    z *= np.float32(std)
    return round_to_bf16_bits(z) if dtype == "bf16" else z


def router_bias(cfg: LayerConfig) -> Optional[np.ndarray]:
    """Per-expert logit bias (fp32) of the skewed workloads, or None."""
    e = np.arange(cfg.E, dtype=np.float64)
    if cfg.bias == "zipf":
        return (1.5 * np.log(1.0 / (e + 1.0))).astype(np.float32)
    if cfg.bias == "forced_empty":
        b = np.zeros(cfg.E, dtype=np.float32)
        b[48:] = -1.0e4
        b[0] = 3.0
        return b
    return None


def make_x(cfg: LayerConfig) -> np.ndarray:
    return _normal(cfg.seed, _X, (cfg.T, cfg.d), cfg.x_std, cfg.dtype)


def make_router_weight(cfg: LayerConfig) -> np.ndarray:
    """W_g in nn.Linear layout [E, d]."""
    return _normal(cfg.seed, _WG, (cfg.E, cfg.d), cfg.wg_std, cfg.dtype)


def make_expert_weights(cfg: LayerConfig, e: int) -> Tuple[np.ndarray, np.ndarray, np.ndarray]:
    """(W_gate [F,d], W_up [F,d], W_down [d,F]) of expert e, nn.Linear layout."""
    base = _EXPERT0 + 3 * e
    wg = _normal(cfg.seed, base + 0, (cfg.F, cfg.d), cfg.w_std, cfg.dtype)
    wu = _normal(cfg.seed, base + 1, (cfg.F, cfg.d), cfg.w_std, cfg.dtype)
    wd = _normal(cfg.seed, base + 2, (cfg.d, cfg.F), cfg.w_std, cfg.dtype)
    return wg, wu, wd


@dataclasses.dataclass
class LayerInputs:
    """Host copies of one workload, in storage dtype."""

    cfg: LayerConfig
    x: np.ndarray
    w_g: np.ndarray
    bias: Optional[np.ndarray]
    w_gate: np.ndarray  # [E, F, d]
    w_up: np.ndarray  # [E, F, d]
    w_down: np.ndarray  # [E, d, F]


def make_inputs(cfg: LayerConfig, threads: int = 0) -> LayerInputs:
    """All tensors of a workload.  The experts are drawn on a thread pool (numpy's
    generators release the GIL); every tensor has its own stream, so the values do
    not depend on the thread count or the order the draws finish in."""
    store = np.uint16 if cfg.dtype == "bf16" else np.float32
    w_gate = np.empty((cfg.E, cfg.F, cfg.d), dtype=store)
    w_up = np.empty((cfg.E, cfg.F, cfg.d), dtype=store)
    w_down = np.empty((cfg.E, cfg.d, cfg.F), dtype=store)

    def fill(e: int) -> None:
        w_gate[e], w_up[e], w_down[e] = make_expert_weights(cfg, e)

    n = threads or min(cfg.E, os.cpu_count() or 1, 16)
    if n > 1 and cfg.E > 1:
        with ThreadPoolExecutor(n) as ex:
            list(ex.map(fill, range(cfg.E)))
    else:
        for e in range(cfg.E):
            fill(e)
    return LayerInputs(cfg, make_x(cfg), make_router_weight(cfg), router_bias(cfg),
                       w_gate, w_up, w_down)


class ExpertsF64(Sequence):
    """Lazy exact fp64 view of stored expert weights: item e -> (W_gate, W_up, W_down)."""

    def __init__(self, w_gate: np.ndarray, w_up: np.ndarray, w_down: np.ndarray):
        self._w = (w_gate, w_up, w_down)

    def __len__(self) -> int:
        return self._w[0].shape[0]

    def __getitem__(self, e):
        return tuple(to_f64(w[e]) for w in self._w)


def small_config(name: str, T: int, d: int, F: int, E: int, k: int, dtype: str = "f32",
                 seed: int = 7, **kw) -> LayerConfig:
    """Ad-hoc shape for tests (several tiles plus a ragged tail)."""
    base = dict(x_std=1.0, w_std=0.05, wg_std=0.1)
    base.update(kw)
    return LayerConfig(name, T=T, d=d, F=F, E=E, k=k, dtype=dtype, seed=seed, **base)
