"""B300-native sparse Mixture-of-Experts SwiGLU layer forward.

Thin Python binding of the C ABI in ``include/moe.h`` (``libmoe.so``, built
in-tree for sm_103a).  The functions here carry the same names as the C entry
points and only marshal arguments: torch provides device memory and the
current CUDA stream, and every step of the layer runs in the library's
kernels.  There is no CPU fallback: without the built library or a CUDA
device the calls raise.
"""

from __future__ import annotations

import ctypes
import math
import os
import re
from typing import Dict, List, Optional

import torch

__all__ = [
    "MoEError", "lib", "declared_symbols", "moe_route", "moe_expert_choice_route",
    "moe_expert_choice_capacity", "moe_expert_choice_workspace_size", "moe_permute", "moe_permute_noalloc", "moe_gather_rows", "moe_grouped_gateup_swiglu",
    "moe_grouped_gateup_swiglu_gather",
    "moe_grouped_down", "moe_experts_swiglu", "moe_combine", "moe_ec_combine", "moe_aux_loss",
    "moe_layer_forward", "moe_layer_workspace_size", "moe_route_aux_rows", "moe_device_error",
    "moe_selftest_wait_expiry", "MoELayer", "HostPipeline",
]

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmoe.so")
HEADER_PATH = os.path.join(os.path.dirname(_PKG), "include", "moe.h")

MOE_F32, MOE_BF16 = 0, 1
MOE_ROUTE_NO_RENORM, MOE_ROUTE_CAPACITY = 1, 2
MOE_ROUTING_TOPK, MOE_ROUTING_EXPERT_CHOICE = 0, 1
_STATUS = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED", 3: "MOE_ERR_WORKSPACE",
           4: "MOE_ERR_CUDA"}


class MoEError(RuntimeError):
    def __init__(self, call: str, status: int):
        self.status = status
        super().__init__(f"{call} failed: {_STATUS.get(status, status)}")


class _Desc(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int), ("d", ctypes.c_int), ("F", ctypes.c_int), ("E", ctypes.c_int),
                ("k", ctypes.c_int), ("routing", ctypes.c_int), ("capacity_factor", ctypes.c_float),
                ("dtype", ctypes.c_int), ("flags", ctypes.c_int)]


class _Weights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("w_g", "bias", "w_gate", "w_up", "w_down")]


_OUT_FIELDS = ("topk_idx", "topk_w", "logits", "counts", "offsets", "f", "p", "loss", "ec_idx",
               "ec_score", "pos", "f_frac", "loss_frac", "dropped", "z_loss")


class _Outputs(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in _OUT_FIELDS]


_lib: Optional[ctypes.CDLL] = None

_P, _I, _F, _Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
_SIGS = {
    "moe_status_string": ([_I], ctypes.c_char_p),
    "moe_device_error": ([ctypes.POINTER(ctypes.c_uint32), _I], _I),
    "moe_selftest_wait_expiry": ([_I, _I, _I, _P, _P, _P, _P, _Z, _P], _I),
    "moe_route_aux_rows": ([_I], _Z),
    "moe_route": ([_P, _P, _P, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _I, _P], _I),
    "moe_expert_choice_capacity": ([_I, _I, _F], _I),
    "moe_expert_choice_workspace_size": ([_I, _I, _F], _Z),
    "moe_expert_choice_route": ([_P, _P, _P, _I, _I, _I, _F, _I, _P, _P, _P, _P, _P, _Z, _P], _I),
    "moe_permute_workspace_size": ([_I, _I, _I], _Z),
    "moe_permute": ([_P, _P, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _Z, _P], _I),
    "moe_gather_rows": ([_P, _P, _I, _I, _I, _I, _I, _P, _P], _I),
    "moe_permute_noalloc": ([_P, _P, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P], _I),
    "moe_grouped_gateup_swiglu": ([_P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _P], _I),
    "moe_grouped_gateup_swiglu_gather": ([_P, _P, _I, _I, _P, _P, _P, _I, _I, _I, _I, _I, _P, _P],
                                         _I),
    "moe_grouped_down": ([_P, _P, _P, _I, _I, _I, _I, _I, _P, _P], _I),
    "moe_experts_swiglu": ([_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _P, _P], _I),
    "moe_combine": ([_P, _P, _P, _I, _I, _I, _P, _P], _I),
    "moe_ec_combine": ([_P, _P, _P, _I, _I, _I, _I, _P, _P], _I),
    "moe_aux_loss": ([_P, _P, _P, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P], _I),
    "moe_layer_workspace_size": ([ctypes.POINTER(_Desc)], _Z),
    "moe_layer_forward": ([ctypes.POINTER(_Desc), ctypes.POINTER(_Weights), _P, _P,
                           ctypes.POINTER(_Outputs), _P, _Z, _P], _I),
}


def lib() -> ctypes.CDLL:
    """Loads libmoe.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise MoEError("load libmoe.so", -1) from FileNotFoundError(
                f"{LIB_PATH} missing: run `python -m sparse_mixture_experts_67_b300.build_lib`")
        handle = ctypes.CDLL(LIB_PATH)
        for name, (args, res) in _SIGS.items():
            fn = getattr(handle, name)
            fn.argtypes = args
            fn.restype = res
        _lib = handle
    return _lib


def declared_symbols() -> List[str]:
    """Function names declared in include/moe.h."""
    with open(HEADER_PATH) as fh:
        text = fh.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z_0-9]+)\s*\(", text)))


# ----------------------------------------------------------------- helpers


def _check(call: str, status: int) -> None:
    if status != 0:
        raise MoEError(call, status)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _dev(*ts: Optional[torch.Tensor]) -> None:
    for t in ts:
        if t is None:
            continue
        if not t.is_cuda:
            raise MoEError("argument check (tensor not on a CUDA device)", 1)
        if not t.is_contiguous():
            raise MoEError("argument check (tensor not contiguous)", 1)


def _bad(what: str) -> MoEError:
    return MoEError(f"argument check ({what})", 1)


def _dims(t: torch.Tensor, ndim: int, name: str) -> None:
    if t.dim() != ndim:
        raise _bad(f"{name} must be {ndim}-D, got shape {tuple(t.shape)}")


def _expect(t: Optional[torch.Tensor], name: str, dtype: Optional[torch.dtype] = None,
            shape=None, min_numel: Optional[int] = None) -> None:
    """Checks one tensor against the sizes and types the library is told about, so
    that no kernel reads or writes past a buffer (None passes: optional argument)."""
    if t is None:
        return
    if dtype is not None and t.dtype != dtype:
        raise _bad(f"{name} has dtype {t.dtype}, expected {dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise _bad(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if min_numel is not None and t.numel() < min_numel:
        raise _bad(f"{name} has {t.numel()} elements, needs at least {min_numel}")


def _dtype(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return MOE_BF16
    if t.dtype == torch.float32:
        return MOE_F32
    raise MoEError(f"argument check (dtype {t.dtype})", 2)


def _stream() -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _empty(shape, dtype, like: torch.Tensor) -> torch.Tensor:
    return torch.empty(shape, dtype=dtype, device=like.device)


# ------------------------------------------------------------- entry points


def moe_device_error(clear: bool = True) -> int:
    word = ctypes.c_uint32(0)
    _check("moe_device_error", lib().moe_device_error(ctypes.byref(word), int(clear)))
    return word.value


def moe_selftest_wait_expiry(T: int, E: int, capacity_factor: float) -> None:
    """Runs the expert-choice selection with waits that nothing satisfies (see
    include/moe.h): each gives up after its bound and sets code 16 in the device
    error word, which the caller reads with moe_device_error()."""
    C = moe_expert_choice_capacity(T, E, capacity_factor)
    dev = torch.device("cuda")
    pos = torch.zeros((E, T), dtype=torch.int32, device=dev)  # all logits 0.0
    ec_idx = torch.empty((E, max(C, 1)), dtype=torch.int32, device=dev)
    ec_score = torch.empty((E, max(C, 1)), dtype=torch.float32, device=dev)
    nbytes = moe_expert_choice_workspace_size(T, E, capacity_factor)
    ws = torch.empty((max(nbytes, 1),), dtype=torch.uint8, device=dev)
    _check("moe_selftest_wait_expiry",
           lib().moe_selftest_wait_expiry(T, E, C, _ptr(ec_idx), _ptr(ec_score), _ptr(pos), _ptr(ws),
                                          nbytes, _stream()))
    torch.cuda.synchronize()


def moe_route_aux_rows(T: int) -> int:
    return int(lib().moe_route_aux_rows(T))


def moe_expert_choice_capacity(T: int, E: int, capacity_factor: float) -> int:
    return int(lib().moe_expert_choice_capacity(T, E, capacity_factor))


def moe_expert_choice_workspace_size(T: int, E: int, capacity_factor: float) -> int:
    return int(lib().moe_expert_choice_workspace_size(T, E, capacity_factor))


def _check_router_args(x: torch.Tensor, w_g: torch.Tensor, bias: Optional[torch.Tensor]) -> None:
    _dims(x, 2, "x")
    _dims(w_g, 2, "w_g")
    E, d = w_g.shape[0], x.shape[1]
    _expect(w_g, "w_g", dtype=x.dtype, shape=(E, d))
    _expect(bias, "bias", dtype=torch.float32, shape=(E,))
    _dev(x, w_g, bias)


def moe_route(x: torch.Tensor, w_g: torch.Tensor, bias: Optional[torch.Tensor], k: int,
              want_logits: bool = False, want_probs: bool = False,
              want_aux: bool = True, renormalize: bool = True) -> Dict[str, torch.Tensor]:
    """Top-k router: returns topk_idx [T,k] int32, topk_w [T,k] fp32 and the optional outputs.
    renormalize=False keeps the selected probabilities as the weights (MOE_ROUTE_NO_RENORM)."""
    _check_router_args(x, w_g, bias)
    T, d = x.shape
    E = w_g.shape[0]
    out = {"topk_idx": _empty((T, k), torch.int32, x), "topk_w": _empty((T, k), torch.float32, x)}
    if want_logits:
        out["logits"] = _empty((T, E), torch.float32, x)
    if want_probs:
        out["probs"] = _empty((T, E), torch.float32, x)
    if want_aux:
        out["aux_partials"] = _empty((max(1, moe_route_aux_rows(T)), E), torch.float32, x)
        out["z_partials"] = _empty((max(1, moe_route_aux_rows(T)),), torch.float32, x)
    _check("moe_route", lib().moe_route(
        _ptr(x), _ptr(w_g), _ptr(bias), T, d, E, k, _dtype(x), _ptr(out["topk_idx"]),
        _ptr(out["topk_w"]), _ptr(out.get("logits")), _ptr(out.get("probs")),
        _ptr(out.get("aux_partials")), _ptr(out.get("z_partials")),
        0 if renormalize else MOE_ROUTE_NO_RENORM, _stream()))
    return out


def moe_expert_choice_route(x: torch.Tensor, w_g: torch.Tensor, bias: Optional[torch.Tensor],
                            capacity_factor: float) -> Dict[str, torch.Tensor]:
    """Expert-choice router: ec_idx [E,C], ec_score [E,C], pos [E,T], logits [T,E]."""
    _check_router_args(x, w_g, bias)
    T, d = x.shape
    E = w_g.shape[0]
    C = moe_expert_choice_capacity(T, E, capacity_factor)
    if C < 0:
        raise MoEError("moe_expert_choice_capacity", 1)
    out = {"ec_idx": _empty((E, C), torch.int32, x), "ec_score": _empty((E, C), torch.float32, x),
           "pos": _empty((E, T), torch.int32, x), "logits": _empty((T, E), torch.float32, x),
           "C": C}
    ws_bytes = int(lib().moe_expert_choice_workspace_size(T, E, capacity_factor))
    ws = _empty((max(ws_bytes, 1),), torch.uint8, x)
    _check("moe_expert_choice_route", lib().moe_expert_choice_route(
        _ptr(x), _ptr(w_g), _ptr(bias), T, d, E, capacity_factor, _dtype(x), _ptr(out["ec_idx"]),
        _ptr(out["ec_score"]), _ptr(out["pos"]), _ptr(out["logits"]), _ptr(ws), ws_bytes,
        _stream()))
    return out


def _check_permute_args(x: torch.Tensor, topk_idx: torch.Tensor, device: bool = True) -> None:
    _dims(x, 2, "x")
    _dims(topk_idx, 2, "topk_idx")
    _expect(topk_idx, "topk_idx", dtype=torch.int32, shape=(x.shape[0], topk_idx.shape[1]))
    if device:
        _dev(x, topk_idx)


def moe_permute(x: torch.Tensor, topk_idx: torch.Tensor, E: int) -> Dict[str, torch.Tensor]:
    """Stable dispatch: x_perm [T*k,d], counts [E], offsets [E+1], perm, inv_perm [T*k]."""
    _check_permute_args(x, topk_idx)
    T, d = x.shape
    k = topk_idx.shape[1]
    A = T * k
    ws_bytes = int(lib().moe_permute_workspace_size(T, E, k))
    ws = _empty((max(ws_bytes, 1),), torch.uint8, x)
    out = {"x_perm": _empty((A, d), x.dtype, x), "counts": _empty((E,), torch.int32, x),
           "offsets": _empty((E + 1,), torch.int32, x), "perm": _empty((A,), torch.int32, x),
           "inv_perm": _empty((A,), torch.int32, x)}
    _check("moe_permute", lib().moe_permute(
        _ptr(x), _ptr(topk_idx), T, d, E, k, _dtype(x), _ptr(out["x_perm"]), _ptr(out["counts"]),
        _ptr(out["offsets"]), _ptr(out["perm"]), _ptr(out["inv_perm"]), _ptr(ws), ws_bytes,
        _stream()))
    return out


def moe_permute_noalloc(x: torch.Tensor, topk_idx: torch.Tensor, E: int,
                        out: Optional[Dict[str, torch.Tensor]] = None) -> Dict[str, torch.Tensor]:
    """moe_permute without a workspace: the library's fixed device scratch is used instead.

    ``out`` may hold preallocated x_perm, counts, offsets, perm, inv_perm tensors
    (missing ones are created here with torch).
    """
    _check_permute_args(x, topk_idx, device=False)
    T, d = x.shape
    k = topk_idx.shape[1]
    A = T * k
    shapes = {"x_perm": ((A, d), x.dtype), "counts": ((E,), torch.int32),
              "offsets": ((E + 1,), torch.int32), "perm": ((A,), torch.int32),
              "inv_perm": ((A,), torch.int32)}
    res = dict(out or {})
    for name, (shape, dtype) in shapes.items():
        _expect(res.get(name), name, dtype=dtype, min_numel=math.prod(shape))
    _dev(x, topk_idx, *res.values())
    for name, (shape, dtype) in shapes.items():
        if name not in res:
            res[name] = _empty(shape, dtype, x)
    _check("moe_permute_noalloc", lib().moe_permute_noalloc(
        _ptr(x), _ptr(topk_idx), T, d, E, k, _dtype(x), _ptr(res["x_perm"]), _ptr(res["counts"]),
        _ptr(res["offsets"]), _ptr(res["perm"]), _ptr(res["inv_perm"]), _stream()))
    return res


def moe_gather_rows(x: torch.Tensor, src: torch.Tensor, div: int) -> torch.Tensor:
    _dims(x, 2, "x")
    _expect(src, "src", dtype=torch.int32)
    _dev(x, src)
    T, d = x.shape
    R = src.numel()
    out = _empty((R, d), x.dtype, x)
    _check("moe_gather_rows", lib().moe_gather_rows(_ptr(x), _ptr(src), R, div, T, d, _dtype(x),
                                                    _ptr(out), _stream()))
    return out


def _check_gateup_args(x: torch.Tensor, offsets: torch.Tensor, w_gate: torch.Tensor,
                       w_up: torch.Tensor) -> None:
    _dims(x, 2, "x")
    _dims(w_gate, 3, "w_gate")
    E, F = w_gate.shape[0], w_gate.shape[1]
    _expect(w_gate, "w_gate", dtype=x.dtype, shape=(E, F, x.shape[1]))
    _expect(w_up, "w_up", dtype=x.dtype, shape=(E, F, x.shape[1]))
    _expect(offsets, "offsets", dtype=torch.int32, min_numel=E + 1)


def moe_grouped_gateup_swiglu(x_perm: torch.Tensor, offsets: torch.Tensor, w_gate: torch.Tensor,
                              w_up: torch.Tensor, h: Optional[torch.Tensor] = None) -> torch.Tensor:
    _check_gateup_args(x_perm, offsets, w_gate, w_up)
    R, d = x_perm.shape
    E, F, _ = w_gate.shape
    _expect(h, "h", dtype=x_perm.dtype, min_numel=R * F)
    _dev(x_perm, offsets, w_gate, w_up, h)
    if h is None:
        h = _empty((R, F), x_perm.dtype, x_perm)
    _check("moe_grouped_gateup_swiglu", lib().moe_grouped_gateup_swiglu(
        _ptr(x_perm), _ptr(offsets), _ptr(w_gate), _ptr(w_up), R, d, F, E, _dtype(x_perm), _ptr(h),
        _stream()))
    return h


def moe_grouped_gateup_swiglu_gather(x: torch.Tensor, src: torch.Tensor, div: int,
                                     offsets: torch.Tensor, w_gate: torch.Tensor,
                                     w_up: torch.Tensor) -> torch.Tensor:
    """Gate/up + SwiGLU reading row r of the grouped input from x[src[r] // div]."""
    _check_gateup_args(x, offsets, w_gate, w_up)
    _expect(src, "src", dtype=torch.int32)
    _dev(x, src, offsets, w_gate, w_up)
    T, d = x.shape
    R = src.numel()
    E, F, _ = w_gate.shape
    h = _empty((R, F), x.dtype, x)
    _check("moe_grouped_gateup_swiglu_gather", lib().moe_grouped_gateup_swiglu_gather(
        _ptr(x), _ptr(src), div, T, _ptr(offsets), _ptr(w_gate), _ptr(w_up), R, d, F, E, _dtype(x),
        _ptr(h), _stream()))
    return h


def moe_grouped_down(h: torch.Tensor, offsets: torch.Tensor, w_down: torch.Tensor,
                     y_perm: Optional[torch.Tensor] = None) -> torch.Tensor:
    _dims(h, 2, "h")
    _dims(w_down, 3, "w_down")
    R, F = h.shape
    E, d, _ = w_down.shape
    _expect(w_down, "w_down", dtype=h.dtype, shape=(E, d, F))
    _expect(offsets, "offsets", dtype=torch.int32, min_numel=E + 1)
    _expect(y_perm, "y_perm", dtype=torch.float32, min_numel=R * d)
    _dev(h, offsets, w_down, y_perm)
    if y_perm is None:
        y_perm = _empty((R, d), torch.float32, h)
    _check("moe_grouped_down", lib().moe_grouped_down(
        _ptr(h), _ptr(offsets), _ptr(w_down), R, d, F, E, _dtype(h), _ptr(y_perm), _stream()))
    return y_perm


def moe_experts_swiglu(x_perm: torch.Tensor, offsets: torch.Tensor, w_gate: torch.Tensor,
                       w_up: torch.Tensor, w_down: torch.Tensor):
    _check_gateup_args(x_perm, offsets, w_gate, w_up)
    R, d = x_perm.shape
    E, F, _ = w_gate.shape
    _expect(w_down, "w_down", dtype=x_perm.dtype, shape=(E, d, F))
    _dev(x_perm, offsets, w_gate, w_up, w_down)
    h = _empty((R, F), x_perm.dtype, x_perm)
    y_perm = _empty((R, d), torch.float32, x_perm)
    _check("moe_experts_swiglu", lib().moe_experts_swiglu(
        _ptr(x_perm), _ptr(offsets), _ptr(w_gate), _ptr(w_up), _ptr(w_down), R, d, F, E,
        _dtype(x_perm), _ptr(h), _ptr(y_perm), _stream()))
    return y_perm, h


def moe_combine(y_perm: torch.Tensor, inv_perm: torch.Tensor, topk_w: torch.Tensor) -> torch.Tensor:
    _dims(y_perm, 2, "y_perm")
    _dims(topk_w, 2, "topk_w")
    T, k = topk_w.shape
    _expect(y_perm, "y_perm", dtype=torch.float32)
    _expect(topk_w, "topk_w", dtype=torch.float32)
    _expect(inv_perm, "inv_perm", dtype=torch.int32, min_numel=T * k)
    _dev(y_perm, inv_perm, topk_w)
    d = y_perm.shape[1]
    y = _empty((T, d), torch.float32, y_perm)
    _check("moe_combine", lib().moe_combine(_ptr(y_perm), _ptr(inv_perm), _ptr(topk_w), T, d, k,
                                            _ptr(y), _stream()))
    return y


def moe_ec_combine(y_perm: torch.Tensor, pos: torch.Tensor, ec_score: torch.Tensor) -> torch.Tensor:
    _dims(y_perm, 2, "y_perm")
    _dims(pos, 2, "pos")
    _dims(ec_score, 2, "ec_score")
    E, T = pos.shape
    C = ec_score.shape[1]
    _expect(pos, "pos", dtype=torch.int32)
    _expect(ec_score, "ec_score", dtype=torch.float32, shape=(E, C))
    _expect(y_perm, "y_perm", dtype=torch.float32, min_numel=E * C * y_perm.shape[1])
    _dev(y_perm, pos, ec_score)
    d = y_perm.shape[1]
    y = _empty((T, d), torch.float32, pos)
    _check("moe_ec_combine", lib().moe_ec_combine(_ptr(y_perm), _ptr(pos), _ptr(ec_score), T, d, E,
                                                  C, _ptr(y), _stream()))
    return y


def moe_aux_loss(counts: torch.Tensor, T: int, k: int, aux_partials: Optional[torch.Tensor] = None,
                 probs: Optional[torch.Tensor] = None,
                 z_partials: Optional[torch.Tensor] = None) -> Dict[str, torch.Tensor]:
    """f [E], p [E], loss [1] from router partial sums (or from probs [T,E]), and the
    fraction-of-assignments convention f_frac [E] = counts / (T k), loss_frac [1] = loss / k;
    with z_partials (from moe_route) also the router z-loss z_loss [1]."""
    E = counts.numel()
    rows = moe_route_aux_rows(T) if T > 0 else 0
    _expect(counts, "counts", dtype=torch.int32)
    _expect(aux_partials, "aux_partials", dtype=torch.float32, min_numel=rows * E)
    _expect(probs, "probs", dtype=torch.float32, min_numel=T * E)
    _expect(z_partials, "z_partials", dtype=torch.float32, min_numel=rows)
    _dev(counts, aux_partials, probs, z_partials)
    if probs is not None and aux_partials is None:
        aux_partials = _empty((max(1, moe_route_aux_rows(T)), E), torch.float32, counts)
    out = {"f": _empty((E,), torch.float32, counts), "p": _empty((E,), torch.float32, counts),
           "loss": _empty((1,), torch.float32, counts),
           "f_frac": _empty((E,), torch.float32, counts),
           "loss_frac": _empty((1,), torch.float32, counts)}
    if z_partials is not None:
        out["z_loss"] = _empty((1,), torch.float32, counts)
    _check("moe_aux_loss", lib().moe_aux_loss(
        _ptr(probs), _ptr(aux_partials), _ptr(counts), T, E, k, _ptr(out["f"]), _ptr(out["p"]),
        _ptr(out["loss"]), _ptr(out["f_frac"]), _ptr(out["loss_frac"]), _ptr(z_partials),
        _ptr(out.get("z_loss")), _stream()))
    return out


def _desc(T, d, F, E, k, routing, capacity_factor, dtype, flags=0) -> _Desc:
    return _Desc(T, d, F, E, k, routing, capacity_factor, dtype, flags)


def moe_layer_workspace_size(T: int, d: int, F: int, E: int, k: int, routing: int = 0,
                             capacity_factor: float = 0.0, dtype: int = MOE_BF16) -> int:
    desc = _desc(T, d, F, E, k, routing, capacity_factor, dtype)
    return int(lib().moe_layer_workspace_size(ctypes.byref(desc)))


def _output_sizes(T: int, E: int, k: int, routing: int, capacity_factor: float):
    """dtype and element count of each optional moe_layer_forward output (fields the
    routing mode does not write need no room)."""
    topk = routing == MOE_ROUTING_TOPK
    kk = k if topk else 0
    C = max(moe_expert_choice_capacity(T, E, capacity_factor), 0) if not topk else 0
    i32, f32 = torch.int32, torch.float32
    t = 1 if topk else 0
    return {"topk_idx": (i32, T * kk), "topk_w": (f32, T * kk), "logits": (f32, T * E),
            "counts": (i32, E * t), "offsets": (i32, (E + 1) * t), "f": (f32, E * t),
            "p": (f32, E * t), "loss": (f32, t), "ec_idx": (i32, E * C), "ec_score": (f32, E * C),
            "pos": (i32, E * T * (1 - t)), "f_frac": (f32, E * t), "loss_frac": (f32, t),
            "dropped": (i32, t), "z_loss": (f32, t)}


def moe_layer_forward(x: torch.Tensor, weights: Dict[str, torch.Tensor], k: int = 2,
                      routing: int = MOE_ROUTING_TOPK, capacity_factor: float = 0.0,
                      outputs: Optional[Dict[str, torch.Tensor]] = None,
                      workspace: Optional[torch.Tensor] = None,
                      y: Optional[torch.Tensor] = None, renormalize: bool = True,
                      capacity: bool = False) -> torch.Tensor:
    """Whole layer forward.  weights: w_g [E,d], bias [E] or None, w_gate/w_up [E,F,d], w_down [E,d,F].
    renormalize=False: top-k combine weights are the selected probabilities (MOE_ROUTE_NO_RENORM).
    capacity=True: top-k with at most int(T / E * capacity_factor * k) assignments per expert
    (MOE_ROUTE_CAPACITY); outputs["dropped"] ([1] int32) receives the number dropped."""
    w_g, bias = weights["w_g"], weights.get("bias")
    w_gate, w_up, w_down = weights["w_gate"], weights["w_up"], weights["w_down"]
    _dims(x, 2, "x")
    _dims(w_gate, 3, "w_gate")
    T, d = x.shape
    E, F, _ = w_gate.shape
    _expect(w_g, "w_g", dtype=x.dtype, shape=(E, d))
    _expect(bias, "bias", dtype=torch.float32, shape=(E,))
    _expect(w_gate, "w_gate", dtype=x.dtype, shape=(E, F, d))
    _expect(w_up, "w_up", dtype=x.dtype, shape=(E, F, d))
    _expect(w_down, "w_down", dtype=x.dtype, shape=(E, d, F))
    _expect(y, "y", dtype=torch.float32, min_numel=T * d)
    sizes = _output_sizes(T, E, k, routing, capacity_factor)
    for name, t in (outputs or {}).items():
        if name not in sizes:
            raise _bad(f"unknown output {name!r}; expected one of {sorted(sizes)}")
        _expect(t, name, dtype=sizes[name][0], min_numel=sizes[name][1])
    _dev(x, w_g, bias, w_gate, w_up, w_down, y, workspace)
    flags = (0 if renormalize else MOE_ROUTE_NO_RENORM) | (MOE_ROUTE_CAPACITY if capacity else 0)
    desc = _desc(T, d, F, E, k, routing, capacity_factor, _dtype(x), flags)
    need = int(lib().moe_layer_workspace_size(ctypes.byref(desc)))
    if workspace is None or workspace.numel() * workspace.element_size() < need:
        workspace = _empty((max(need, 1),), torch.uint8, x)
    if y is None:
        y = _empty((T, d), torch.float32, x)
    outs = _Outputs()
    for name, t in (outputs or {}).items():
        _dev(t)
        setattr(outs, name, t.data_ptr())
    wts = _Weights(w_g.data_ptr(), bias.data_ptr() if bias is not None else None,
                   w_gate.data_ptr(), w_up.data_ptr(), w_down.data_ptr())
    _check("moe_layer_forward", lib().moe_layer_forward(
        ctypes.byref(desc), ctypes.byref(wts), _ptr(x), _ptr(y), ctypes.byref(outs), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream()))
    return y


class MoELayer:
    """Holds device weights and a workspace; calls moe_layer_forward."""

    def __init__(self, weights: Dict[str, torch.Tensor], k: int = 2, routing: int = MOE_ROUTING_TOPK,
                 capacity_factor: float = 0.0, renormalize: bool = True, capacity: bool = False):
        self.weights = weights
        self.k, self.routing, self.capacity_factor = k, routing, capacity_factor
        self.renormalize, self.capacity = renormalize, capacity
        self._ws: Optional[torch.Tensor] = None

    def workspace(self, x: torch.Tensor) -> torch.Tensor:
        E, F, d = self.weights["w_gate"].shape
        need = moe_layer_workspace_size(x.shape[0], d, F, E, self.k, self.routing,
                                        self.capacity_factor, _dtype(x))
        if self._ws is None or self._ws.numel() < need:
            self._ws = _empty((max(need, 1),), torch.uint8, x)
        return self._ws

    def __call__(self, x: torch.Tensor, outputs=None, y=None) -> torch.Tensor:
        return moe_layer_forward(x, self.weights, self.k, self.routing, self.capacity_factor,
                                 outputs=outputs, workspace=self.workspace(x), y=y,
                                 renormalize=self.renormalize, capacity=self.capacity)


class HostPipeline:
    """Runs a MoELayer over batches held in pinned host memory with the copies
    overlapped: while batch i runs on the current stream, the host-to-device
    copy of batch i+1 runs on one copy stream and the device-to-host copy of
    batch i-1 on another.  Device buffers are double-buffered; every hazard
    between the three streams is ordered with CUDA events, so results equal
    those of copying, running and copying back one batch at a time."""

    def __init__(self, layer: MoELayer, T: int, d: int, dtype: torch.dtype,
                 device: Optional[torch.device] = None, depth: int = 2):
        if depth < 1:
            raise ValueError("depth must be >= 1")
        dev = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
        self.layer, self.depth = layer, depth
        self.h2d = torch.cuda.Stream(dev)
        self.d2h = torch.cuda.Stream(dev)
        self.xd = [torch.empty((T, d), dtype=dtype, device=dev) for _ in range(depth)]
        self.yd = [torch.empty((T, d), dtype=torch.float32, device=dev) for _ in range(depth)]
        ev = lambda: [torch.cuda.Event() for _ in range(depth)]  # noqa: E731
        self._x_ready, self._done, self._y_copied = ev(), ev(), ev()
        self._used = [False] * depth

    def run(self, xs_host: List[torch.Tensor], ys_host: List[torch.Tensor]) -> None:
        """ys_host[i] <- layer(xs_host[i]) for every i; enqueue only (synchronise on the
        current stream, or on the returned work, before reading ys_host).  xs_host[i] are
        pinned [T, d] tensors of the layer's dtype, ys_host[i] pinned [T, d] fp32."""
        if len(xs_host) != len(ys_host):
            raise ValueError("one output per input batch")
        compute = torch.cuda.current_stream(self.xd[0].device)
        start = torch.cuda.Event()
        start.record(compute)
        self.h2d.wait_event(start)
        self.d2h.wait_event(start)
        for i, (xh, yh) in enumerate(zip(xs_host, ys_host)):
            b = i % self.depth
            if self._used[b]:
                self.h2d.wait_event(self._done[b])       # batch i-depth finished reading xd[b]
                compute.wait_event(self._y_copied[b])    # and its result left yd[b]
            with torch.cuda.stream(self.h2d):
                self.xd[b].copy_(xh, non_blocking=True)
                self._x_ready[b].record(self.h2d)
            compute.wait_event(self._x_ready[b])
            self.layer(self.xd[b], y=self.yd[b])
            self._done[b].record(compute)
            self.d2h.wait_event(self._done[b])
            with torch.cuda.stream(self.d2h):
                yh.copy_(self.yd[b], non_blocking=True)
                self._y_copied[b].record(self.d2h)
            self._used[b] = True
        for b in range(self.depth):  # the current stream ends after every copy back
            if self._used[b]:
                compute.wait_event(self._y_copied[b])
