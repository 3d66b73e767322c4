"""Host-side checks of the C ABI: the library loads, exports every symbol the
header declares, and rejects bad arguments before touching the device."""

import ctypes

import pytest

import sparse_mixture_experts_67_b300 as moe
from sparse_mixture_experts_67_b300 import build_lib


@pytest.fixture(scope="module")
def L():
    build_lib.build()
    return moe.lib()


def test_header_symbols_exported(L):
    declared = moe.declared_symbols()
    assert "moe_layer_forward" in declared and len(declared) >= 15
    for name in declared:
        assert hasattr(L, name), f"{name} declared in include/moe.h but not exported"


def test_status_strings(L):
    for code, name in enumerate(["MOE_OK", "MOE_ERR_INVALID_ARG", "MOE_ERR_UNSUPPORTED",
                                 "MOE_ERR_WORKSPACE", "MOE_ERR_CUDA"]):
        assert L.moe_status_string(code).decode() == name


def test_capacity_rule(L):
    assert L.moe_expert_choice_capacity(8192, 16, 2.0) == 1024
    assert L.moe_expert_choice_capacity(4, 2, 1.0) == 2
    assert L.moe_expert_choice_capacity(10, 4, 0.3) == 0
    assert L.moe_expert_choice_capacity(10, 3, 1.0) == 3
    assert L.moe_expert_choice_capacity(10, 4, 0.0) == -1


def test_aux_rows(L):
    # one row per router block of 32 tokens
    assert L.moe_route_aux_rows(0) == 0
    assert L.moe_route_aux_rows(1) == 1
    assert L.moe_route_aux_rows(32) == 1
    assert L.moe_route_aux_rows(33) == 2
    assert L.moe_route_aux_rows(8192) == 256


def _nullp():
    return ctypes.c_void_p(0)


def _p(v=4096):
    return ctypes.c_void_p(v)


def test_route_argument_errors(L):
    z = _nullp()
    # k > E, E > 256, k < 1, negative T: invalid before any device work
    assert L.moe_route(_p(), _p(), z, 8, 64, 4, 5, 1, _p(), _p(), z, z, z, z, 0, z) == 1
    assert L.moe_route(_p(), _p(), z, 8, 64, 300, 2, 1, _p(), _p(), z, z, z, z, 0, z) == 1
    assert L.moe_route(_p(), _p(), z, 8, 64, 8, 0, 1, _p(), _p(), z, z, z, z, 0, z) == 1
    assert L.moe_route(_p(), _p(), z, -1, 64, 8, 2, 1, _p(), _p(), z, z, z, z, 0, z) == 1
    # null required pointers
    assert L.moe_route(z, _p(), z, 8, 64, 8, 2, 1, _p(), _p(), z, z, z, z, 0, z) == 1
    assert L.moe_route(_p(), _p(), z, 8, 64, 8, 2, 1, z, _p(), z, z, z, z, 0, z) == 1
    # bf16 with d not a multiple of 64, unknown dtype, misaligned bf16 pointer
    assert L.moe_route(_p(), _p(), z, 8, 96, 8, 2, 1, _p(), _p(), z, z, z, z, 0, z) == 2
    assert L.moe_route(_p(), _p(), z, 8, 64, 8, 2, 7, _p(), _p(), z, z, z, z, 0, z) == 2
    assert L.moe_route(_p(4098), _p(), z, 8, 64, 8, 2, 1, _p(), _p(), z, z, z, z, 0, z) == 2
    # unknown routing flag bits
    assert L.moe_route(_p(), _p(), z, 8, 64, 8, 2, 1, _p(), _p(), z, z, z, z, 2, z) == 1
    # T == 0 is a no-op
    assert L.moe_route(z, z, z, 0, 64, 8, 2, 1, z, z, z, z, z, z, 0, z) == 0


def test_expert_choice_argument_errors(L):
    z = _nullp()
    ws = L.moe_expert_choice_workspace_size(8, 4, 1.0)
    assert ws > 0
    assert L.moe_expert_choice_route(_p(), _p(), z, 8, 64, 4, 0.0, 1, _p(), _p(), _p(), _p(), _p(), ws, z) == 1
    # capacity above T
    assert L.moe_expert_choice_route(_p(), _p(), z, 8, 64, 2, 4.0, 1, _p(), _p(), _p(), _p(), _p(), ws, z) == 1
    assert L.moe_expert_choice_route(_p(), _p(), z, 8, 64, 4, 1.0, 1, _p(), _p(), z, _p(), _p(), ws, z) == 1
    # the select's scratch: missing or one byte short
    assert L.moe_expert_choice_route(_p(), _p(), z, 8, 64, 4, 1.0, 1, _p(), _p(), _p(), _p(), z, ws, z) == 3
    assert L.moe_expert_choice_route(_p(), _p(), z, 8, 64, 4, 1.0, 1, _p(), _p(), _p(), _p(), _p(), ws - 1, z) == 3
    # no token limit: the scratch grows with T (slices of 1024 tokens)
    big = L.moe_expert_choice_workspace_size(40000, 16, 2.0)
    assert big >= 16 * 40 * 1024 * 8


def test_wait_expiry_selftest_argument_errors(L):
    z = _nullp()
    ws = L.moe_expert_choice_workspace_size(8192, 16, 2.0)
    # T, E or C out of range, or a NULL array: refused before any launch
    assert L.moe_selftest_wait_expiry(0, 16, 1, _p(), _p(), _p(), _p(), ws, z) == 1
    assert L.moe_selftest_wait_expiry(8192, 0, 1024, _p(), _p(), _p(), _p(), ws, z) == 1
    assert L.moe_selftest_wait_expiry(8192, 16, 0, _p(), _p(), _p(), _p(), ws, z) == 1
    assert L.moe_selftest_wait_expiry(8192, 16, 9000, _p(), _p(), _p(), _p(), ws, z) == 1
    assert L.moe_selftest_wait_expiry(8192, 16, 1024, _p(), z, _p(), _p(), ws, z) == 1
    # the selection's scratch: missing or one byte short
    assert L.moe_selftest_wait_expiry(8192, 16, 1024, _p(), _p(), _p(), z, ws, z) == 3
    assert L.moe_selftest_wait_expiry(8192, 16, 1024, _p(), _p(), _p(), _p(), ws - 1, z) == 3


def test_permute_and_experts_errors(L):
    z = _nullp()
    ws = L.moe_permute_workspace_size(100, 8, 2)
    assert ws > 0
    # tile counts and tile bases (tiles of 32 tokens' assignments at E <= 16, 64 above),
    # plus the block sums of the scan over all SMs (up to 160 blocks of E counts)
    for T, E, k in ((100, 8, 2), (200000, 64, 4), (20000, 256, 2)):
        tiles = -(-T * k // ((32 if E <= 16 else 64) * k))
        assert L.moe_permute_workspace_size(T, E, k) >= 4 * (2 * tiles * E + 160 * E)
    assert L.moe_permute(_p(), _p(), 100, 64, 8, 2, 1, _p(), _p(), _p(), _p(), _p(), _p(), ws - 1, z) == 3
    assert L.moe_permute(_p(), _p(), 100, 64, 8, 2, 1, _p(), _p(), _p(), _p(), _p(), z, ws, z) == 3
    assert L.moe_permute(_p(), _p(), 100, 64, 8, 9, 1, _p(), _p(), _p(), _p(), _p(), _p(), ws, z) == 1
    assert L.moe_grouped_gateup_swiglu(_p(), _p(), _p(), _p(), 10, 64, 100, 8, 1, _p(), z) == 2
    assert L.moe_grouped_gateup_swiglu(_p(), z, _p(), _p(), 10, 64, 128, 8, 1, _p(), z) == 1
    assert L.moe_grouped_down(_p(), _p(), _p(), 10, 64, 128, 0, 1, _p(), z) == 1
    assert L.moe_grouped_down(_p(), _p(), _p(), 0, 64, 128, 8, 1, z, z) == 0
    assert L.moe_combine(_p(), _p(), _p(), 4, 6, 2, _p(), z) == 2
    assert L.moe_combine(z, _p(), _p(), 4, 8, 2, _p(), z) == 1
    assert L.moe_ec_combine(_p(), _p(), _p(), 4, 8, 2, 5, _p(), z) == 1
    assert L.moe_aux_loss(z, z, _p(), 4, 8, 2, z, z, z, z, z, z, z, z) == 1


def test_layer_workspace_and_errors(L):
    d = moe._Desc(8192, 1024, 4096, 8, 2, 0, 0.0, 1)
    ws = L.moe_layer_workspace_size(ctypes.byref(d))
    A = 8192 * 2
    # bf16 top-2 combines inside the down GEMM: at least x_perm + h (bf16), no y_perm
    assert A * 1024 * 2 + A * 4096 * 2 <= ws < A * 1024 * 2 + A * 4096 * 2 + A * 1024 * 4
    # top-4 keeps the [R, d] fp32 y_perm for the separate combine
    d4 = moe._Desc(8192, 1024, 4096, 8, 4, 0, 0.0, 1)
    A4 = 8192 * 4
    assert L.moe_layer_workspace_size(ctypes.byref(d4)) >= A4 * 1024 * 2 + A4 * 4096 * 2 + A4 * 1024 * 4
    ec = moe._Desc(8192, 1024, 4096, 16, 0, 1, 2.0, 1)
    R = 16 * 1024
    assert L.moe_layer_workspace_size(ctypes.byref(ec)) >= R * 1024 * 2 + R * 4096 * 2 + R * 1024 * 4
    bad = moe._Desc(8192, 1024, 4096, 8, 9, 0, 0.0, 1)
    assert L.moe_layer_workspace_size(ctypes.byref(bad)) == 0
    w = moe._Weights(4096, 0, 4096, 4096, 4096)
    z = _nullp()
    assert L.moe_layer_forward(ctypes.byref(d), ctypes.byref(w), _p(), _p(), None, _p(), ws - 1, z) == 3
    assert L.moe_layer_forward(ctypes.byref(bad), ctypes.byref(w), _p(), _p(), None, _p(), ws, z) == 1
    fp = moe._Desc(16, 64, 102, 8, 2, 0, 0.0, 0)  # fp32 F not a multiple of 4
    assert L.moe_layer_forward(ctypes.byref(fp), ctypes.byref(w), _p(), _p(), None, _p(), 1 << 30, z) == 2
    flagged = moe._Desc(8192, 1024, 4096, 8, 2, 0, 0.0, 1, 4)  # unknown routing flag bits
    assert L.moe_layer_forward(ctypes.byref(flagged), ctypes.byref(w), _p(), _p(), None, _p(), ws, z) == 1
    # capacity-limited routing needs a positive factor, top-k routing and renormalised weights
    cap0 = moe._Desc(8192, 1024, 4096, 8, 2, 0, 0.0, 1, moe.MOE_ROUTE_CAPACITY)
    assert L.moe_layer_forward(ctypes.byref(cap0), ctypes.byref(w), _p(), _p(), None, _p(), ws, z) == 1
    cap_nr = moe._Desc(8192, 1024, 4096, 8, 2, 0, 1.25, 1,
                       moe.MOE_ROUTE_CAPACITY | moe.MOE_ROUTE_NO_RENORM)
    assert L.moe_layer_forward(ctypes.byref(cap_nr), ctypes.byref(w), _p(), _p(), None, _p(), ws, z) == 1
    cap_ec = moe._Desc(8192, 1024, 4096, 16, 0, 1, 2.0, 1, moe.MOE_ROUTE_CAPACITY)
    ws_ec = L.moe_layer_workspace_size(ctypes.byref(cap_ec))
    assert L.moe_layer_forward(ctypes.byref(cap_ec), ctypes.byref(w), _p(), _p(), None, _p(), ws_ec,
                               z) == 1


def test_no_cpu_fallback_without_device():
    torch = pytest.importorskip("torch")
    x = torch.zeros(4, 64)
    with pytest.raises(moe.MoEError):
        moe.moe_route(x, torch.zeros(8, 64), None, 2)


def test_alignment_checked_before_any_launch(L):
    """A misaligned caller pointer is MOE_ERR_UNSUPPORTED from the argument checks.
    Without a device any launch would fail with MOE_ERR_CUDA (4), so a 2 here also
    shows that no stage was enqueued before the check.  The pointers are not real
    allocations, so this runs only where no CUDA device is visible."""
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("uses placeholder pointers: host-only check")
    z = _nullp()
    d = moe._Desc(64, 1024, 4096, 8, 2, 0, 0.0, 1)
    ws = L.moe_layer_workspace_size(ctypes.byref(d))
    good = dict(w_g=4096, bias=0, w_gate=4096, w_up=4096, w_down=4096)
    # aligned pointers reach the first launch, which fails without a device
    assert L.moe_layer_forward(ctypes.byref(d), ctypes.byref(moe._Weights(*good.values())), _p(),
                               _p(), None, _p(), ws, z) == 4
    for field in ("w_g", "w_gate", "w_up", "w_down"):
        w = moe._Weights(*dict(good, **{field: 4104}).values())
        assert L.moe_layer_forward(ctypes.byref(d), ctypes.byref(w), _p(), _p(), None, _p(), ws,
                                   z) == 2, field
    w = moe._Weights(*good.values())
    assert L.moe_layer_forward(ctypes.byref(d), ctypes.byref(w), _p(4104), _p(), None, _p(), ws, z) == 2
    assert L.moe_layer_forward(ctypes.byref(d), ctypes.byref(w), _p(), _p(4104), None, _p(), ws, z) == 2
    # the same for expert choice and for the k > 2 path (separate combine)
    ec = moe._Desc(64, 1024, 4096, 8, 0, 1, 2.0, 1)
    ws_ec = L.moe_layer_workspace_size(ctypes.byref(ec))
    assert L.moe_layer_forward(ctypes.byref(ec), ctypes.byref(w), _p(), _p(4104), None, _p(), ws_ec,
                               z) == 2
    k4 = moe._Desc(64, 1024, 4096, 8, 4, 0, 0.0, 1)
    ws4 = L.moe_layer_workspace_size(ctypes.byref(k4))
    w_bad_down = moe._Weights(*dict(good, w_down=4104).values())
    assert L.moe_layer_forward(ctypes.byref(k4), ctypes.byref(w_bad_down), _p(), _p(), None, _p(),
                               ws4, z) == 2
    # both expert GEMMs' arguments are checked before the first one is enqueued
    args = [_p(), _p(), _p(), _p(), _p(), 256, 1024, 4096, 8, 1, _p(), _p(), z]
    assert L.moe_experts_swiglu(*args) == 4
    for i in (4, 11):  # w_down, y_perm
        bad = list(args)
        bad[i] = _p(4104)
        assert L.moe_experts_swiglu(*bad) == 2, i
    missing = list(args)
    missing[4] = z
    assert L.moe_experts_swiglu(*missing) == 1
