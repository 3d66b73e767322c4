"""The allocation-free dispatch entry point against the regular one.

moe_permute_noalloc is for callers that cannot give the library device
scratch: plugin hosts that hand a kernel only its input and output buffers,
and deployments whose device memory is reserved up front by another
allocator.  It keeps its scratch in a fixed array in the library's device
memory, so it must return exactly what moe_permute returns (the dispatch is
integer work: bit-exact), including on the second of two calls in a row,
after the first call has left its contents in the shared array.

This file is collected last so that a run stopping at the first failure has
already run every other test.
"""

import ctypes

import numpy as np
import pytest

from helpers import require_gpu, to_dev
from sparse_mixture_experts_67_b300 import synth

pytestmark = pytest.mark.gpu

MOE_ERR_WORKSPACE = 3


def _call_noalloc(moe, torch, x, idx, E, dt):
    T, d = x.shape
    k = idx.shape[1]
    A = T * k
    out = {"x_perm": torch.empty((A, d), dtype=x.dtype, device="cuda"),
           "counts": torch.empty((E,), dtype=torch.int32, device="cuda"),
           "offsets": torch.empty((E + 1,), dtype=torch.int32, device="cuda"),
           "perm": torch.empty((A,), dtype=torch.int32, device="cuda"),
           "inv_perm": torch.empty((A,), dtype=torch.int32, device="cuda")}
    p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    status = moe.lib().moe_permute_noalloc(
        p(x), p(idx), T, d, E, k, dt, p(out["x_perm"]), p(out["counts"]), p(out["offsets"]),
        p(out["perm"]), p(out["inv_perm"]), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert status == 0, moe.lib().moe_status_string(status)
    return out


def test_noalloc_permute_matches_workspace_permute_twice():
    torch = require_gpu()
    import sparse_mixture_experts_67_b300 as moe

    # first call spans more tiles and experts than the second, so stale
    # entries of the shared scratch lie inside and beyond the second's range;
    # the third has 293 tiles of 2048 assignments, so 293^2 * 64 > 4 Mi reads
    # sends it through the separate one-CTA scan, which writes the tile bases
    # into the second half of the array (293 * 64 entries fit in that half)
    cases = [("noalloc_a", 6000, 128, 64, 4, "bf16"), ("noalloc_b", 1500, 64, 8, 2, "bf16"),
             ("noalloc_scan", 150000, 64, 64, 4, "bf16")]
    for name, T, d, E, k, dt in cases:
        rng = np.random.default_rng(T + E)
        # k distinct experts per token: the first k of a random order of the E
        idx = np.argsort(rng.random((T, E)), axis=1)[:, :k].astype(np.int32)
        x = to_dev(synth.make_x(synth.small_config(name, T, d, 64, E, k, dt, seed=T)))
        idx_d = torch.from_numpy(idx).cuda()
        ref = moe.moe_permute(x, idx_d, E)
        got = _call_noalloc(moe, torch, x, idx_d, E, 1 if dt == "bf16" else 0)
        torch.cuda.synchronize()
        for key in ("counts", "offsets", "perm", "inv_perm", "x_perm"):
            assert torch.equal(got[key], ref[key]), f"{name}: {key} differs from moe_permute"


def test_noalloc_permute_rejects_sizes_beyond_its_scratch():
    require_gpu()
    import sparse_mixture_experts_67_b300 as moe

    z = ctypes.c_void_p(0)
    # ceil(300000*2/2048) * 256 = 75008 tile-expert entries > 32768: refused before any work
    status = moe.lib().moe_permute_noalloc(z, z, 300000, 64, 256, 2, 1, z, z, z, z, z, z)
    assert status == MOE_ERR_WORKSPACE
