"""Host-side checks of the Python binding: every tensor's dtype and shape is checked
against the sizes handed to the library before anything reaches the device, so a
mismatched buffer is an exception, never an out-of-bounds kernel access.  The
tensors here live on the CPU: a well-formed call gets as far as the device check
and stops there (no CPU fallback)."""

import pytest

torch = pytest.importorskip("torch")

import sparse_mixture_experts_67_b300 as moe  # noqa: E402
from sparse_mixture_experts_67_b300 import build_lib  # noqa: E402

T, d, F, E, k = 12, 64, 128, 4, 2
bf16, f32, i32 = torch.bfloat16, torch.float32, torch.int32


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build_lib.build()
    moe.lib()


def _weights(**over):
    w = {"w_g": torch.zeros(E, d, dtype=bf16), "bias": None,
         "w_gate": torch.zeros(E, F, d, dtype=bf16), "w_up": torch.zeros(E, F, d, dtype=bf16),
         "w_down": torch.zeros(E, d, F, dtype=bf16)}
    w.update(over)
    return w


def _raises(fn, *needles):
    with pytest.raises(moe.MoEError) as ei:
        fn()
    msg = str(ei.value)
    for n in needles:
        assert n in msg, msg
    return msg


def _reaches_device_check(fn):
    _raises(fn, "not on a CUDA device")


x = torch.zeros(T, d, dtype=bf16)


def test_router_arguments():
    _reaches_device_check(lambda: moe.moe_route(x, torch.zeros(E, d, dtype=bf16), None, k))
    _raises(lambda: moe.moe_route(x, torch.zeros(E, d + 64, dtype=bf16), None, k), "w_g", "shape")
    _raises(lambda: moe.moe_route(x, torch.zeros(E, d, dtype=f32), None, k), "w_g", "dtype")
    _raises(lambda: moe.moe_route(x, torch.zeros(E, d, dtype=bf16), torch.zeros(E, dtype=torch.float64),
                                  k), "bias", "dtype")
    _raises(lambda: moe.moe_route(x, torch.zeros(E, d, dtype=bf16), torch.zeros(E + 1), k), "bias",
            "shape")
    _raises(lambda: moe.moe_route(x.view(-1), torch.zeros(E, d, dtype=bf16), None, k), "x", "2-D")
    _raises(lambda: moe.moe_expert_choice_route(x, torch.zeros(E, 32, dtype=bf16), None, 1.0), "w_g")


def test_dispatch_arguments():
    idx = torch.zeros(T, k, dtype=i32)
    _reaches_device_check(lambda: moe.moe_permute(x, idx, E))
    _raises(lambda: moe.moe_permute(x, idx.long(), E), "topk_idx", "dtype")
    _raises(lambda: moe.moe_permute(x, idx[:-1], E), "topk_idx", "shape")
    small = {"perm": torch.zeros(T * k - 1, dtype=i32)}
    _raises(lambda: moe.moe_permute_noalloc(x, idx, E, out=small), "perm", "elements")
    _raises(lambda: moe.moe_gather_rows(x, torch.zeros(5, dtype=torch.int64), 1), "src", "dtype")


def test_expert_gemm_arguments():
    R = T * k
    xp = torch.zeros(R, d, dtype=bf16)
    off = torch.zeros(E + 1, dtype=i32)
    w = _weights()
    _reaches_device_check(lambda: moe.moe_grouped_gateup_swiglu(xp, off, w["w_gate"], w["w_up"]))
    _raises(lambda: moe.moe_grouped_gateup_swiglu(xp, off[:E], w["w_gate"], w["w_up"]), "offsets")
    _raises(lambda: moe.moe_grouped_gateup_swiglu(xp, off, w["w_gate"], w["w_up"][:, :, :32]),
            "w_up", "shape")
    _raises(lambda: moe.moe_grouped_gateup_swiglu(xp, off, w["w_gate"], w["w_up"],
                                                  torch.zeros(R, F - 1, dtype=bf16)), "h")
    _raises(lambda: moe.moe_grouped_gateup_swiglu_gather(x, torch.zeros(R, dtype=i32), k, off,
                                                         w["w_gate"].float(), w["w_up"]), "w_gate")
    h = torch.zeros(R, F, dtype=bf16)
    _reaches_device_check(lambda: moe.moe_grouped_down(h, off, w["w_down"]))
    # W_down given in the [E, F, d] layout of W_gate: transposed, rejected
    _raises(lambda: moe.moe_grouped_down(h, off, w["w_gate"]), "w_down", "shape")
    _raises(lambda: moe.moe_grouped_down(h, off, w["w_down"], torch.zeros(R, d, dtype=bf16)),
            "y_perm", "dtype")
    _raises(lambda: moe.moe_experts_swiglu(xp, off, w["w_gate"], w["w_up"], w["w_gate"]), "w_down")


def test_combine_and_aux_arguments():
    R = T * k
    yp = torch.zeros(R, d)
    tw = torch.zeros(T, k)
    _reaches_device_check(lambda: moe.moe_combine(yp, torch.zeros(R, dtype=i32), tw))
    _raises(lambda: moe.moe_combine(yp, torch.zeros(R - 1, dtype=i32), tw), "inv_perm")
    _raises(lambda: moe.moe_combine(yp.to(bf16), torch.zeros(R, dtype=i32), tw), "y_perm", "dtype")
    C = 3
    pos = torch.zeros(E, T, dtype=i32)
    _reaches_device_check(lambda: moe.moe_ec_combine(torch.zeros(E * C, d), pos, torch.zeros(E, C)))
    _raises(lambda: moe.moe_ec_combine(torch.zeros(E * C - 1, d), pos, torch.zeros(E, C)), "y_perm")
    _raises(lambda: moe.moe_ec_combine(torch.zeros(E * C, d), pos, torch.zeros(E + 1, C)), "ec_score")
    counts = torch.zeros(E, dtype=i32)
    rows = moe.moe_route_aux_rows(T)
    _reaches_device_check(lambda: moe.moe_aux_loss(counts, T, k, aux_partials=torch.zeros(rows, E)))
    _raises(lambda: moe.moe_aux_loss(counts, T, k, aux_partials=torch.zeros(rows * E - 1)),
            "aux_partials")
    _raises(lambda: moe.moe_aux_loss(counts, T, k, probs=torch.zeros(T, E - 1)), "probs")
    _raises(lambda: moe.moe_aux_loss(counts.long(), T, k, probs=torch.zeros(T, E)), "counts")
    _raises(lambda: moe.moe_aux_loss(counts, T, k, aux_partials=torch.zeros(rows, E),
                                     z_partials=torch.zeros(rows - 1)), "z_partials")


def test_layer_arguments():
    _reaches_device_check(lambda: moe.moe_layer_forward(x, _weights(), k=k))
    _reaches_device_check(lambda: moe.moe_layer_forward(
        x, _weights(), k=k, outputs={"topk_idx": torch.zeros(T, k, dtype=i32),
                                     "z_loss": torch.zeros(1), "dropped": torch.zeros(1, dtype=i32)}))
    _raises(lambda: moe.moe_layer_forward(x, _weights(w_down=torch.zeros(E, F, d, dtype=bf16)), k=k),
            "w_down", "shape")
    _raises(lambda: moe.moe_layer_forward(x, _weights(w_up=torch.zeros(E, F, d)), k=k), "w_up", "dtype")
    _raises(lambda: moe.moe_layer_forward(x, _weights(bias=torch.zeros(E, dtype=bf16)), k=k), "bias")
    _raises(lambda: moe.moe_layer_forward(x, _weights(), k=k, y=torch.zeros(T - 1, d)), "y")
    _raises(lambda: moe.moe_layer_forward(x, _weights(), k=k,
                                          outputs={"topk_idx": torch.zeros(T, k, dtype=torch.int64)}),
            "topk_idx", "dtype")
    _raises(lambda: moe.moe_layer_forward(x, _weights(), k=k,
                                          outputs={"logits": torch.zeros(T, E - 1)}), "logits")
    _raises(lambda: moe.moe_layer_forward(x, _weights(), k=k, outputs={"zloss": torch.zeros(1)}),
            "unknown output")
    # expert choice: C = floor(T cf / E) = 6 picks per expert need room in ec_idx / ec_score
    C = moe.moe_expert_choice_capacity(T, E, 2.0)
    assert C == 6
    ec_out = {"ec_idx": torch.zeros(E, C, dtype=i32), "ec_score": torch.zeros(E, C),
              "pos": torch.zeros(E, T, dtype=i32)}
    _reaches_device_check(lambda: moe.moe_layer_forward(x, _weights(), routing=1, capacity_factor=2.0,
                                                        outputs=ec_out))
    _raises(lambda: moe.moe_layer_forward(x, _weights(), routing=1, capacity_factor=2.0,
                                          outputs=dict(ec_out, ec_idx=torch.zeros(E, C - 1, dtype=i32))),
            "ec_idx")
    # top-k outputs are not written in expert-choice mode and need no room there
    _reaches_device_check(lambda: moe.moe_layer_forward(
        x, _weights(), routing=1, capacity_factor=2.0,
        outputs={"topk_idx": torch.zeros(0, dtype=i32)}))


def test_every_output_at_its_documented_size_is_accepted():
    """All optional outputs at the sizes include/moe.h documents, in both routings and
    both dtypes, pass the checks (the call then stops at the device check)."""
    full = {"topk_idx": torch.zeros(T, k, dtype=i32), "topk_w": torch.zeros(T, k),
            "logits": torch.zeros(T, E), "counts": torch.zeros(E, dtype=i32),
            "offsets": torch.zeros(E + 1, dtype=i32), "f": torch.zeros(E), "p": torch.zeros(E),
            "loss": torch.zeros(1), "f_frac": torch.zeros(E), "loss_frac": torch.zeros(1),
            "dropped": torch.zeros(1, dtype=i32), "z_loss": torch.zeros(1)}
    for dt in (bf16, f32):
        xx = torch.zeros(T, d, dtype=dt)
        w = {n: t.to(dt) if t is not None else None for n, t in _weights().items()}
        w["bias"] = torch.zeros(E)
        _reaches_device_check(lambda: moe.moe_layer_forward(xx, w, k=k, outputs=full,
                                                            y=torch.zeros(T, d)))
        _reaches_device_check(lambda: moe.moe_layer_forward(xx, w, k=k, capacity_factor=1.25,
                                                            capacity=True, outputs=full))
        C = moe.moe_expert_choice_capacity(T, E, 1.5)
        ec = {"logits": torch.zeros(T, E), "ec_idx": torch.zeros(E, C, dtype=i32),
              "ec_score": torch.zeros(E, C), "pos": torch.zeros(E, T, dtype=i32)}
        _reaches_device_check(lambda: moe.moe_layer_forward(xx, w, k=0, routing=1,
                                                            capacity_factor=1.5, outputs=ec))
    # zero tokens: empty x and y
    _reaches_device_check(lambda: moe.moe_layer_forward(x[:0], _weights(), k=k, y=torch.zeros(0, d)))
