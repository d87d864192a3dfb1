"""GPU parity at the edges of the supported shapes: the largest hidden size (H = 24576, whose
768 output-column blocks fill the down projection's counter table exactly), the smallest layer
(H = I = 32, one expert, k = 1; the tensor arm refuses it), every expert picked (k = E), and
k = 32 of E = 256 on both arms.  Same bars as the other layer tests."""
import numpy as np
import pytest

import oracle
from mixture_experts_layer_09_gb300 import inputs as gen
from tests import workloads as wk

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    import torch
    import mixture_experts_layer_09_gb300 as m
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    m.build()
    return m


def _run(moe, inp, arm):
    import torch
    x, r, W_r, E, S = wk.upload(inp)
    wl = inp.wl
    I_sh = S.I_sh if S is not None else 0
    ws = torch.zeros(moe.moe_workspace_size(wl.T, wl.E, wl.k, wl.H, wl.I, I_sh), dtype=torch.uint8, device="cuda")
    y = wk.poison(torch.empty((wl.T, wl.H), dtype=torch.float32, device="cuda"))
    ids = wk.poison(torch.empty((wl.T, wl.k), dtype=torch.int32, device="cuda"))
    w = wk.poison(torch.empty((wl.T, wl.k), dtype=torch.float32, device="cuda"))
    moe.moe_layer_forward(x, r, W_r, E, S, wl.k, y, ws, ids, w, arm=arm)
    assert moe.moe_device_status(ws) == 0
    return y.cpu().numpy(), ids.cpu().numpy(), w.cpu().numpy()


def _check(moe, inp, arm):
    ref = oracle.layer_forward(inp)
    y, ids, w = _run(moe, inp, arm)
    assert np.array_equal(ids, ref["ids"]), "routing differs"
    wk.assert_close(w, ref["w"], "topk_w")
    wk.assert_close(y, ref["y"], f"y arm={arm}")


@pytest.mark.parametrize("arm", [1, 2])
def test_largest_hidden_size(moe, arm):
    H = 24576  # MOE_MAX_H
    wl = gen.Workload("hmax", 3, H, 64, 4, 2, I_sh=64, seed=5)
    _check(moe, wk.enforce_margin_x(gen.draw_layer(wl)), arm)


def test_smallest_layer(moe):
    wl = gen.Workload("hmin", 1, 32, 32, 1, 1, I_sh=32, seed=6)
    inp = wk.enforce_margin_x(gen.draw_layer(wl))
    _check(moe, inp, 1)
    ref = oracle.layer_forward(inp)
    assert ref["w"][0, 0] == 1.0  # one expert: weight one
    with pytest.raises(moe.MoeError):
        _run(moe, inp, 2)  # K = 32 is not a whole tensor-arm K-step


@pytest.mark.parametrize("arm", [1, 2])
def test_every_expert_picked(moe, arm):
    wl = gen.Workload("kE", 5, 64, 64, 2, 2, seed=7)
    _check(moe, wk.enforce_margin_x(gen.draw_layer(wl)), arm)


@pytest.mark.parametrize("arm", [1, 2])
def test_k32_of_256_experts(moe, arm):
    wl = gen.Workload("k32", 40, 256, 128, 256, 32, I_sh=128, seed=8)
    _check(moe, wk.enforce_margin_x(gen.draw_layer(wl)), arm)


@pytest.mark.parametrize("T,H,I,E,k,I_sh", [
    (300, 2176, 128, 64, 8, 0),      # 34 K-steps: the router GEMM in 2 K ranges
    (1, 2048, 128, 64, 8, 128),      # one token on the tensor arm (4 K ranges, one top-k CTA)
    (77, 3136, 192, 33, 3, 64),      # 49 K-steps: one K range; odd E
    (4100, 1024, 64, 16, 2, 0),      # above 64 * 16 tokens: 8 tokens per top-k warp, 33 count rows
    (4100, 256, 64, 256, 8, 0),      # E=256: the top-k stages its rows in four rounds of 2 tokens per warp
    (2000, 512, 64, 255, 4, 64),     # E=255 + the shared gate: 256-wide logit rows, 63 count rows
])
def test_tensor_arm_routing_shapes(moe, T, H, I, E, k, I_sh):
    """The tensor arm's routing at shapes that take its other branches: the router's partial
    planes (1, 2 or 4), the counted top-k with several tokens per warp and several staging rounds
    per CTA, the scatter's count table with a ragged last CTA, and the tile list it writes."""
    wl = gen.Workload("route", T, H, I, E, k, I_sh=I_sh, seed=9)
    _check(moe, wk.enforce_margin_x(gen.draw_layer(wl)), 2)
