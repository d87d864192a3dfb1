"""The bounded device waits, made to run out.

Every mbarrier wait in the library's kernels gives up after a limit, records
MOE_ERR_DEVICE_TIMEOUT in the workspace's status word and lets its CTA drain its own copies and
MMAs, free its tensor memory and return, so a lost copy turns into a status the host reads
instead of a hung GPU.  The workspace's test hook shortens the limit and makes the first CTA of
the tensor arm's gate/up kernel withhold one token-tile copy (a copy that never arrives); the
call must return, report the timeout, and leave a context in which the next call -- after
moe_workspace_init -- meets the oracle."""
import numpy as np
import pytest

import oracle
from tests import workloads as wk

pytestmark = pytest.mark.gpu

MOE_ERR_DEVICE_TIMEOUT = -4


@pytest.fixture(scope="module")
def moe():
    import torch
    import mixture_experts_layer_09_gb300 as m
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    m.build()
    return m


def test_withheld_copy_times_out_and_the_workspace_recovers(moe):
    import torch
    inp = wk.layer("tiny", T=200, I_sh=128)
    x, r, W_r, E, S = wk.upload(inp)
    wl = inp.wl
    layer = moe.MoeLayer(W_r, E, S, wl.k, wl.T)
    y = wk.poison(torch.empty((wl.T, wl.H), dtype=torch.float32, device="cuda"))
    # about a millisecond at the GPU's clock: far above any wait of this small layer
    moe.moe_workspace_test_timeout(layer.ws, 2_000_000)
    layer.forward(x, r, y=y, arm=moe.ARM_GEMM)
    torch.cuda.synchronize()
    assert moe.moe_device_status(layer.ws) == MOE_ERR_DEVICE_TIMEOUT
    # the hook stays until the workspace is re-initialised: the next call times out again
    layer.forward(x, r, y=y, arm=moe.ARM_GEMM)
    assert moe.moe_device_status(layer.ws) == MOE_ERR_DEVICE_TIMEOUT
    # after moe_workspace_init the same workspace serves a normal call, to parity
    moe.moe_workspace_init(layer.ws)
    ids = wk.poison(torch.empty((wl.T, wl.k), dtype=torch.int32, device="cuda"))
    y = wk.poison(torch.empty((wl.T, wl.H), dtype=torch.float32, device="cuda"))
    layer.forward(x, r, y=y, topk_ids_out=ids, arm=moe.ARM_GEMM)
    assert moe.moe_device_status(layer.ws) == 0
    ref = oracle.layer_forward(inp)
    assert np.array_equal(ids.cpu().numpy(), ref["ids"])
    wk.assert_close(y.cpu().numpy(), ref["y"], "y after recovery")


def test_hook_argument_checks(moe):
    import torch
    ws = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    with pytest.raises(moe.MoeError):
        moe.moe_workspace_test_timeout(ws, -1)
    small = torch.zeros(1024, dtype=torch.uint8, device="cuda")
    with pytest.raises(moe.MoeError):
        moe.moe_workspace_test_timeout(small, 1000)
