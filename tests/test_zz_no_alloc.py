"""moe_dispatch_static -- dispatch for callers that cannot allocate device memory at call
time -- must give the same buckets as moe_dispatch with a caller workspace.

The variant keeps its scratch in one array inside the library that every call on the device
shares, so the check runs two calls in a row with different inputs: the second must not see
anything left over from the first.  Both the one-CTA path and the multi-CTA path (which uses
the per-CTA count table) are covered.  This file is collected last on purpose."""
import ctypes as C

import numpy as np
import pytest

from mixture_experts_layer_09_gb300 import inputs as gen

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    import torch
    import mixture_experts_layer_09_gb300 as m
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    m.build()
    return m


def _ids(seed, T, E, k):
    g = gen.rng(seed, T, E, k)
    return np.stack([np.sort(g.choice(E, size=k, replace=False)) for _ in range(T)]).astype(np.int32)


def _outputs(torch, T, k, E):
    mk = lambda n: torch.full((n,), -7, dtype=torch.int32, device="cuda")  # noqa: E731
    return mk(E), mk(E + 1), mk(T * k), mk(T * k)


def test_static_dispatch_matches_workspace_dispatch(moe):
    import torch
    L = moe.lib()
    for (T, E, k, seed) in [(16384, 256, 8, 1), (3000, 60, 4, 2), (16, 128, 8, 3), (700, 8, 2, 4)]:
        ids_np = _ids(seed, T, E, k)
        ids = torch.from_numpy(ids_np).cuda()
        ref = _outputs(torch, T, k, E)
        ws = torch.zeros(moe.moe_dispatch_workspace_size(T, k, E), dtype=torch.uint8, device="cuda")
        moe.moe_dispatch(ids, E, *ref, ws)
        for call in range(2):  # two calls in a row through the C ABI
            got = _outputs(torch, T, k, E)
            rc = L.moe_dispatch_static(ids.data_ptr(), T, k, E, *[t.data_ptr() for t in got],
                                       C.c_void_p(torch.cuda.current_stream().cuda_stream))
            assert rc == 0
            torch.cuda.synchronize()
            for name, a, b in zip(("counts", "offsets", "perm", "inv"), got, ref):
                assert torch.equal(a, b), f"{name} differs (T={T}, E={E}, k={k}, call {call})"
    assert moe.moe_device_status(ws) == 0


def test_static_dispatch_rejects_oversize(moe):
    import torch
    L = moe.lib()
    fake = C.c_void_p(0x1000)
    T, k = (1 << 20) // 8 + 1, 8  # one token past the fixed array's capacity
    assert L.moe_dispatch_static(fake, T, k, 256, None, fake, fake, fake, None) == -1
    torch.cuda.synchronize()
