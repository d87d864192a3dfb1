"""moe_dispatch_static -- dispatch for callers that cannot allocate device memory at call
time -- must give the same buckets as moe_dispatch with a caller workspace.

The variant keeps its scratch in one array inside the library that every call on the device
shares, so the check runs two calls in a row with different inputs: the second must not see
anything left over from the first.  Both the one-CTA path and the multi-CTA path (which uses
the per-CTA count table) are covered.  The file is collected last so that, if it fails, a run
that stops at the first failure has already run every other test."""
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


def test_static_dispatch_out_of_range_ids_and_empty_batch(moe):
    """The documented edge behaviour: an id outside [0, E) lands in no bucket and its inv entry
    is -1; T = 0 is accepted with null id, perm and inv pointers and gives zero offsets."""
    import torch
    L = moe.lib()
    T, k, E = 5, 2, 8
    ids_np = _ids(9, T, E, k)
    ids_np[1, 0] = -1
    ids_np[3, 1] = E
    ids = torch.from_numpy(ids_np).cuda()
    counts, offsets, perm, inv = _outputs(torch, T, k, E)
    stream = C.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert L.moe_dispatch_static(ids.data_ptr(), T, k, E, counts.data_ptr(), offsets.data_ptr(), perm.data_ptr(),
                                 inv.data_ptr(), stream) == 0
    torch.cuda.synchronize()
    inv_np = inv.cpu().numpy()
    assert inv_np[1 * k + 0] == -1 and inv_np[3 * k + 1] == -1
    assert int(offsets[E]) == T * k - 2
    valid = [a for a in range(T * k) if a not in (1 * k + 0, 3 * k + 1)]
    assert sorted(perm.cpu().numpy()[:T * k - 2].tolist()) == valid
    # empty batch: no ids, no perm, no inv
    counts0, offsets0, _, _ = _outputs(torch, 1, 1, E)
    assert L.moe_dispatch_static(None, 0, k, E, counts0.data_ptr(), offsets0.data_ptr(), None, None, stream) == 0
    torch.cuda.synchronize()
    assert torch.count_nonzero(offsets0).item() == 0
    assert torch.count_nonzero(counts0).item() == 0
