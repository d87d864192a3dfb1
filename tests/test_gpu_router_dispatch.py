"""GPU parity of stage 1 (router logits, softmax top-k) and stage 2 (dispatch) against the
fp64 oracle.  Routing outputs are compared bit for bit; weights and logits within tolerance."""
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


def _topk_gpu(moe, logits_t, E, k):
    import torch
    T = logits_t.shape[0]
    ids = wk.poison(torch.empty((T, k), dtype=torch.int32, device="cuda"))
    w = wk.poison(torch.empty((T, k), dtype=torch.float32, device="cuda"))
    moe.moe_router_topk(logits_t, E, k, ids, w)
    torch.cuda.synchronize()
    return ids.cpu().numpy(), w.cpu().numpy()


@pytest.mark.parametrize("E", [32, 64, 128, 256])
@pytest.mark.parametrize("T", [1, 64, 1024, 16384])
def test_topk_sweep_bf16_logits(moe, E, T):
    import torch
    k = 8
    L = wk.margin_logits(100 + E, T, E, k)
    ref_ids, ref_w = oracle.router_topk(gen.bf16_to_f32(L).astype(np.float64), k)
    ids, w = _topk_gpu(moe, wk.dev(L.view(np.int16), torch.bfloat16), E, k)
    assert np.array_equal(ids, ref_ids)
    wk.assert_close(w, ref_w, "topk_w")
    assert np.allclose(w.sum(axis=1), 1.0, atol=1e-5)


@pytest.mark.parametrize("E,k,bias,renorm,scale", [(60, 4, True, True, 1.0), (60, 4, True, False, 2.5),
                                                    (256, 8, True, True, 2.5), (256, 8, False, False, 1.0),
                                                    (128, 32, True, False, 1.0), (37, 5, False, True, 0.5)])
def test_router_topk_variants(moe, E, k, bias, renorm, scale):
    """Selection bias, no renormalisation, scaled weights against the oracle's definition; the
    k-th margin is enforced on the biased scores, so no near-tie decides a pick."""
    import torch
    T = 333
    g = gen.rng(7, E, k)
    L = (g.normal(0.0, 2.0, size=(T, E))).astype(np.float32)
    b = (g.normal(0.0, 0.5, size=E)).astype(np.float32) if bias else np.zeros(E, np.float32)
    for t in range(T):
        for a in range(64):
            if wk.kth_margin(L[t].astype(np.float64) + b.astype(np.float64), k) >= wk.MARGIN:
                break
            L[t] = gen.rng(7, E, k, t, a).normal(0.0, 2.0, size=E).astype(np.float32)
    ref_ids, ref_w = oracle.router_topk_v(L.astype(np.float64), k, bias=b.astype(np.float64) if bias else None,
                                          renormalize=renorm, scale=scale)
    ids = wk.poison(torch.empty((T, k), dtype=torch.int32, device="cuda"))
    w = wk.poison(torch.empty((T, k), dtype=torch.float32, device="cuda"))
    moe.moe_router_topk_v(wk.dev(L), E, k, ids, w, sel_bias=wk.dev(b) if bias else None, renormalize=renorm,
                          scale=scale)
    torch.cuda.synchronize()
    assert np.array_equal(ids.cpu().numpy(), ref_ids)
    wk.assert_close(w.cpu().numpy(), ref_w, "topk_w (variant)")


@pytest.mark.parametrize("E,k", [(8, 2), (60, 4), (256, 32), (37, 5), (256, 1), (16, 16)])
def test_topk_ties_fp32(moe, E, k):
    """Tie-heavy rows (values from a set of 8): ties inside the picks and at the k-th boundary
    are decided by the lowest index on both sides, on the same exact values."""
    import torch
    T = 512
    g = gen.rng(5, E, k)
    L = (g.integers(0, 8, size=(T, E)) * 0.25).astype(np.float32)
    ref_ids, ref_w = oracle.router_topk(L.astype(np.float64), k)
    ids, w = _topk_gpu(moe, wk.dev(L), E, k)
    assert np.array_equal(ids, ref_ids)
    wk.assert_close(w, ref_w, "topk_w")


def test_topk_strided_rows_and_nan(moe):
    import torch
    T, E, k, ld = 64, 60, 4, 61
    g = gen.rng(6)
    L = g.normal(size=(T, ld)).astype(np.float32)
    L[:, E] = 100.0  # the column past E (a shared gate logit) must never be picked
    ref_ids, ref_w = oracle.router_topk(L[:, :E].astype(np.float64), k)
    ids, w = _topk_gpu(moe, wk.dev(L), E, k)
    assert np.array_equal(ids, ref_ids)
    wk.assert_close(w, ref_w, "topk_w")
    # a NaN logit is never picked (treated as -inf)
    L2 = L.copy()
    L2[3, ref_ids[3, 0]] = np.nan
    ids2, _ = _topk_gpu(moe, wk.dev(L2), E, k)
    assert ref_ids[3, 0] not in ids2[3]


@pytest.mark.parametrize("T,E,H,with_g", [(1, 128, 2048, False), (16, 128, 2048, False), (8, 256, 6144, False),
                                          (512, 60, 2048, True), (100, 8, 256, True), (4096, 60, 2048, True),
                                          # tensor-core path: second MMA column chunk (E + 1 = 257), E = 1,
                                          # and the fp32 GEMM fallback (H not a multiple of 64)
                                          (300, 256, 1024, True), (200, 1, 128, True), (40, 128, 2080, False)])
def test_router_logits(moe, T, E, H, with_g):
    import torch
    x = gen.draw_x(3, T, H)
    W = gen.draw_router(3, E, H)
    gv = gen.bf16_bits(gen.rng(3, 99).normal(0, 0.02, size=H)) if with_g else None
    ref = oracle.router_logits(x, W, gv)
    out = wk.poison(torch.empty(ref.shape, dtype=torch.float32, device="cuda"))
    moe.moe_router_logits(wk.dev(x.view(np.int16), torch.bfloat16), wk.dev(W.view(np.int16), torch.bfloat16),
                          wk.dev(gv.view(np.int16), torch.bfloat16) if gv is not None else None, out)
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    # fp32 accumulation of exact bf16 products: absolute error far below the 1e-3 routing margin
    assert np.max(np.abs(got - ref)) < 1e-4
    wk.assert_close(got, ref, "logits")


def _dispatch_gpu(moe, ids_np, E):
    import torch
    T, k = ids_np.shape
    ids = wk.dev(ids_np.astype(np.int32))
    counts = wk.poison(torch.empty(E, dtype=torch.int32, device="cuda"))
    offsets = wk.poison(torch.empty(E + 1, dtype=torch.int32, device="cuda"))
    perm = wk.poison(torch.empty(T * k, dtype=torch.int32, device="cuda"))
    inv = wk.poison(torch.empty(T * k, dtype=torch.int32, device="cuda"))
    ws = torch.zeros(moe.moe_dispatch_workspace_size(T, k, E), dtype=torch.uint8, device="cuda")
    moe.moe_dispatch(ids, E, counts, offsets, perm, inv, ws)
    st = moe.moe_device_status(ws)
    return [t.cpu().numpy() for t in (counts, offsets, perm, inv)], st


@pytest.mark.parametrize("T,E,k", [(1, 8, 2), (4, 8, 2), (16, 128, 8), (8, 256, 32), (512, 8, 4), (2049, 16, 1),
                                   (1024, 64, 8), (1023, 60, 4), (2048, 256, 8), (16384, 256, 8), (16384, 32, 8),
                                   (8192, 8, 2)])
def test_dispatch_bit_exact(moe, T, E, k):
    """Both dispatch paths against the oracle: one CTA up to 2048 slots (512 x 4 is the last),
    count -> scatter above (2049 x 1 leaves one slot to its last CTA), with count tables at
    their row cap (16384 x 32) and entry cap (2048 x 256 and 16384 x 256)."""
    g = gen.rng(7, T, E, k)
    ids = np.stack([np.sort(g.choice(E, size=k, replace=False)) for _ in range(T)]).astype(np.int32)
    ref = oracle.dispatch(ids, E)
    got, st = _dispatch_gpu(moe, ids, E)
    assert st == 0
    for name, a, b in zip(("counts", "offsets", "perm", "inv"), got, ref):
        assert np.array_equal(a, b), name


def test_dispatch_skewed(moe):
    """Zipf-like popularity: most slots land in a few buckets, several buckets stay empty."""
    T, E, k = 12000, 64, 2
    g = gen.rng(8)
    p = 1.0 / np.arange(1, E + 1) ** 1.1
    p /= p.sum()
    ids = np.stack([np.sort(g.choice(E, size=k, replace=False, p=p)) for _ in range(T)]).astype(np.int32)
    ids[:, :] = np.where(ids >= 40, ids % 3, ids)  # leave experts 40..63 empty
    ids = np.sort(ids, axis=1)
    ids[:, 1] = np.where(ids[:, 1] == ids[:, 0], ids[:, 0] + 1, ids[:, 1])
    ref = oracle.dispatch(ids, E)
    got, st = _dispatch_gpu(moe, ids, E)
    assert st == 0
    for name, a, b in zip(("counts", "offsets", "perm", "inv"), got, ref):
        assert np.array_equal(a, b), name


def test_dispatch_bad_id_is_reported(moe):
    T, E, k = 32, 8, 2
    ids = np.tile(np.array([[0, 1]], dtype=np.int32), (T, 1))
    ids[5, 1] = 9  # out of range
    (counts, offsets, perm, inv), st = _dispatch_gpu(moe, ids, E)
    assert st == -5
    assert offsets[E] == T * k - 1
    assert inv[5 * k + 1] == -1
