"""GPU parity of MXFP4 expert weights (e2m1 codes, one ue8m0 scale per 32 columns; the fmt=7
format of colibri PR #418's Kimi K3 tier) against the fp64 oracle: the upload-time scale
expansion bit for bit, the expert MLP of both arms, and whole layers with the routed and the
shared expert in either format.  Same bars as the int4 tests: routing bit-exact, floats within
rel-L2 1e-3 and max-abs 2e-3 * max|ref|."""
import numpy as np
import pytest

import oracle
from mixture_experts_layer_09_gb300 import inputs as gen
from tests import workloads as wk

pytestmark = pytest.mark.gpu

MOE_ERR_DEVICE_RANGE = -6


@pytest.fixture(scope="module")
def moe():
    import torch
    import mixture_experts_layer_09_gb300 as m
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    m.build()
    return m


def test_scale_expansion_every_exponent(moe):
    import torch
    e8 = np.arange(256, dtype=np.uint8)
    s = torch.full((256,), float("nan"), dtype=torch.float16, device="cuda")
    ws = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    moe.moe_mxfp4_scales(wk.dev(e8), s, ws)
    assert moe.moe_device_status(ws) == MOE_ERR_DEVICE_RANGE  # 0..103, 141..255 are out of range
    got = s.cpu().view(torch.int16).numpy().view(np.uint16)
    for e in range(256):
        if 104 <= e <= 140:
            # 2^(e - 128) as fp16, from the ue8m0 value the oracle decodes, halved
            want = np.float16(oracle.ue8m0_to_f64(e) / 2.0).view(np.uint16)
            assert got[e] == want, e
        else:
            assert got[e] == 0, e
    # the supported range alone records nothing
    ok = np.arange(104, 141, dtype=np.uint8)
    s2 = torch.empty(ok.size, dtype=torch.float16, device="cuda")
    moe.moe_mxfp4_scales(wk.dev(ok), s2, ws)
    assert moe.moe_device_status(ws) == 0


def test_upload_rejects_out_of_range_exponent(moe):
    q = np.zeros((1, 32, 16), dtype=np.uint8)
    e8 = np.full((1, 32, 1), 127, dtype=np.uint8)
    e8[0, 5, 0] = 255
    with pytest.raises(moe.MoeError):
        moe.upload_q4(q, e8, "mxfp4")


def _routing(inp):
    logits = oracle.router_logits(inp.x, inp.W_r).astype(np.float32).astype(np.float64)
    ids, w = oracle.router_topk(logits, inp.wl.k)
    return ids, w, oracle.dispatch(ids, inp.wl.E)


@pytest.mark.parametrize("arm", [1, 2])
@pytest.mark.parametrize("shape", [dict(T=4, H=256, I=128, E=8, k=2), dict(T=37, H=512, I=256, E=16, k=4),
                                   dict(T=200, H=256, I=192, E=8, k=2), dict(T=3, H=2048, I=768, E=128, k=8)])
def test_expert_mlp_rows_mxfp4(moe, arm, shape):
    import torch
    wl = gen.Workload("mlp", shape["T"], shape["H"], shape["I"], shape["E"], shape["k"], seed=13,
                      fmt=gen.FMT_MXFP4)
    inp = wk.enforce_margin_x(gen.draw_layer(wl))
    ids, w, (counts, offsets, perm, inv) = _routing(inp)
    ref = oracle.expert_mlp(inp.x, inp.experts, ids, perm)
    x, r, W_r, E, S = wk.upload(inp)
    T, k = wl.T, wl.k
    rows = wk.poison(torch.empty((T * k, wl.H), dtype=torch.float32, device="cuda"))
    ws = torch.zeros(moe.moe_expert_mlp_workspace_size(T, k, wl.E, wl.H, wl.I), dtype=torch.uint8, device="cuda")
    moe.moe_expert_mlp(x, k, E, wk.dev(offsets), wk.dev(perm), rows, ws, arm=arm)
    assert moe.moe_device_status(ws) == 0
    wk.assert_close(rows.cpu().numpy(), ref, f"mxfp4 rows arm={arm}")


def _check_layer(moe, inp, arm=0, sample=None):
    import torch
    T = inp.wl.T
    if sample is None:
        mask, toks = None, np.arange(T)
    else:
        toks = wk.bucket_sample_tokens(inp)
        mask = np.zeros(T, dtype=np.uint8)
        mask[toks] = 1
    ref = oracle.layer_forward(inp, token_mask=mask)
    x, r, W_r, E, S = wk.upload(inp)
    wl = inp.wl
    I_sh = S.I_sh if S is not None else 0
    ws = torch.zeros(moe.moe_workspace_size(wl.T, wl.E, wl.k, wl.H, wl.I, I_sh), dtype=torch.uint8, device="cuda")
    y = wk.poison(torch.empty((wl.T, wl.H), dtype=torch.float32, device="cuda"))
    ids = wk.poison(torch.empty((wl.T, wl.k), dtype=torch.int32, device="cuda"))
    moe.moe_layer_forward(x, r, W_r, E, S, wl.k, y, ws, ids, None, arm=arm)
    assert moe.moe_device_status(ws) == 0
    assert np.array_equal(ids.cpu().numpy(), ref["ids"]), "routing differs"
    wk.assert_close(y.cpu().numpy()[toks], ref["y"][toks], f"mxfp4 layer arm={arm}")


@pytest.mark.parametrize("arm", [1, 2])
@pytest.mark.parametrize("fmt,sh_fmt", [("mxfp4", "int4"), ("int4", "mxfp4"), ("mxfp4", "mxfp4")])
def test_layer_tiny_formats(moe, arm, fmt, sh_fmt):
    """Routed and shared experts in either format: the kernels pick the decode per work item."""
    inp = wk.layer("tiny", I_sh=128, T=40, fmt=fmt, sh_fmt=sh_fmt)
    assert inp.experts.fmt == fmt and inp.shared.fmt == sh_fmt
    _check_layer(moe, inp, arm)


def test_layer_qwen3_decode_t16_mxfp4(moe):
    _check_layer(moe, wk.layer("qwen3_30b_decode_t16_mxfp4"))


def test_layer_qwen15_prefill_t4096_mxfp4(moe):
    """MXFP4 routed experts with the int4 shared expert at T=4096, on tokens covering every token
    tile of every expert (every element passes too, in about 100 s of oracle time on 16 cores;
    the int4 twin of this layer is compared whole in test_gpu_layer.py)."""
    _check_layer(moe, wk.layer("qwen15_prefill_t4096_mxfp4"), sample="buckets")
