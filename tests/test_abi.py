"""The C-ABI library builds for sm_103a, loads, and exports every entry point its header
declares.  Host-side argument checks run before any CUDA call, so they are testable here
(no compute call is made without a GPU)."""
import ctypes as C
import os
import re

import numpy as np
import pytest

import mixture_experts_layer_09_gb300 as moe
from mixture_experts_layer_09_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    moe.build()
    return moe.lib()


def header_symbols():
    names = set()
    for h in os.listdir(os.path.join(ROOT, "include")):
        if h.endswith(".h"):
            txt = open(os.path.join(ROOT, "include", h)).read()
            names |= set(re.findall(r"^MOE_API\s+[\w\s\*]+?\b(moe_\w+)\s*\(", txt, flags=re.M))
    return names


def test_header_declares_the_entry_points():
    names = header_symbols()
    for n in ["moe_router_topk", "moe_dispatch", "moe_expert_mlp", "moe_combine", "moe_layer_forward",
              "moe_workspace_size", "moe_router_logits"]:
        assert n in names


def test_every_declared_symbol_is_exported(L):
    for n in header_symbols():
        assert hasattr(L, n), n
    assert set(moe.exported_symbols()) >= header_symbols()


def test_library_is_sm103a_only():
    assert "arch=compute_103a,code=sm_103a" in " ".join(_build.ARCH)


def test_version_and_status_strings(L):
    assert "sm_103a" in moe.moe_version()
    assert L.moe_status_string(0) == b"ok"
    assert L.moe_status_string(-4).startswith(b"device-side wait")


def test_workspace_sizes_are_positive_and_monotone(L):
    a = L.moe_workspace_size(1, 128, 8, 2048, 768, 0)
    b = L.moe_workspace_size(16, 128, 8, 2048, 768, 0)
    c = L.moe_workspace_size(4096, 60, 4, 2048, 1408, 5632)
    assert 0 < a < b < c
    assert L.moe_workspace_size(1, 0, 8, 2048, 768, 0) == 0
    assert L.moe_dispatch_workspace_size(16384, 8, 256) > L.moe_dispatch_workspace_size(16, 8, 256)


def test_host_argument_checks(L):
    fake = C.c_void_p(0x1000)
    # k > E, E > 256, ld < E: rejected before any device work
    assert L.moe_router_topk(fake, 0, 8, 4, 8, 9, fake, fake, None) == -1
    assert L.moe_router_topk(fake, 0, 300, 4, 300, 8, fake, fake, None) == -1
    assert L.moe_router_topk(fake, 0, 4, 4, 8, 2, fake, fake, None) == -1
    # T = 0 is a no-op
    assert L.moe_router_topk(None, 0, 8, 0, 8, 2, None, None, None) == 0
    # router variants: a non-finite scale, a misaligned bias, k > E
    f = C.c_float
    assert L.moe_router_topk_v(fake, 0, 8, 4, 8, 2, None, 1, f(float("nan")), fake, fake, None) == -1
    assert L.moe_router_topk_v(fake, 0, 8, 4, 8, 2, None, 1, f(float("inf")), fake, fake, None) == -1
    assert L.moe_router_topk_v(fake, 0, 8, 4, 8, 2, C.c_void_p(0x1002), 1, f(1.0), fake, fake, None) == -1
    assert L.moe_router_topk_v(fake, 0, 8, 4, 8, 9, None, 1, f(1.0), fake, fake, None) == -1
    assert L.moe_router_topk_v(None, 0, 8, 0, 8, 2, None, 0, f(2.0), None, None, None) == 0
    # null pointers / misaligned pointers / H not a multiple of 32
    assert L.moe_router_logits(None, fake, None, 4, 256, 8, fake, None) == -1
    assert L.moe_router_logits(C.c_void_p(0x1002), fake, None, 4, 256, 8, fake, None) == -1
    assert L.moe_router_logits(fake, fake, None, 4, 100, 8, fake, None) == -1
    # workspace too small
    assert L.moe_dispatch(fake, 4, 2, 8, None, fake, fake, fake, C.c_void_p(0x10000), 16, None) == -1
    # experts struct checks
    q = moe.moe_q4(0x1000, 0x2000)
    bad = moe.moe_experts(8, 256, 100, q, q, q)  # I % 32 != 0
    assert L.moe_expert_mlp(fake, 4, 2, C.byref(bad), fake, fake, fake, 0, C.c_void_p(0x10000), 1 << 30, None) == -1
    big = moe.moe_experts(300, 256, 128, q, q, q)  # E > 256
    assert L.moe_layer_forward(fake, None, fake, C.byref(big), None, 4, 2, fake, None, None, 0,
                               C.c_void_p(0x10000), 1 << 30, None) == -1
    ok = moe.moe_experts(8, 256, 128, q, q, q)
    assert L.moe_layer_forward(fake, None, fake, C.byref(ok), None, 4, 9, fake, None, None, 0,
                               C.c_void_p(0x10000), 1 << 30, None) == -1   # k > E
    assert L.moe_layer_forward(fake, None, fake, C.byref(ok), None, 4, 2, fake, None, None, 7,
                               C.c_void_p(0x10000), 1 << 30, None) == -1   # unknown arm
    assert L.moe_layer_forward(fake, None, fake, C.byref(ok), None, 0, 2, fake, None, None, 0,
                               C.c_void_p(0x10000), 1 << 30, None) == 0    # T = 0
    # weight formats: unknown format codes are rejected, for the routed and the shared set
    badfmt = moe.moe_experts(8, 256, 128, q, q, q, 2)
    assert L.moe_layer_forward(fake, None, fake, C.byref(badfmt), None, 4, 2, fake, None, None, 0,
                               C.c_void_p(0x10000), 1 << 30, None) == -1
    sh_bad = moe.moe_shared(64, q, q, q, None, -1)
    assert L.moe_layer_forward(fake, None, fake, C.byref(ok), C.byref(sh_bad), 4, 2, fake, None, None, 0,
                               C.c_void_p(0x10000), 1 << 30, None) == -1
    # MXFP4 scale expansion: null pointers, a short workspace, a misaligned output
    assert L.moe_mxfp4_scales(None, 16, fake, fake, 4096, None) == -1
    assert L.moe_mxfp4_scales(fake, 16, fake, fake, 100, None) == -1
    assert L.moe_mxfp4_scales(fake, 16, C.c_void_p(0x1001), fake, 4096, None) == -1
    assert L.moe_mxfp4_scales(fake, 0, fake, fake, 4096, None) == 0
    assert L.moe_status_string(-6).startswith(b"MXFP4 scale exponent")


def test_binding_weight_format_checks():
    # gate/up/down must share one format; the struct carries its code
    q4 = moe.Q4(None, None, "int4")
    fp4 = moe.Q4(None, None, "mxfp4")
    assert moe._fmt_of(fp4, fp4, fp4) == 1 and moe._fmt_of(q4, q4, q4) == 0
    with pytest.raises(moe.MoeError):
        moe._fmt_of(q4, fp4, q4)
    with pytest.raises(moe.MoeError):
        moe._fmt_of(moe.Q4(None, None, "nf4"))
    with pytest.raises(moe.MoeError):
        moe.upload_q4(np.zeros((1, 32, 16), np.uint8), np.zeros((1, 32, 1), np.uint16), "nf4")


def test_no_cpu_fallback_without_device(L):
    """With valid arguments but no usable sm_103a device, a compute call fails loudly."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    fake = C.c_void_p(0x1000)
    rc = L.moe_router_topk(fake, 0, 8, 4, 8, 2, fake, fake, None)
    assert rc in (-3, -2)


def test_auto_arm_constants_match_the_header():
    """The binding's copy of the AUTO arm rule's constants equals the header's."""
    import re

    import mixture_experts_layer_09_gb300 as moe
    hdr = open(os.path.join(ROOT, "include", "moe.h")).read()
    vals = dict(re.findall(r"#define (MOE_AUTO_GEMV_\w+) (\d+)", hdr))
    assert int(vals["MOE_AUTO_GEMV_ROWS_PER_EXPERT"]) == moe.AUTO_GEMV_ROWS_PER_EXPERT
    assert int(vals["MOE_AUTO_GEMV_MAX_T_SHARED"]) == moe.AUTO_GEMV_MAX_T_SHARED
