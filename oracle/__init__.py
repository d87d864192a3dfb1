"""ctypes wrapper of the fp64 C oracle of the routed MoE layer (moe_oracle.c).

TEST INFRASTRUCTURE, NOT PART OF THE PRODUCT.  Only the tests, the smoke check
and the benchmark's CPU-baseline / reference leg import this package.  The CUDA
library never calls it and shares no code with it.

``build()`` compiles moe_oracle.c with gcc into ``oracle/libmoe_oracle.so``
(in-tree, git-ignored).  Independent rows run on every available host core by
default (``set_threads``); the per-row arithmetic is the same sequential loop
for any thread count.  The functions below take numpy arrays (bf16/fp16 as
uint16 bit patterns) and return numpy arrays.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
from typing import Optional

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "moe_oracle.c")
LIB = os.path.join(HERE, "libmoe_oracle.so")

_lib = None


def build(force: bool = False) -> str:
    if force or not os.path.exists(LIB) or os.path.getmtime(LIB) < max(
            os.path.getmtime(SRC), os.path.getmtime(os.path.join(HERE, "moe_oracle.h"))):
        tmp = LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c99", "-pthread", "-fPIC", "-shared", "-o", tmp, SRC, "-lm"])
        os.replace(tmp, LIB)
    return LIB


def lib():
    global _lib
    if _lib is None:
        build()
        _lib = C.CDLL(LIB)
        _lib.mo_bf16_to_f64.restype = C.c_double
        _lib.mo_bf16_to_f64.argtypes = [C.c_uint16]
        _lib.mo_f16_to_f64.restype = C.c_double
        _lib.mo_f16_to_f64.argtypes = [C.c_uint16]
        _lib.mo_e2m1_to_f64.restype = C.c_double
        _lib.mo_e2m1_to_f64.argtypes = [C.c_int]
        _lib.mo_ue8m0_to_f64.restype = C.c_double
        _lib.mo_ue8m0_to_f64.argtypes = [C.c_uint8]
        _lib.mo_set_threads(default_threads())
    return _lib


def default_threads() -> int:
    """Worker threads of the oracle: the host cores this process may run on."""
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except (AttributeError, OSError):
        return max(1, os.cpu_count() or 1)


def set_threads(n: int) -> None:
    """Worker threads for independent rows; results are bit-identical for any count."""
    lib().mo_set_threads(int(n))


def get_threads() -> int:
    return int(lib().mo_get_threads())


def _p(a: Optional[np.ndarray]):
    if a is None:
        return None
    assert a.flags.c_contiguous
    return a.ctypes.data_as(C.c_void_p)


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


def _check(rc: int, what: str):
    if rc != 0:
        raise ValueError(f"oracle {what} failed with code {rc}")


def bf16_to_f64(bits: int) -> float:
    return lib().mo_bf16_to_f64(int(bits))


def f16_to_f64(bits: int) -> float:
    return lib().mo_f16_to_f64(int(bits))


def dequant(q, s, rows: int, K: int) -> np.ndarray:
    q, s = _c(q, np.uint8), _c(s, np.uint16)
    w = np.empty((rows, K), dtype=np.float64)
    _check(lib().mo_dequant(_p(q), _p(s), rows, K, _p(w)), "dequant")
    return w


# weight formats (MO_FMT_INT4 / MO_FMT_MXFP4 of moe_oracle.h) and their scale element types
FMT_CODES = {"int4": 0, "mxfp4": 1}
SCALE_DTYPES = {"int4": np.uint16, "mxfp4": np.uint8}


def e2m1_to_f64(nibble: int) -> float:
    return lib().mo_e2m1_to_f64(int(nibble))


def ue8m0_to_f64(e: int) -> float:
    return lib().mo_ue8m0_to_f64(int(e))


def dequant_mxfp4(q, e8, rows: int, K: int) -> np.ndarray:
    q, e8 = _c(q, np.uint8), _c(e8, np.uint8)
    w = np.empty((rows, K), dtype=np.float64)
    _check(lib().mo_dequant_mxfp4(_p(q), _p(e8), rows, K, _p(w)), "dequant_mxfp4")
    return w


def router_logits(x, W_r, g=None) -> np.ndarray:
    x, W_r, g = _c(x, np.uint16), _c(W_r, np.uint16), _c(g, np.uint16)
    T, H = x.shape
    E = W_r.shape[0]
    out = np.empty((T, E + (g is not None)), dtype=np.float64)
    _check(lib().mo_router_logits(_p(x), _p(W_r), _p(g), T, H, E, _p(out)), "router_logits")
    return out


def router_topk(logits, k: int, E: Optional[int] = None):
    logits = _c(logits, np.float64)
    T, ld = logits.shape
    E = ld if E is None else E
    ids = np.empty((T, k), dtype=np.int32)
    w = np.empty((T, k), dtype=np.float64)
    _check(lib().mo_router_topk(_p(logits), ld, T, E, k, _p(ids), _p(w)), "router_topk")
    return ids, w


def router_topk_v(logits, k: int, bias=None, renormalize: bool = True, scale: float = 1.0,
                  E: Optional[int] = None):
    """Router variants: selection over logits + bias, weights from the unbiased softmax,
    renormalised over the picks or not, times scale."""
    logits = _c(logits, np.float64)
    T, ld = logits.shape
    E = ld if E is None else E
    b = None if bias is None else _c(bias, np.float64)
    ids = np.empty((T, k), dtype=np.int32)
    w = np.empty((T, k), dtype=np.float64)
    _check(lib().mo_router_topk_v(_p(logits), ld, T, E, k, _p(b), 1 if renormalize else 0, C.c_double(scale),
                                  _p(ids), _p(w)), "router_topk_v")
    return ids, w


def rmsnorm(y, gamma_bits, eps: float) -> np.ndarray:
    """out[t] = y[t] / sqrt(mean(y[t]^2) + eps) * gamma (gamma as bf16 bits)."""
    y = _c(y, np.float64)
    T, H = y.shape
    g = _c(gamma_bits, np.uint16)
    out = np.empty((T, H), dtype=np.float64)
    _check(lib().mo_rmsnorm(_p(y), _p(g), T, H, C.c_double(eps), _p(out)), "rmsnorm")
    return out


def dispatch(ids, E: int):
    ids = _c(ids, np.int32)
    T, k = ids.shape
    counts = np.empty(E, dtype=np.int32)
    offsets = np.empty(E + 1, dtype=np.int32)
    perm = np.empty(T * k, dtype=np.int32)
    inv = np.empty(T * k, dtype=np.int32)
    _check(lib().mo_dispatch(_p(ids), T, k, E, _p(counts), _p(offsets), _p(perm), _p(inv)), "dispatch")
    return counts, offsets, perm, inv


def expert_row(x_row, gate, up, down, H: int, I: int, fmt: str = "int4") -> np.ndarray:
    """gate/up/down: (q, s) pairs of one expert; s fp16 bits (int4) or ue8m0 bytes (mxfp4)."""
    x_row = _c(x_row, np.uint16)
    sd = SCALE_DTYPES[fmt]
    arrs = [_c(gate[0], np.uint8), _c(gate[1], sd), _c(up[0], np.uint8), _c(up[1], sd),
            _c(down[0], np.uint8), _c(down[1], sd)]
    o = np.empty(H, dtype=np.float64)
    _check(lib().mo_expert_row_fmt(_p(x_row), H, I, FMT_CODES[fmt], *[_p(a) for a in arrs], _p(o)),
           "expert_row")
    return o


def _exp_ptrs(ex):
    sd = SCALE_DTYPES[ex.fmt]
    arrs = [_c(ex.gate.q, np.uint8), _c(ex.gate.s, sd), _c(ex.up.q, np.uint8),
            _c(ex.up.s, sd), _c(ex.down.q, np.uint8), _c(ex.down.s, sd)]
    return arrs


def expert_mlp(x, ex, ids, perm, token_mask=None) -> np.ndarray:
    x, ids, perm = _c(x, np.uint16), _c(ids, np.int32), _c(perm, np.int32)
    T, H = x.shape
    k = ids.shape[1]
    arrs = _exp_ptrs(ex)
    tm = _c(token_mask, np.uint8)
    rows = np.zeros((T * k, H), dtype=np.float64)
    _check(lib().mo_expert_mlp_fmt(_p(x), T, H, ex.I, ex.E, k, FMT_CODES[ex.fmt], *[_p(a) for a in arrs],
                                   _p(ids), _p(perm), _p(tm), _p(rows)), "expert_mlp")
    return rows


def shared_expert(x, sh, token_mask=None) -> np.ndarray:
    x = _c(x, np.uint16)
    T, H = x.shape
    arrs = _exp_ptrs(sh)
    g = _c(sh.g, np.uint16)
    tm = _c(token_mask, np.uint8)
    y = np.zeros((T, H), dtype=np.float64)
    _check(lib().mo_shared_expert_fmt(_p(x), T, H, sh.I_sh, FMT_CODES[sh.fmt], *[_p(a) for a in arrs], _p(g),
                                      _p(tm), _p(y)), "shared_expert")
    return y


def combine(rows, inv, w, shared=None, residual=None, token_mask=None) -> np.ndarray:
    rows, inv, w = _c(rows, np.float64), _c(inv, np.int32), _c(w, np.float64)
    shared, residual = _c(shared, np.float64), _c(residual, np.uint16)
    T, k = w.shape
    H = rows.shape[1]
    tm = _c(token_mask, np.uint8)
    y = np.zeros((T, H), dtype=np.float64)
    _check(lib().mo_combine(_p(rows), _p(inv), _p(w), _p(shared), _p(residual), T, k, H, _p(tm), _p(y)),
           "combine")
    return y


def layer_forward(inp, token_mask=None):
    """inp: mixture_experts_layer_09_gb300.inputs.LayerInputs.  Returns dict with the fp32-rounded
    router logits, ids, w and y (fp64)."""
    wl = inp.wl
    x = _c(inp.x, np.uint16)
    T, H = x.shape
    ex, sh = inp.experts, inp.shared
    arrs = _exp_ptrs(ex)
    if sh is not None:
        sarrs = _exp_ptrs(sh)
        sg = _c(sh.g, np.uint16)
        I_sh, fmt_s = sh.I_sh, FMT_CODES[sh.fmt]
    else:
        sarrs, sg, I_sh, fmt_s = [None] * 6, None, 0, 0
    tm = _c(token_mask, np.uint8)
    logits = np.empty((T, ex.E), dtype=np.float64)
    ids = np.empty((T, wl.k), dtype=np.int32)
    w = np.empty((T, wl.k), dtype=np.float64)
    y = np.zeros((T, H), dtype=np.float64)
    r = _c(inp.residual, np.uint16)
    W_r = _c(inp.W_r, np.uint16)
    _check(lib().mo_layer_forward_fmt(_p(x), _p(r), _p(W_r), T, H, ex.I, ex.E, wl.k, FMT_CODES[ex.fmt],
                                      *[_p(a) for a in arrs], I_sh, fmt_s, *[_p(a) for a in sarrs], _p(sg),
                                      _p(tm), _p(logits), _p(ids), _p(w), _p(y)), "layer_forward")
    return {"logits": logits, "ids": ids, "w": w, "y": y}
