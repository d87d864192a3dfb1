"""Routed Mixture-of-Experts layer for one GB300 (sm_103a): Python binding of libmoe_gb300.so.

Argument marshalling only: every step of the layer runs in the library's CUDA kernels.
PyTorch supplies device memory and the current stream.  The binding has the C entry points'
names (include/moe.h) and takes torch tensors:

* bf16 tensors (x, residual, W_r, g) as ``torch.bfloat16``, fp16 scales as ``torch.float16``
  (or any 16-bit dtype with the same bit patterns), packed nibbles as ``torch.uint8``,
  ids/offsets/perm/inv as ``torch.int32``, logits / weights / outputs as ``torch.float32``.
* Every call enqueues on ``torch.cuda.current_stream()`` and returns without synchronising.

There is no CPU fallback: without the built library, or without an sm_103a device, every call
raises ``MoeError``.  Call :func:`build` (nvcc) once to compile the library in-tree.
"""
from __future__ import annotations

import ctypes as C
import os
from dataclasses import dataclass
from typing import Optional

from . import _build

ARM_AUTO, ARM_GEMV, ARM_GEMM = 0, 1, 2
AUTO_GEMV_ROWS_PER_EXPERT = 4   # MOE_AUTO_GEMV_ROWS_PER_EXPERT
AUTO_GEMV_MAX_T_SHARED = 16     # MOE_AUTO_GEMV_MAX_T_SHARED

_lib = None


class MoeError(RuntimeError):
    def __init__(self, code: int, what: str):
        msg = _lib.moe_status_string(code).decode() if _lib is not None else str(code)
        super().__init__(f"{what}: {msg} ({code})")
        self.code = code


def build(force: bool = False) -> str:
    """Compile the CUDA library for sm_103a (nvcc) into the package directory."""
    return _build.build(force=force)


class moe_q4(C.Structure):
    _fields_ = [("q", C.c_void_p), ("s", C.c_void_p)]


class moe_experts(C.Structure):
    _fields_ = [("E", C.c_int), ("H", C.c_int), ("I", C.c_int),
                ("gate", moe_q4), ("up", moe_q4), ("down", moe_q4), ("fmt", C.c_int)]


class moe_shared(C.Structure):
    _fields_ = [("I_sh", C.c_int), ("gate", moe_q4), ("up", moe_q4), ("down", moe_q4), ("g", C.c_void_p),
                ("fmt", C.c_int)]


# weight formats (MOE_WFMT_*)
WFMT = {"int4": 0, "mxfp4": 1}


_P, _I, _S = C.c_void_p, C.c_int, C.c_size_t
_SIGS = {
    "moe_status_string": (C.c_char_p, [_I]),
    "moe_version": (C.c_char_p, []),
    "moe_router_logits": (_I, [_P, _P, _P, _I, _I, _I, _P, _P]),
    "moe_router_topk": (_I, [_P, _I, _I, _I, _I, _I, _P, _P, _P]),
    "moe_router_topk_v": (_I, [_P, _I, _I, _I, _I, _I, _P, _I, C.c_float, _P, _P, _P]),
    "moe_dispatch_workspace_size": (_S, [_I, _I, _I]),
    "moe_dispatch": (_I, [_P, _I, _I, _I, _P, _P, _P, _P, _P, _S, _P]),
    "moe_dispatch_static": (_I, [_P, _I, _I, _I, _P, _P, _P, _P, _P]),
    "moe_expert_mlp_workspace_size": (_S, [_I, _I, _I, _I, _I]),
    "moe_expert_mlp": (_I, [_P, _I, _I, C.POINTER(moe_experts), _P, _P, _P, _I, _P, _S, _P]),
    "moe_combine": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _P, _P]),
    "moe_workspace_size": (_S, [_I, _I, _I, _I, _I, _I]),
    "moe_layer_forward": (_I, [_P, _P, _P, C.POINTER(moe_experts), C.POINTER(moe_shared), _I, _I, _P, _P, _P,
                               _I, _P, _S, _P]),
    "moe_rmsnorm": (_I, [_P, _P, _I, _I, C.c_float, _P, _P]),
    "moe_layer_forward_norm": (_I, [_P, _P, _P, C.POINTER(moe_experts), C.POINTER(moe_shared), _I, _I, _P, _P,
                                    C.c_float, _P, _P, _P, _I, _P, _S, _P]),
    "moe_workspace_init": (_I, [_P, _S, _P]),
    "moe_workspace_test_timeout": (_I, [_P, _S, C.c_longlong, _P]),
    "moe_mxfp4_scales": (_I, [_P, _S, _P, _P, _S, _P]),
    "moe_device_status": (_I, [_P, _S, C.POINTER(C.c_int), _P]),
    "moe_launch_count": (C.c_longlong, []),
    "moe_profile_enable": (_I, [_I]),
    "moe_profile_read": (_I, [_I, C.c_char_p, _I, C.POINTER(C.c_double), C.POINTER(C.c_long), C.POINTER(C.c_int)]),
}


def lib_path() -> str:
    return _build.LIB


def lib():
    """The loaded CUDA library; raises MoeError-like RuntimeError when it was never built."""
    global _lib
    if _lib is None:
        if not os.path.exists(_build.LIB):
            raise RuntimeError(f"CUDA library not built ({_build.LIB} missing): call "
                               "mixture_experts_layer_09_gb300.build() first -- there is no CPU fallback")
        L = C.CDLL(_build.LIB)
        for name, (res, args) in _SIGS.items():
            f = getattr(L, name)
            f.restype, f.argtypes = res, args
        _lib = L
    return _lib


def exported_symbols():
    return sorted(_SIGS)


# ----------------------------------------------------------------------------- helpers

def _ptr(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(stream=None) -> int:
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _check(rc: int, what: str):
    if rc != 0:
        raise MoeError(rc, what)


def _need(t, dtype_size: int, what: str):
    if t is None:
        return
    if not t.is_cuda:
        raise MoeError(-1, f"{what} must be a CUDA tensor")
    if not t.is_contiguous():
        raise MoeError(-1, f"{what} must be contiguous")
    if t.element_size() != dtype_size:
        raise MoeError(-1, f"{what} must have {dtype_size}-byte elements")


@dataclass
class Q4:
    """One 4-bit matrix stack on the device: q uint8 [n][rows][K/2], s fp16 [n][rows][K/32].
    fmt "int4": offset-binary nibbles and their scales; "mxfp4": e2m1 codes and the scales
    moe_mxfp4_scales() expanded from the ue8m0 exponents (see upload_q4)."""
    q: "torch.Tensor"
    s: "torch.Tensor"
    fmt: str = "int4"

    def c(self) -> moe_q4:
        _need(self.q, 1, "q")
        _need(self.s, 2, "s")
        return moe_q4(self.q.data_ptr(), self.s.data_ptr())


def _fmt_of(*mats: Q4) -> int:
    fmts = {m.fmt for m in mats}
    if len(fmts) != 1 or next(iter(fmts)) not in WFMT:
        raise MoeError(-1, f"gate, up and down must share one known weight format, got {sorted(fmts)}")
    return WFMT[fmts.pop()]


@dataclass
class Experts:
    E: int
    H: int
    I: int
    gate: Q4
    up: Q4
    down: Q4

    def c(self) -> moe_experts:
        return moe_experts(self.E, self.H, self.I, self.gate.c(), self.up.c(), self.down.c(),
                           _fmt_of(self.gate, self.up, self.down))


@dataclass
class Shared:
    I_sh: int
    gate: Q4
    up: Q4
    down: Q4
    g: Optional["torch.Tensor"] = None  # bf16 [H] or None (ungated)

    def c(self) -> moe_shared:
        _need(self.g, 2, "g")
        return moe_shared(self.I_sh, self.gate.c(), self.up.c(), self.down.c(), _ptr(self.g),
                          _fmt_of(self.gate, self.up, self.down))


def _workspace(nbytes: int, device):
    import torch
    return torch.zeros(max(int(nbytes), 4096), dtype=torch.uint8, device=device)


# ----------------------------------------------------------------------------- entry points

def moe_version() -> str:
    return lib().moe_version().decode()


def moe_mxfp4_scales(e8, s, ws, stream=None):
    """Expands ue8m0 exponents e8 (uint8, device) into the fp16 scales s = 2^(e - 128) the
    kernels read; an exponent outside [104, 140] is recorded in ws's status word."""
    _need(e8, 1, "e8")
    _need(s, 2, "s")
    if e8.numel() != s.numel():
        raise MoeError(-1, "e8 and s must have the same number of elements")
    _check(lib().moe_mxfp4_scales(_ptr(e8), e8.numel(), _ptr(s), _ptr(ws), ws.numel() * ws.element_size(),
                                  _stream(stream)), "moe_mxfp4_scales")
    return s


def upload_q4(q, s, fmt: str = "int4", device="cuda") -> Q4:
    """Device copy of one host matrix stack (numpy): q uint8 codes; s fp16 bits (int4) or
    ue8m0 exponent bytes (mxfp4, expanded on the device by moe_mxfp4_scales).  Synchronises
    and raises when an exponent is out of range."""
    import numpy as np
    import torch
    if fmt not in WFMT:
        raise MoeError(-1, f"unknown weight format {fmt!r}")
    qd = torch.from_numpy(np.ascontiguousarray(q, dtype=np.uint8)).to(device)
    if fmt == "int4":
        sd = torch.from_numpy(np.ascontiguousarray(s, dtype=np.uint16).view(np.int16)).to(device).view(torch.float16)
        return Q4(qd, sd, "int4")
    e8 = torch.from_numpy(np.ascontiguousarray(s, dtype=np.uint8)).to(device)
    sd = torch.empty(e8.shape, dtype=torch.float16, device=device)
    ws = _workspace(4096, device)
    moe_mxfp4_scales(e8, sd, ws)
    st = moe_device_status(ws)
    if st != 0:
        raise MoeError(st, "moe_mxfp4_scales: scale exponent outside [104, 140]")
    return Q4(qd, sd, "mxfp4")


def moe_router_logits(x, W_r, g, logits, stream=None):
    T, H = x.shape
    E = W_r.shape[0]
    for t, n, w in ((x, 2, "x"), (W_r, 2, "W_r"), (g, 2, "g"), (logits, 4, "logits")):
        _need(t, n, w)
    _check(lib().moe_router_logits(_ptr(x), _ptr(W_r), _ptr(g), T, H, E, _ptr(logits), _stream(stream)),
           "moe_router_logits")
    return logits


def moe_router_topk(logits, E: int, k: int, topk_ids, topk_w, stream=None):
    T, ld = logits.shape
    _need(logits, logits.element_size(), "logits")
    _need(topk_ids, 4, "topk_ids")
    _need(topk_w, 4, "topk_w")
    is_bf16 = 1 if logits.element_size() == 2 else 0
    _check(lib().moe_router_topk(_ptr(logits), is_bf16, ld, T, E, k, _ptr(topk_ids), _ptr(topk_w),
                                 _stream(stream)), "moe_router_topk")
    return topk_ids, topk_w


def moe_router_topk_v(logits, E: int, k: int, topk_ids, topk_w, sel_bias=None, renormalize: bool = True,
                      scale: float = 1.0, stream=None):
    """Router variants: selection over logits + sel_bias (fp32 [E] or None), weights from the
    unbiased softmax, renormalised over the picks or not, times scale."""
    T, ld = logits.shape
    _need(logits, logits.element_size(), "logits")
    _need(topk_ids, 4, "topk_ids")
    _need(topk_w, 4, "topk_w")
    if sel_bias is not None:
        _need(sel_bias, 4, "sel_bias")
    is_bf16 = 1 if logits.element_size() == 2 else 0
    _check(lib().moe_router_topk_v(_ptr(logits), is_bf16, ld, T, E, k, _ptr(sel_bias), 1 if renormalize else 0,
                                   float(scale), _ptr(topk_ids), _ptr(topk_w), _stream(stream)),
           "moe_router_topk_v")
    return topk_ids, topk_w


def moe_dispatch_workspace_size(T: int, k: int, E: int) -> int:
    return lib().moe_dispatch_workspace_size(T, k, E)


def moe_dispatch(topk_ids, E: int, counts, offsets, perm, inv, ws, stream=None):
    T, k = topk_ids.shape
    for t, w in ((topk_ids, "topk_ids"), (counts, "counts"), (offsets, "offsets"), (perm, "perm"), (inv, "inv")):
        _need(t, 4, w)
    _check(lib().moe_dispatch(_ptr(topk_ids), T, k, E, _ptr(counts), _ptr(offsets), _ptr(perm), _ptr(inv),
                              _ptr(ws), ws.numel(), _stream(stream)), "moe_dispatch")
    return counts, offsets, perm, inv


def moe_dispatch_static(topk_ids, E: int, counts, offsets, perm, inv, stream=None):
    """moe_dispatch without a workspace, for callers that cannot allocate device memory at call
    time; scratch lives in a fixed array inside the library, shared by every call on a device
    (overlapping calls race).  T*k is limited to 2**20."""
    T, k = topk_ids.shape
    for t, w in ((topk_ids, "topk_ids"), (counts, "counts"), (offsets, "offsets"), (perm, "perm"), (inv, "inv")):
        _need(t, 4, w)
    _check(lib().moe_dispatch_static(_ptr(topk_ids), T, k, E, _ptr(counts), _ptr(offsets), _ptr(perm), _ptr(inv),
                                     _stream(stream)), "moe_dispatch_static")
    return counts, offsets, perm, inv


def moe_expert_mlp_workspace_size(T: int, k: int, E: int, H: int, I: int) -> int:
    return lib().moe_expert_mlp_workspace_size(T, k, E, H, I)


def moe_expert_mlp(x, k: int, W: Experts, offsets, perm, rows, ws, arm: int = ARM_AUTO, stream=None):
    T = x.shape[0]
    _need(x, 2, "x")
    _need(rows, 4, "rows")
    cw = W.c()
    _check(lib().moe_expert_mlp(_ptr(x), T, k, C.byref(cw), _ptr(offsets), _ptr(perm), _ptr(rows), arm, _ptr(ws),
                                ws.numel(), _stream(stream)), "moe_expert_mlp")
    return rows


def moe_combine(rows, inv, topk_w, shared, residual, y, stream=None):
    T, k = topk_w.shape
    H = y.shape[1]
    for t, n, w in ((rows, 4, "rows"), (inv, 4, "inv"), (topk_w, 4, "topk_w"), (shared, 4, "shared"),
                    (residual, 2, "residual"), (y, 4, "y")):
        _need(t, n, w)
    _check(lib().moe_combine(_ptr(rows), _ptr(inv), _ptr(topk_w), _ptr(shared), _ptr(residual), T, k, H, _ptr(y),
                             _stream(stream)), "moe_combine")
    return y


def moe_workspace_size(T: int, E: int, k: int, H: int, I: int, I_sh: int = 0) -> int:
    return lib().moe_workspace_size(T, E, k, H, I, I_sh)


def moe_layer_forward(x, residual, W_r, W: Experts, sh: Optional[Shared], k: int, y, ws, topk_ids_out=None,
                      topk_w_out=None, arm: int = ARM_AUTO, stream=None):
    T = x.shape[0]
    for t, n, w in ((x, 2, "x"), (residual, 2, "residual"), (W_r, 2, "W_r"), (y, 4, "y"),
                    (topk_ids_out, 4, "topk_ids_out"), (topk_w_out, 4, "topk_w_out")):
        _need(t, n, w)
    cw = W.c()
    cs = sh.c() if sh is not None else None
    _check(lib().moe_layer_forward(_ptr(x), _ptr(residual), _ptr(W_r), C.byref(cw),
                                   C.byref(cs) if cs is not None else None, T, k, _ptr(y), _ptr(topk_ids_out),
                                   _ptr(topk_w_out), arm, _ptr(ws), ws.numel(), _stream(stream)),
           "moe_layer_forward")
    return y


def moe_rmsnorm(y, gamma, eps: float, y_norm, stream=None):
    """y_norm (bf16 [T][H]) = y / sqrt(mean(y^2) + eps) * gamma, per row of y (fp32 [T][H])."""
    T, H = y.shape
    _need(y, 4, "y")
    _need(gamma, 2, "gamma")
    _need(y_norm, 2, "y_norm")
    _check(lib().moe_rmsnorm(_ptr(y), _ptr(gamma), T, H, float(eps), _ptr(y_norm), _stream(stream)), "moe_rmsnorm")
    return y_norm


def moe_workspace_init(ws, stream=None):
    _check(lib().moe_workspace_init(_ptr(ws), ws.numel(), _stream(stream)), "moe_workspace_init")


def moe_workspace_test_timeout(ws, wait_limit_cycles: int, stream=None):
    """Test hook: the next tensor-arm gate/up kernel on this workspace uses this wait limit and
    withholds one copy in its first CTA, so a bounded wait runs out (cleared by
    moe_workspace_init)."""
    _check(lib().moe_workspace_test_timeout(_ptr(ws), ws.numel(), int(wait_limit_cycles), _stream(stream)),
           "moe_workspace_test_timeout")


def moe_device_status(ws, stream=None) -> int:
    out = C.c_int(0)
    _check(lib().moe_device_status(_ptr(ws), ws.numel(), C.byref(out), _stream(stream)), "moe_device_status")
    return out.value


def moe_launch_count() -> int:
    return int(lib().moe_launch_count())


def moe_profile_enable(on: bool = True):
    _check(lib().moe_profile_enable(1 if on else 0), "moe_profile_enable")


def moe_profile_read(max_n: int = 64, name_len: int = 64) -> dict:
    """{kernel name: (total device ms, launches)} since moe_profile_enable."""
    names = C.create_string_buffer(max_n * name_len)
    ms = (C.c_double * max_n)()
    la = (C.c_long * max_n)()
    n = C.c_int(0)
    _check(lib().moe_profile_read(max_n, names, name_len, ms, la, C.byref(n)), "moe_profile_read")
    out = {}
    for i in range(min(n.value, max_n)):
        nm = names.raw[i * name_len:(i + 1) * name_len].split(b"\0", 1)[0].decode()
        out[nm] = (ms[i], la[i])
    return out


# ----------------------------------------------------------------------------- convenience

class MoeLayer:
    """Device-resident weights of one layer plus a reusable workspace.

    ``forward(x, residual)`` runs moe_layer_forward on the current stream and returns y (fp32).
    """

    def __init__(self, W_r, experts: Experts, shared: Optional[Shared], k: int, max_T: int):
        self.W_r, self.experts, self.shared, self.k, self.max_T = W_r, experts, shared, k, max_T
        I_sh = shared.I_sh if shared is not None else 0
        self.ws_bytes = moe_workspace_size(max_T, experts.E, k, experts.H, experts.I, I_sh)
        self.ws = _workspace(self.ws_bytes, W_r.device)
        self._cw = experts.c()
        self._cs = shared.c() if shared is not None else None

    def forward(self, x, residual=None, y=None, topk_ids_out=None, topk_w_out=None, arm: int = ARM_AUTO,
                stream=None, norm_gamma=None, eps: float = 1e-6, y_norm=None):
        """y (fp32) = the layer; with norm_gamma and y_norm (bf16 [T][H]) also the RMSNorm of y."""
        import torch
        T = x.shape[0]
        if T > self.max_T:
            raise MoeError(-1, f"T={T} above this layer's workspace size (max_T={self.max_T})")
        if y is None:
            y = torch.empty((T, self.experts.H), dtype=torch.float32, device=x.device)
        if norm_gamma is not None:
            _check(lib().moe_layer_forward_norm(_ptr(x), _ptr(residual), _ptr(self.W_r), C.byref(self._cw),
                                                C.byref(self._cs) if self._cs is not None else None, T, self.k,
                                                _ptr(y), _ptr(norm_gamma), float(eps), _ptr(y_norm),
                                                _ptr(topk_ids_out), _ptr(topk_w_out), arm, _ptr(self.ws),
                                                self.ws.numel(), _stream(stream)), "moe_layer_forward_norm")
            return y
        _check(lib().moe_layer_forward(_ptr(x), _ptr(residual), _ptr(self.W_r), C.byref(self._cw),
                                       C.byref(self._cs) if self._cs is not None else None, T, self.k, _ptr(y),
                                       _ptr(topk_ids_out), _ptr(topk_w_out), arm, _ptr(self.ws), self.ws.numel(),
                                       _stream(stream)), "moe_layer_forward")
        return y
