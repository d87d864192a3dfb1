"""Test-side helpers: margin-enforced inputs (via the oracle), device upload, tolerance.

Margin rule: every token's k-th and (k+1)-th largest router logits differ by at least 1e-3,
so no near-tie can flip the routed set between the fp64 oracle and the fp32 kernels.  A token
that misses it gets its hidden row (or, for the router-only sweep, its logit row) redrawn from
the next sub-seed (seed, row, attempt), up to 64 attempts.
"""
from __future__ import annotations

import numpy as np

import oracle
from mixture_experts_layer_09_gb300 import inputs as gen

MARGIN = 1e-3
REL_L2_TOL = 1e-3
MAX_ABS_FRAC = 2e-3


def kth_margin(row: np.ndarray, k: int) -> float:
    if k >= row.shape[0]:
        return np.inf
    s = np.sort(row)[::-1]
    return float(s[k - 1] - s[k])


def enforce_margin_x(inp: gen.LayerInputs, max_attempts: int = 64) -> gen.LayerInputs:
    wl = inp.wl
    logits = oracle.router_logits(inp.x, inp.W_r)
    attempts = {}
    for t in range(wl.T):
        a = 0
        while kth_margin(logits[t], wl.k) < MARGIN:
            a += 1
            if a > max_attempts:
                raise RuntimeError(f"token {t}: no margin after {max_attempts} redraws")
            inp.x[t] = gen.draw_x_row(wl.seed, t, wl.H, a)
            if wl.zipf > 0:
                inp.x[t, 0] = gen.ONE_BF16  # keep the bias channel
            logits[t] = oracle.router_logits(inp.x[t:t + 1], inp.W_r)[0]
        if a:
            attempts[t] = a
    inp.wl.extra["redrawn_rows"] = len(attempts)
    return inp


def margin_logits(seed: int, T: int, E: int, k: int, max_attempts: int = 64) -> np.ndarray:
    L = gen.draw_logits(seed, T, E)
    for t in range(T):
        a = 0
        while kth_margin(gen.bf16_to_f32(L[t]).astype(np.float64), k) < MARGIN:
            a += 1
            if a > max_attempts:
                raise RuntimeError(f"logit row {t}: no margin after {max_attempts} redraws")
            L[t] = gen.draw_logit_row(seed, t, E, a)
    return L


def layer(name: str, seed: int = 0, **over) -> gen.LayerInputs:
    wl = gen.WORKLOADS[name]
    wl = gen.Workload(**{**wl.__dict__, "extra": {}, "seed": seed, **over})
    return enforce_margin_x(gen.draw_layer(wl))


def bucket_sample_tokens(inp: gen.LayerInputs, stride: int = 64) -> np.ndarray:
    """Tokens to compare on a layer too large for the oracle to finish whole: every expert
    bucket (from the oracle's own routing of all tokens) contributes its first and last
    dispatched row and every `stride`-th row between, and the tokens of those rows are taken.
    Buckets are cut into token tiles of at most 256 rows, so every tile of every expert holds
    sampled rows at several positions; the tokens fall across the whole batch, so every tile
    of the shared expert is sampled too."""
    wl = inp.wl
    logits = oracle.router_logits(inp.x, inp.W_r).astype(np.float32).astype(np.float64)
    ids, _ = oracle.router_topk(logits, wl.k)
    _, offsets, perm, _ = oracle.dispatch(ids, wl.E)
    rows = []
    for e in range(wl.E):
        b0, b1 = int(offsets[e]), int(offsets[e + 1])
        if b1 > b0:
            rows.extend(range(b0, b1, stride))
            rows.append(b1 - 1)
    return np.unique(perm[np.asarray(rows, dtype=np.int64)] // wl.k)


def rel_errors(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    err = got - ref
    rel_l2 = float(np.linalg.norm(err) / max(np.linalg.norm(ref), 1e-300))
    max_abs = float(np.max(np.abs(err))) if err.size else 0.0
    ref_max = float(np.max(np.abs(ref))) if ref.size else 0.0
    return rel_l2, max_abs, ref_max


def assert_close(got, ref, what="value", rel_l2_tol=REL_L2_TOL, max_abs_frac=MAX_ABS_FRAC):
    rel_l2, max_abs, ref_max = rel_errors(got, ref)
    assert np.all(np.isfinite(np.asarray(got))), f"{what}: non-finite output"
    assert rel_l2 <= rel_l2_tol, f"{what}: rel-L2 {rel_l2:.3e} > {rel_l2_tol}"
    assert max_abs <= max_abs_frac * ref_max, f"{what}: max-abs {max_abs:.3e} > {max_abs_frac} * {ref_max:.3e}"
    return rel_l2, max_abs


# ----------------------------------------------------------------------------- device upload

def dev(a: np.ndarray, dtype=None):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.view(dtype)
    return t.cuda()


def upload(inp: gen.LayerInputs):
    """Device copies: (x, residual, W_r, Experts, Shared|None) as binding objects."""
    import torch
    import mixture_experts_layer_09_gb300 as moe

    def q4(m: gen.Q4):
        return moe.upload_q4(m.q, m.s, m.fmt)

    ex = inp.experts
    E = moe.Experts(ex.E, ex.H, ex.I, q4(ex.gate), q4(ex.up), q4(ex.down))
    S = None
    if inp.shared is not None:
        sh = inp.shared
        g = dev(sh.g.view(np.int16), torch.bfloat16) if sh.g is not None else None
        S = moe.Shared(sh.I_sh, q4(sh.gate), q4(sh.up), q4(sh.down), g)
    x = dev(inp.x.view(np.int16), torch.bfloat16)
    r = dev(inp.residual.view(np.int16), torch.bfloat16) if inp.residual is not None else None
    W_r = dev(inp.W_r.view(np.int16), torch.bfloat16)
    return x, r, W_r, E, S


def poison(t):
    """Fill an output with a NaN / sentinel pattern before a launch."""
    import torch
    if t.dtype in (torch.float32, torch.float16, torch.bfloat16):
        t.fill_(float("nan"))
    else:
        t.fill_(0x7fffffff if t.dtype == torch.int32 else -1)
    return t
