"""Whole-layer pin of the oracle: an fp64 numpy restatement of the routed MoE layer, written
from the definitions alone and calling nothing in oracle/, must agree with
oracle.layer_forward to 1e-12.

The restatement takes each step in its plainest library form, so that it shares no loop,
helper or decode with the C oracle:
  * weights: the nibbles unpacked with numpy bit operations (even column in the low
    nibble, value = nibble - 8; colibri PR #418 "Vulkan backend: expert tier + dense + MLA
    attention on any Vulkan 1.2 GPU", Correctness), times numpy's own IEEE-half decode of
    the per-32-column scale ("Grouped scales in the Vulkan kernels");
  * router: a dense matmul, rounded to fp32 (the router consumes fp32 logits), selection by
    a stable argsort on the negated logits (largest first, the lower index first on a tie;
    vllm.cpp PR #481 "gate(#378): the first DEVICE run of the warp MoE router"), picks
    written in ascending expert id, weights = softmax over all E renormalised over the picks
    (daScript PR #3988 "dasLLAMA vulkan: a MoE that fits the card ...", routed-block commit);
  * experts: dense matmuls per expert on the tokens that picked it, SwiGLU h = silu(g) * u
    (colibri PR #418, Summary);
  * shared expert scaled by sigmoid(x . g), weight 1 when ungated, and the combine onto the
    residual (daScript PR #3988, decode span and combine-folded residual commits).
The restatement never dispatches: it walks the experts and adds each pick's weighted row to
its token directly, so the oracle's histogram / scan / permutation / inverse map are pinned
too (a wrong inverse would send a row to the wrong token)."""
import numpy as np
import pytest

import oracle
from mixture_experts_layer_09_gb300 import inputs as gen

TOL = 1e-12


def _bf16(bits):
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _dequant(q, s):
    """One int4 matrix: q [rows][K/2] uint8, s [rows][K/32] fp16 bits -> fp64 [rows][K]."""
    rows, half = q.shape
    vals = np.empty((rows, 2 * half), dtype=np.float64)
    vals[:, 0::2] = (q & 0x0F).astype(np.float64) - 8.0
    vals[:, 1::2] = (q >> 4).astype(np.float64) - 8.0
    scale = np.asarray(s, dtype=np.uint16).view(np.float16).astype(np.float64)
    return vals * np.repeat(scale, 32, axis=1)


def _swiglu_mlp(xs, Wg, Wu, Wd):
    g = xs @ Wg.T
    u = xs @ Wu.T
    h = g / (1.0 + np.exp(-g)) * u
    return h @ Wd.T


def numpy_layer(inp):
    wl = inp.wl
    x = _bf16(inp.x)
    logits = (x @ _bf16(inp.W_r).T).astype(np.float32).astype(np.float64)
    picks = np.argsort(-logits, axis=1, kind="stable")[:, :wl.k]
    ids = np.sort(picks, axis=1).astype(np.int32)
    p = np.exp(logits - logits.max(axis=1, keepdims=True))
    p /= p.sum(axis=1, keepdims=True)
    sel = np.take_along_axis(p, ids, axis=1)
    w = sel / sel.sum(axis=1, keepdims=True)
    y = np.zeros_like(x) if inp.residual is None else _bf16(inp.residual).copy()
    routed = np.zeros_like(x)
    ex = inp.experts
    for e in np.unique(ids):
        tok, slot = np.nonzero(ids == e)
        o = _swiglu_mlp(x[tok], _dequant(ex.gate.q[e], ex.gate.s[e]), _dequant(ex.up.q[e], ex.up.s[e]),
                        _dequant(ex.down.q[e], ex.down.s[e]))
        routed[tok] += w[tok, slot][:, None] * o
    y += routed
    if inp.shared is not None:
        sh = inp.shared
        ys = _swiglu_mlp(x, _dequant(sh.gate.q[0], sh.gate.s[0]), _dequant(sh.up.q[0], sh.up.s[0]),
                         _dequant(sh.down.q[0], sh.down.s[0]))
        if sh.g is not None:
            ys *= (1.0 / (1.0 + np.exp(-(x @ _bf16(sh.g)))))[:, None]
        y += ys
    return ids, w, y


def _close(a, b):
    scale = max(float(np.max(np.abs(b))), 1e-300)
    return float(np.max(np.abs(a - b))) / scale


@pytest.mark.parametrize("name,over", [
    ("tiny", {}),
    ("tiny", {"I_sh": 64}),                                          # gated shared expert
    ("tiny", {"I_sh": 96, "gated_shared": False, "residual": False, "T": 9}),
    ("qwen3_30b_decode_t1", {}),
    ("qwen3_30b_decode_t4", {}),
    ("qwen3_30b_decode_t16", {}),
])
def test_oracle_layer_equals_numpy_restatement(name, over):
    wl = gen.WORKLOADS[name]
    wl = gen.Workload(**{**wl.__dict__, "extra": {}, **over})
    inp = gen.draw_layer(wl)
    ref = oracle.layer_forward(inp)
    ids, w, y = numpy_layer(inp)
    assert np.array_equal(ids, ref["ids"]), "selected experts differ"
    assert _close(w, ref["w"]) <= TOL
    assert _close(y, ref["y"]) <= TOL, f"y differs by {_close(y, ref['y']):.3e} of max|y|"


def test_restatement_sees_a_planted_slip():
    """The comparison is sharp enough to see a one-row slip: dropping one pick's row from the
    restatement moves y far beyond the tolerance."""
    inp = gen.draw_layer(gen.WORKLOADS["tiny"])
    ref = oracle.layer_forward(inp)
    ids, w, y = numpy_layer(inp)
    ex = inp.experts
    e = int(ids[0, 0])
    o = _swiglu_mlp(_bf16(inp.x[:1]), _dequant(ex.gate.q[e], ex.gate.s[e]), _dequant(ex.up.q[e], ex.up.s[e]),
                    _dequant(ex.down.q[e], ex.down.s[e]))
    y[0] -= w[0, 0] * o[0]
    assert _close(y, ref["y"]) > 1e-6


@pytest.mark.parametrize("name,over", [("tiny", {"I_sh": 64, "T": 23}), ("qwen3_30b_decode_t4", {})])
def test_oracle_threads_do_not_change_results(name, over):
    """Rows spread over worker threads are computed by the same sequential loops: results are
    bit-identical for one thread and for several."""
    wl = gen.WORKLOADS[name]
    inp = gen.draw_layer(gen.Workload(**{**wl.__dict__, "extra": {}, **over}))
    n0 = oracle.get_threads()
    try:
        oracle.set_threads(1)
        a = oracle.layer_forward(inp)
        oracle.set_threads(5)
        b = oracle.layer_forward(inp)
    finally:
        oracle.set_threads(n0)
    for key in ("logits", "ids", "w", "y"):
        assert np.array_equal(a[key], b[key]), key
