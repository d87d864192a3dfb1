"""Pins of the fp64 oracle against what the pages and the mathematics fix.

Each pin would fail under a plausible slip in the oracle: a swapped nibble order,
an off-by-one scale group, a wrong tie-break, a dropped renormalisation, an
unstable bucket order, a missing silu, a transposed matrix, the shared gate
applied twice, a slot read through perm instead of inv.
"""
import json
import math
import os

import numpy as np
import pytest

from mixture_experts_layer_09_gb300 import inputs as gen

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _gold(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


# --------------------------------------------------------------------------- scalar decodes

def test_f16_decode_matches_ieee(oracle_lib):
    # fixed points and a library routine (numpy's IEEE binary16) on every bit pattern
    assert oracle_lib.f16_to_f64(0x3C00) == 1.0
    assert oracle_lib.f16_to_f64(0xC000) == -2.0
    assert oracle_lib.f16_to_f64(0x7BFF) == 65504.0
    assert oracle_lib.f16_to_f64(0x0001) == 2.0 ** -24
    assert oracle_lib.f16_to_f64(0x03FF) == 1023 * 2.0 ** -24
    allbits = np.arange(0, 65536, dtype=np.uint32)
    finite = [b for b in allbits[::7] if (b >> 10) & 0x1F != 31]
    ref = np.array(finite, dtype=np.uint16).view(np.float16).astype(np.float64)
    got = np.array([oracle_lib.f16_to_f64(int(b)) for b in finite])
    assert np.array_equal(ref, got)


def test_bf16_decode(oracle_lib):
    assert oracle_lib.bf16_to_f64(0x3F80) == 1.0
    assert oracle_lib.bf16_to_f64(0xC040) == -3.0
    assert oracle_lib.bf16_to_f64(0x0001) == float(np.array([1], np.uint32).view(np.float32)[0]) * 65536


def test_nibble_decode_golden(oracle_lib):
    d = _gold("nibble_decode.json")
    K = d["K"]
    q = np.full((1, K // 2), int(d["default_byte"], 16), dtype=np.uint8)
    for pos, b in d["bytes"].items():
        q[0, int(pos)] = int(b, 16)
    s = np.array([[int(v, 16) for v in d["scales_f16"]]], dtype=np.uint16)
    w = oracle_lib.dequant(q, s, 1, K)
    for col, val in d["expected"].items():
        assert w[0, int(col)] == val, col
    # every column not named is zero
    named = {int(c) for c in d["expected"]}
    others = [c for c in range(K) if c not in named and c // 2 not in {int(p) for p in d["bytes"]}]
    assert np.all(w[0, others] == 0.0)


def test_scale_group_boundary(oracle_lib):
    # all nibbles 9 (value +1): each column equals its group's scale; group g covers 32g..32g+31
    K, rows = 128, 3
    q = np.full((rows, K // 2), 0x99, dtype=np.uint8)
    sv = np.array([[0.5, 0.25, 2.0, 4.0], [1.0, 1.5, 3.0, 0.125], [8.0, 0.75, 0.0625, 1.0]])
    s = gen.f16_bits(sv)
    w = oracle_lib.dequant(q, s, rows, K)
    for r in range(rows):
        for c in range(K):
            assert w[r, c] == sv[r, c // 32]


# --------------------------------------------------------------------------- router

def _brute_topk(l, k):
    order = sorted(range(len(l)), key=lambda e: (-l[e], e))
    return sorted(order[:k])


def test_topk_golden(oracle_lib):
    for c in _gold("topk_ties.json")["cases"]:
        ids, w = oracle_lib.router_topk(np.array([c["logits"]]), c["k"])
        assert ids[0].tolist() == c["ids"], c
        assert np.allclose(w[0], c["w"], rtol=0, atol=1e-15), c


@pytest.mark.parametrize("E,k", [(8, 2), (32, 8), (64, 8), (256, 8), (256, 32), (60, 4), (7, 7), (9, 1)])
def test_topk_vs_full_sort(oracle_lib, E, k):
    g = gen.rng(123, E, k)
    T = 64
    cont = g.normal(size=(T, E)) * 2
    ties = g.integers(0, 8, size=(T, E)).astype(np.float64) * 0.25  # tie-heavy rows
    for logits in (cont, ties):
        ids, w = oracle_lib.router_topk(logits, k)
        for t in range(T):
            assert ids[t].tolist() == _brute_topk(list(logits[t]), k)
            # renormalised: weights sum to one, lie in (0, 1], and keep the softmax ratios
            assert abs(w[t].sum() - 1.0) <= 1e-12
            assert np.all(w[t] > 0) and np.all(w[t] <= 1.0)
            l = logits[t, ids[t]]
            for j in range(1, k):
                assert math.isclose(w[t, j] / w[t, 0], math.exp(l[j] - l[0]), rel_tol=1e-12)


def test_topk_special_cases(oracle_lib):
    g = gen.rng(7)
    logits = g.normal(size=(16, 12))
    ids, w = oracle_lib.router_topk(logits, 1)
    assert np.all(w == 1.0)
    assert np.array_equal(ids[:, 0], np.argmax(logits, axis=1))  # library argmax: first maximum
    ids, w = oracle_lib.router_topk(logits, 12)
    assert np.array_equal(ids, np.tile(np.arange(12), (16, 1)))
    # k = E: the weights are the full softmax, which is invariant to a shift of the row
    ids2, w2 = oracle_lib.router_topk(logits + 3.5, 12)
    assert np.allclose(w, w2, atol=1e-14)
    with pytest.raises(ValueError):
        oracle_lib.router_topk(np.array([[0.0, np.nan]]), 1)
    with pytest.raises(ValueError):
        oracle_lib.router_topk(np.array([[0.0, 1.0]]), 3)


def test_router_logits_is_a_matmul(oracle_lib):
    g = gen.rng(5)
    x = gen.bf16_bits(g.normal(size=(3, 64)))
    W = gen.bf16_bits(g.normal(size=(5, 64)) * 0.02)
    gv = gen.bf16_bits(g.normal(size=64) * 0.02)
    out = oracle_lib.router_logits(x, W, gv)
    xf = gen.bf16_to_f32(x).astype(np.float64)
    ref = xf @ gen.bf16_to_f32(W).astype(np.float64).T   # library matmul
    assert out.shape == (3, 6)
    assert np.allclose(out[:, :5], ref, rtol=0, atol=1e-12)
    assert np.allclose(out[:, 5], xf @ gen.bf16_to_f32(gv).astype(np.float64), rtol=0, atol=1e-12)


# --------------------------------------------------------------------------- dispatch

def test_dispatch_golden(oracle_lib):
    d = _gold("dispatch_small.json")
    counts, offsets, perm, inv = oracle_lib.dispatch(np.array(d["ids"]), d["E"])
    assert counts.tolist() == d["counts"]
    assert offsets.tolist() == d["offsets"]
    assert perm.tolist() == d["perm"]
    assert inv.tolist() == d["inv"]


@pytest.mark.parametrize("T,E,k", [(1, 8, 2), (5, 8, 8), (64, 60, 4), (300, 256, 8), (129, 32, 8)])
def test_dispatch_invariants(oracle_lib, T, E, k):
    g = gen.rng(11, T, E, k)
    ids = np.stack([np.sort(g.choice(E, size=k, replace=False)) for _ in range(T)]).astype(np.int32)
    counts, offsets, perm, inv = oracle_lib.dispatch(ids, E)
    flat = ids.reshape(-1)
    assert counts.sum() == T * k and offsets[0] == 0 and offsets[E] == T * k
    assert np.all(np.diff(offsets) == counts) and np.all(counts >= 0)
    assert np.array_equal(np.sort(perm), np.arange(T * k))          # a permutation
    assert np.array_equal(inv[perm], np.arange(T * k))              # inv o perm = id
    tok = perm // k
    assert np.array_equal(np.bincount(tok, minlength=T), np.full(T, k))  # each token k times
    for e in range(E):
        b = perm[offsets[e]:offsets[e + 1]]
        assert np.all(flat[b] == e)
        assert np.all(np.diff(b) > 0)                                 # stable: ascending slots
    # brute force: a stable sort of slot indices by expert id (library routine)
    assert np.array_equal(perm, np.argsort(flat, kind="stable"))


# --------------------------------------------------------------------------- expert MLP

def _const_q4(rows, K, nib, scale_bits):
    q = np.full((rows, K // 2), nib | (nib << 4), dtype=np.uint8)
    s = np.full((rows, K // 32), scale_bits, dtype=np.uint16)
    return q, s


def _silu(z):
    return z / (1.0 + math.exp(-z))


def test_mlp_all_zero_weights(oracle_lib):
    H, I = 64, 32
    x = gen.bf16_bits(gen.rng(1).normal(size=H))
    z = _const_q4(I, H, 8, 0x3C00)
    d = _const_q4(H, I, 8, 0x3C00)
    o = oracle_lib.expert_row(x, z, z, d, H, I)
    assert np.all(o == 0.0)


@pytest.mark.parametrize("cg,cu,cd", [(9, 10, 7), (3, 12, 15), (0, 15, 8)])
def test_mlp_constant_weights_closed_form(oracle_lib, cg, cu, cd):
    H, I = 96, 64
    x = gen.bf16_bits(gen.rng(2, cg).normal(size=H))
    X = float(gen.bf16_to_f32(x).astype(np.float64).sum())
    sg, su, sd = 0.5, 0.25, 0.125
    gate = _const_q4(I, H, cg, int(gen.f16_bits([sg])[0]))
    up = _const_q4(I, H, cu, int(gen.f16_bits([su])[0]))
    down = _const_q4(H, I, cd, int(gen.f16_bits([sd])[0]))
    o = oracle_lib.expert_row(x, gate, up, down, H, I)
    g = (cg - 8) * sg * X
    u = (cu - 8) * su * X
    h = _silu(g) * u
    expect = (cd - 8) * sd * I * h
    assert np.allclose(o, expect, rtol=1e-13, atol=1e-13)


def test_mlp_single_weight_hand_value(oracle_lib):
    # gate row 0 = [+2, +1, 0...] (nibbles 10, 9), up row 0 = [+3, 0...] (nibble 11),
    # down column 0 = (n % 5) - 2; x = [1, 2, 0...]; scales 1.0
    H = I = 32
    x = np.zeros(H, dtype=np.uint16)
    x[0], x[1] = gen.bf16_bits([1.0, 2.0])
    gq, gs = _const_q4(I, H, 8, 0x3C00)
    uq, us = _const_q4(I, H, 8, 0x3C00)
    dq, ds = _const_q4(H, I, 8, 0x3C00)
    gq[0, 0] = 0x9A
    uq[0, 0] = 0x8B
    for n in range(H):
        dq[n, 0] = 0x80 | (6 + n % 5)
    o = oracle_lib.expert_row(x, (gq, gs), (uq, us), (dq, ds), H, I)
    h0 = 4.0 / (1.0 + math.exp(-4.0)) * 3.0
    expect = np.array([((n % 5) - 2) * h0 for n in range(H)])
    assert np.allclose(o, expect, rtol=1e-14, atol=0)


def test_mlp_is_dense_restatement(oracle_lib):
    # a dequantised-matrix restatement with library matmuls on a random expert
    H, I = 64, 96
    ex = gen.draw_experts(3, 1, H, I)
    x = gen.bf16_bits(gen.rng(4).normal(size=H))
    o = oracle_lib.expert_row(x, (ex.gate.q[0], ex.gate.s[0]), (ex.up.q[0], ex.up.s[0]),
                              (ex.down.q[0], ex.down.s[0]), H, I)
    Wg = oracle_lib.dequant(ex.gate.q[0], ex.gate.s[0], I, H)
    Wu = oracle_lib.dequant(ex.up.q[0], ex.up.s[0], I, H)
    Wd = oracle_lib.dequant(ex.down.q[0], ex.down.s[0], H, I)
    xf = gen.bf16_to_f32(x).astype(np.float64)
    g, u = Wg @ xf, Wu @ xf
    ref = Wd @ (g / (1 + np.exp(-g)) * u)
    assert np.allclose(o, ref, rtol=1e-12, atol=1e-12)


def test_dequant_independent_of_layout_helpers(oracle_lib):
    # unpack nibbles with numpy bit operations and compare (nibble order + group pin)
    ex = gen.draw_experts(9, 1, 64, 32)
    q, s = ex.gate.q[0], ex.gate.s[0]
    lo, hi = (q & 0xF).astype(np.int64), (q >> 4).astype(np.int64)
    nib = np.empty((q.shape[0], q.shape[1] * 2), dtype=np.int64)
    nib[:, 0::2], nib[:, 1::2] = lo, hi
    ref = (nib - 8) * np.repeat(gen.f16_to_f32(s).astype(np.float64), 32, axis=1)
    assert np.array_equal(oracle_lib.dequant(q, s, 32, 64), ref)


# --------------------------------------------------------------------------- shared expert, combine

def test_shared_gate(oracle_lib):
    H, I = 64, 32
    sh = gen.draw_shared(5, H, I, gated=True)
    x = gen.draw_x(5, 3, H)
    ung = gen.Shared(sh.I_sh, sh.gate, sh.up, sh.down, None)
    y1 = oracle_lib.shared_expert(x, ung)
    # g = 0 -> sigmoid(0) = 1/2 exactly
    zero = gen.Shared(sh.I_sh, sh.gate, sh.up, sh.down, np.zeros(H, dtype=np.uint16))
    yh = oracle_lib.shared_expert(x, zero)
    assert np.array_equal(yh, y1 * 0.5)
    yg = oracle_lib.shared_expert(x, sh)
    z = gen.bf16_to_f32(x).astype(np.float64) @ gen.bf16_to_f32(sh.g).astype(np.float64)
    assert np.allclose(yg, y1 / (1 + np.exp(-z))[:, None], rtol=1e-14, atol=1e-14)
    # ungated shared expert row == a routed expert row with the same matrices
    o = oracle_lib.expert_row(x[1], (sh.gate.q[0], sh.gate.s[0]), (sh.up.q[0], sh.up.s[0]),
                              (sh.down.q[0], sh.down.s[0]), H, I)
    assert np.array_equal(o, y1[1])


def test_combine_hand_and_zero_weight(oracle_lib):
    # T=2, k=2, H=3; rows in dispatch order; inv maps slot -> row
    rows = np.array([[1., 2., 3.], [10., 20., 30.], [100., 200., 300.], [-1., -1., -1.]])
    inv = np.array([2, 0, 3, 1], dtype=np.int32)
    w = np.array([[0.25, 0.75], [0.5, 0.5]])
    sh = np.array([[1., 1., 1.], [2., 2., 2.]])
    r = gen.bf16_bits(np.array([[0.5, 0.5, 0.5], [-4., 0., 4.]]))
    y = oracle_lib.combine(rows, inv, w, sh, r)
    expect = np.array([[1 + 0.25 * 100 + 0.75 * 1 + 0.5, 1 + 50 + 1.5 + 0.5, 1 + 75 + 2.25 + 0.5],
                       [2 - 0.5 + 5 - 4, 2 - 0.5 + 10, 2 - 0.5 + 15 + 4]])
    assert np.allclose(y, expect, rtol=0, atol=1e-12)
    # a zero weight: perturbing that slot's row leaves y bit-identical
    w0 = w.copy()
    w0[0, 1] = 0.0
    ya = oracle_lib.combine(rows, inv, w0, sh, r)
    rows2 = rows.copy()
    rows2[inv[1]] += 12345.0
    yb = oracle_lib.combine(rows2, inv, w0, sh, r)
    assert np.array_equal(ya, yb)


def test_layer_composition_and_token_mask(oracle_lib):
    wl = gen.Workload("t", 6, 64, 32, 8, 2, I_sh=32)
    inp = gen.draw_layer(wl)
    out = oracle_lib.layer_forward(inp)
    # recompose from the stage functions
    logits = oracle_lib.router_logits(inp.x, inp.W_r).astype(np.float32).astype(np.float64)
    assert np.array_equal(logits, out["logits"])
    ids, w = oracle_lib.router_topk(logits, wl.k)
    assert np.array_equal(ids, out["ids"])
    counts, offsets, perm, inv = oracle_lib.dispatch(ids, wl.E)
    rows = oracle_lib.expert_mlp(inp.x, inp.experts, ids, perm)
    ysh = oracle_lib.shared_expert(inp.x, inp.shared)
    y = oracle_lib.combine(rows, inv, w, ysh, inp.residual)
    assert np.array_equal(y, out["y"])
    # per-row restatement: each token's output is its own k experts + gated shared + residual
    t = 3
    acc = np.zeros(wl.H)
    for j in range(wl.k):
        e = ids[t, j]
        acc += w[t, j] * oracle_lib.expert_row(inp.x[t], (inp.experts.gate.q[e], inp.experts.gate.s[e]),
                                               (inp.experts.up.q[e], inp.experts.up.s[e]),
                                               (inp.experts.down.q[e], inp.experts.down.s[e]), wl.H, wl.I)
    acc += ysh[t] + gen.bf16_to_f32(inp.residual[t])
    assert np.allclose(acc, out["y"][t], rtol=1e-13, atol=1e-12)
    # token mask computes the same values for the selected tokens
    mask = np.zeros(wl.T, dtype=np.uint8)
    mask[[1, 4]] = 1
    outm = oracle_lib.layer_forward(inp, token_mask=mask)
    assert np.array_equal(outm["y"][[1, 4]], out["y"][[1, 4]])


def test_planted_mistakes_are_caught(oracle_lib):
    """A swapped nibble order or a missing renormalisation would change these values."""
    # swapped nibble order: byte 0x8F must give col0 = +7, not 0
    q = np.full((1, 16), 0x88, dtype=np.uint8)
    q[0, 0] = 0x8F
    w = oracle_lib.dequant(q, np.full((1, 1), 0x3C00, dtype=np.uint16), 1, 32)
    assert w[0, 0] == 7.0 and w[0, 1] == 0.0
    # renormalisation: top-2 of [0, 0, 0, 0] gives 1/2 each, not 1/4
    _, wt = oracle_lib.router_topk(np.zeros((1, 4)), 2)
    assert np.allclose(wt, 0.5)


# ----------------------------------------------------------------------------- router variants
def test_router_variants_closed_form(oracle_lib):
    """logits ln(1..4): softmax = (1 2 3 4)/10; top-2 = experts 2, 3."""
    import math
    L = np.log(np.array([[1.0, 2.0, 3.0, 4.0]]))
    ids, w = oracle_lib.router_topk_v(L, 2, renormalize=False)
    assert ids.tolist() == [[2, 3]]
    np.testing.assert_allclose(w, [[0.3, 0.4]], rtol=1e-14)
    ids, w = oracle_lib.router_topk_v(L, 2, renormalize=True)
    np.testing.assert_allclose(w, [[3 / 7, 4 / 7]], rtol=1e-14)
    ids, w = oracle_lib.router_topk_v(L, 2, renormalize=True, scale=2.5)
    np.testing.assert_allclose(w, [[7.5 / 7, 10 / 7]], rtol=1e-14)
    ids, w = oracle_lib.router_topk_v(L, 2, renormalize=False, scale=2.5)
    np.testing.assert_allclose(w, [[0.75, 1.0]], rtol=1e-14)
    assert math.isclose(float(w.sum()), 1.75, rel_tol=1e-14)


def test_router_variants_bias_moves_selection_only(oracle_lib):
    L = np.array([[0.0, 0.0, 0.0, 1.0]])
    bias = np.array([5.0, 0.0, 0.0, 0.0])
    ids, w = oracle_lib.router_topk_v(L, 1, bias=bias, renormalize=False)
    assert ids.tolist() == [[0]]
    np.testing.assert_allclose(w, [[1.0 / (3.0 + np.e)]], rtol=1e-14)  # unbiased softmax of expert 0
    ids, w = oracle_lib.router_topk_v(L, 1, bias=bias, renormalize=True)
    np.testing.assert_allclose(w, [[1.0]], rtol=1e-14)
    # a tie on the biased scores keeps the lower index
    ids, _ = oracle_lib.router_topk_v(np.array([[1.0, 0.0]]), 1, bias=np.array([0.0, 1.0]))
    assert ids.tolist() == [[0]]


def test_router_variants_brute_force_selection(oracle_lib):
    g = np.random.default_rng(11)
    for _ in range(200):
        E = int(g.integers(2, 9))
        k = int(g.integers(1, E + 1))
        L = g.choice([-1.0, 0.0, 0.5, 1.0], size=(1, E))
        b = g.choice([0.0, 0.5, -0.5], size=E)
        ids, _ = oracle_lib.router_topk_v(L, k, bias=b, renormalize=bool(g.integers(0, 2)))
        s = L[0] + b
        order = sorted(range(E), key=lambda e: (-s[e], e))[:k]
        assert ids[0].tolist() == sorted(order)


def test_router_variants_reduce_to_the_softmax_router(oracle_lib):
    L = np.random.default_rng(12).normal(0, 2, size=(16, 60))
    ids0, w0 = oracle_lib.router_topk(L, 4)
    ids1, w1 = oracle_lib.router_topk_v(L, 4)
    assert np.array_equal(ids0, ids1)
    np.testing.assert_allclose(w1, w0, rtol=1e-15)


# ----------------------------------------------------------------------------- RMSNorm after the combine
def test_rmsnorm_closed_forms(oracle_lib):
    one = gen.bf16_bits(np.ones(2, np.float32))
    # y = (3, 4): mean of squares 12.5
    out = oracle_lib.rmsnorm(np.array([[3.0, 4.0]]), one, 0.0)
    np.testing.assert_allclose(out, [[3 / math.sqrt(12.5), 4 / math.sqrt(12.5)]], rtol=1e-15)
    # gamma scales each column; eps enters under the root
    g = gen.bf16_bits(np.array([2.0, 0.5], np.float32))
    out = oracle_lib.rmsnorm(np.array([[3.0, 4.0]]), g, 0.5)
    np.testing.assert_allclose(out, [[6 / math.sqrt(13.0), 2 / math.sqrt(13.0)]], rtol=1e-15)
    # a zero row stays zero; a constant row c normalises to sign(c) when eps = 0
    out = oracle_lib.rmsnorm(np.array([[0.0, 0.0], [-7.0, -7.0]]), one, 1e-6)
    assert np.all(out[0] == 0.0)
    np.testing.assert_allclose(out[1], [-7 / math.sqrt(49 + 1e-6)] * 2, rtol=1e-15)


def test_rmsnorm_is_scale_invariant(oracle_lib):
    y = np.random.default_rng(13).normal(0, 1, size=(5, 64))
    g = gen.bf16_bits(np.random.default_rng(14).normal(1, 0.1, size=64).astype(np.float32))
    a = oracle_lib.rmsnorm(y, g, 0.0)
    b = oracle_lib.rmsnorm(37.5 * y, g, 0.0)
    np.testing.assert_allclose(a, b, rtol=1e-13)
    # unit root mean square before gamma
    ones = gen.bf16_bits(np.ones(64, np.float32))
    u = oracle_lib.rmsnorm(y, ones, 0.0)
    np.testing.assert_allclose(np.sqrt(np.mean(u ** 2, axis=1)), 1.0, rtol=1e-13)


# --------------------------------------------------------------------------- MXFP4 weights

def test_e2m1_and_ue8m0_tables(oracle_lib):
    # the element and scale value tables of the OCP MX specification, every code
    d = _gold("mxfp4_decode.json")
    for code, val in enumerate(d["e2m1_values"]):
        got = oracle_lib.e2m1_to_f64(code)
        assert got == val and math.copysign(1.0, got) == math.copysign(1.0, val), code
    for e, val in d["ue8m0"].items():
        assert oracle_lib.ue8m0_to_f64(int(e)) == val, e
    assert math.isnan(oracle_lib.ue8m0_to_f64(255))


def test_mxfp4_nibble_decode_golden(oracle_lib):
    d = _gold("mxfp4_decode.json")
    K = d["K"]
    q = np.full((1, K // 2), int(d["default_byte"], 16), dtype=np.uint8)
    for pos, b in d["bytes"].items():
        q[0, int(pos)] = int(b, 16)
    e8 = np.array([d["scales_e8"]], dtype=np.uint8)
    w = oracle_lib.dequant_mxfp4(q, e8, 1, K)
    for col, val in d["expected"].items():
        got = w[0, int(col)]
        assert got == val and math.copysign(1.0, got) == math.copysign(1.0, val), col
    named = {int(c) for c in d["expected"]}
    others = [c for c in range(K) if c not in named and c // 2 not in {int(p) for p in d["bytes"]}]
    assert np.all(w[0, others] == 0.0)


def test_mxfp4_nan_scale_is_rejected(oracle_lib):
    q = np.zeros((1, 16), dtype=np.uint8)
    e8 = np.array([[255]], dtype=np.uint8)
    with pytest.raises(ValueError):
        oracle_lib.dequant_mxfp4(q, e8, 1, 32)
    x = gen.draw_x(3, 1, 32)
    e8_ok = np.full((32, 1), 127, dtype=np.uint8)
    with pytest.raises(ValueError):
        oracle_lib.expert_row(x[0], (np.zeros((32, 16), np.uint8), e8_ok), (np.zeros((32, 16), np.uint8), e8_ok),
                              (np.zeros((32, 16), np.uint8), np.full((32, 1), 255, np.uint8)), 32, 32, "mxfp4")


def _int4_twin(q, e8):
    """An int4 matrix holding the same weights as an MXFP4 matrix whose codes all have |2v| <= 7:
    nibble 8 + 2v, fp16 scale 2^(e - 128) (exact in fp16 for the exponents used here)."""
    two_v = {0: 0, 1: 1, 2: 2, 3: 3, 4: 4, 5: 6, 8: 0, 9: -1, 10: -2, 11: -3, 12: -4, 13: -6}
    lo, hi = q & 0xF, q >> 4
    lut = np.zeros(16, dtype=np.int64)
    for c, v in two_v.items():
        lut[c] = 8 + v
    q4 = (lut[lo] | (lut[hi] << 4)).astype(np.uint8)
    s = gen.f16_bits(np.ldexp(1.0, e8.astype(np.int64) - 128).astype(np.float32))
    return q4, s


def test_mxfp4_mlp_equals_its_int4_twin(oracle_lib):
    # Codes 0..5 and 8..13 (values up to 3 in size) are int4 values 2v at half the scale, so
    # both formats hold the same weights exactly and the two MLPs must agree to the last bit:
    # a swapped nibble, a misplaced scale group or a transposed matrix on the MXFP4 side fails.
    H, I = 64, 96
    r = gen.rng(11, 1)
    codes = np.array([0, 1, 2, 3, 4, 5, 8, 9, 10, 11, 12, 13], dtype=np.uint8)

    def mat(rows, K):
        lo = codes[r.integers(0, len(codes), size=(rows, K // 2))]
        hi = codes[r.integers(0, len(codes), size=(rows, K // 2))]
        return (lo | (hi << 4)).astype(np.uint8), r.integers(119, 123, size=(rows, K // 32)).astype(np.uint8)

    g, u, d = mat(I, H), mat(I, H), mat(H, I)
    x = gen.draw_x(5, 1, H)[0]
    o_fp4 = oracle_lib.expert_row(x, g, u, d, H, I, "mxfp4")
    o_int4 = oracle_lib.expert_row(x, _int4_twin(*g), _int4_twin(*u), _int4_twin(*d), H, I)
    assert np.array_equal(o_fp4, o_int4)
    # and the weights themselves
    assert np.array_equal(oracle_lib.dequant_mxfp4(*g, I, H), oracle_lib.dequant(*_int4_twin(*g), I, H))


def test_mxfp4_mlp_closed_form(oracle_lib):
    # every gate and up weight +1.0 * 2^(e-127), every down weight -6 * 2^(e-127): with S = sum x,
    # g = u = S * 2^(eg-127), h = silu(g) * u for every i, o[n] = -6 * 2^(ed-127) * I * h
    H, I = 64, 32
    x = gen.draw_x(7, 1, H)[0]
    S = float(np.sum(gen.bf16_to_f32(x).astype(np.float64)))
    one, m6 = 0x22, 0xFF  # both nibbles code 2 (+1.0); both nibbles code 15 (-6.0)
    eg, ed = 126, 129
    gq = np.full((I, H // 2), one, np.uint8)
    ge = np.full((I, H // 32), eg, np.uint8)
    dq = np.full((H, I // 2), m6, np.uint8)
    de = np.full((H, I // 32), ed, np.uint8)
    o = oracle_lib.expert_row(x, (gq, ge), (gq, ge), (dq, de), H, I, "mxfp4")
    gv = S * 2.0 ** (eg - 127)
    h = gv / (1.0 + math.exp(-gv)) * gv
    ref = -6.0 * 2.0 ** (ed - 127) * I * h
    assert np.allclose(o, ref, rtol=1e-12, atol=0)


def test_mxfp4_layer_routes_like_int4(oracle_lib):
    # the weight format changes the expert outputs, not the routing; with the routed experts in
    # MXFP4 and the shared expert in int4 the layer is the sum of its parts
    wl = gen.Workload("t", 3, 64, 32, 8, 2, I_sh=32, fmt=gen.FMT_MXFP4)
    inp = gen.draw_layer(wl)
    wl4 = gen.Workload("t", 3, 64, 32, 8, 2, I_sh=32)
    inp4 = gen.draw_layer(wl4)
    assert np.array_equal(inp.x, inp4.x) and inp.shared.fmt == "int4" and inp.experts.fmt == "mxfp4"
    out = oracle_lib.layer_forward(inp)
    out4 = oracle_lib.layer_forward(inp4)
    assert np.array_equal(out["ids"], out4["ids"]) and np.array_equal(out["w"], out4["w"])
    _, _, perm, inv = oracle_lib.dispatch(out["ids"], wl.E)
    rows = oracle_lib.expert_mlp(inp.x, inp.experts, out["ids"], perm)
    ysh = oracle_lib.shared_expert(inp.x, inp.shared)
    y = oracle_lib.combine(rows, inv, out["w"], ysh, inp.residual)
    assert np.allclose(out["y"], y, rtol=0, atol=1e-12)
    assert not np.allclose(out["y"], out4["y"])


def test_mxfp4_generator_ranges():
    m = gen.draw_mxfp4(0, gen.TAG_GATE, 2, 32, 256)
    assert m.fmt == "mxfp4" and m.s.dtype == np.uint8 and m.s.shape == (2, 32, 8)
    lo, hi = gen.MXFP4_EXP_RANGE
    assert m.s.min() >= lo and m.s.max() <= hi and len(np.unique(m.s)) == hi - lo + 1
    # the codes are the int4 set's nibbles: same stream
    assert np.array_equal(m.q, gen.draw_q4(0, gen.TAG_GATE, 2, 32, 256).q)


def test_mxfp4_dequant_by_numpy_table(oracle_lib):
    # unpack the codes with numpy bit operations and the OCP value table, scale by 2^(e-127)
    d = _gold("mxfp4_decode.json")
    table = np.array(d["e2m1_values"], dtype=np.float64)
    m = gen.draw_mxfp4(9, gen.TAG_GATE, 1, 32, 96)
    q, e8 = m.q[0], m.s[0]
    codes = np.empty((32, 96), dtype=np.int64)
    codes[:, 0::2], codes[:, 1::2] = q & 0xF, q >> 4
    ref = table[codes] * np.repeat(np.ldexp(1.0, e8.astype(np.int64) - 127), 32, axis=1)
    assert np.array_equal(oracle_lib.dequant_mxfp4(q, e8, 32, 96), ref)


def test_mxfp4_mlp_is_dense_restatement(oracle_lib):
    H, I = 64, 96
    ex = gen.draw_experts(3, 1, H, I, gen.FMT_MXFP4)
    x = gen.bf16_bits(gen.rng(4).normal(size=H))
    o = oracle_lib.expert_row(x, (ex.gate.q[0], ex.gate.s[0]), (ex.up.q[0], ex.up.s[0]),
                              (ex.down.q[0], ex.down.s[0]), H, I, "mxfp4")
    Wg = oracle_lib.dequant_mxfp4(ex.gate.q[0], ex.gate.s[0], I, H)
    Wu = oracle_lib.dequant_mxfp4(ex.up.q[0], ex.up.s[0], I, H)
    Wd = oracle_lib.dequant_mxfp4(ex.down.q[0], ex.down.s[0], H, I)
    xf = gen.bf16_to_f32(x).astype(np.float64)
    g, u = Wg @ xf, Wu @ xf
    ref = Wd @ (g / (1 + np.exp(-g)) * u)
    assert np.allclose(o, ref, rtol=1e-12, atol=1e-12)
