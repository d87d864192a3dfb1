"""Host check of the e2m1 decode tables in csrc/fp4.cuh against the oracle's e2m1 values.

The kernels expand MXFP4 codes with byte permutes (prmt: byte n of the result is byte
selector_n of the 8-byte pair {hi word, lo word}) over constant tables.  This test reads the
tables from the source, emulates the permutes on the host, and checks every code in every
position against the oracle's decode: the signed bytes 2v of the GEMV (split into even and odd
columns) and the fp16 2v of the tensor arm (in its K order c0 c4 c1 c5 c2 c6 c3 c7)."""
import os
import re

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
FP4 = os.path.join(HERE, "..", "mixture_experts_layer_09_gb300", "csrc", "fp4.cuh")
M32 = 0xFFFFFFFF


def _tables():
    src = open(FP4).read()
    return {n: int(v, 16) for n, v in re.findall(r"(kE2m1\w+) = (0x[0-9A-Fa-f]+)u", src)}


def _perm(x, y, s):
    b = (y << 32) | x
    out = 0
    for n in range(4):
        sel = (s >> (4 * n)) & 0xF
        assert sel < 8, "the kernels keep every selector nibble below 8"
        out |= ((b >> (8 * sel)) & 0xFF) << (8 * n)
    return out


def _x4_i8(t, c):
    sel = c & 0x7777
    pos = _perm(t["kE2m1PosLo"], t["kE2m1PosHi"], sel)
    neg = _perm(t["kE2m1NegLo"], t["kE2m1NegHi"], sel)
    msk = _perm(0, M32, (c >> 1) & 0x4444)
    return ((pos & ~msk) | (neg & msk)) & M32


def _x8_i8(t, w):
    a, b = _x4_i8(t, w & M32), _x4_i8(t, (w >> 16) & M32)
    return _perm(a, b, 0x6420), _perm(a, b, 0x7531)


def _x8_f16(t, w):
    lo, hi = t["kE2m1HalfLo"], t["kE2m1HalfHi"]
    hx = _perm(lo, hi, ((w << 4) & 0x70) | ((w >> 4) & 0x7000)) | ((w << 12) & 0x80008000)
    hy = _perm(lo, hi, (w & 0x70) | ((w >> 8) & 0x7000)) | ((w << 8) & 0x80008000)
    hz = _perm(lo, hi, ((w >> 4) & 0x70) | ((w >> 12) & 0x7000)) | ((w << 4) & 0x80008000)
    hw = _perm(lo, hi, ((w >> 8) & 0x70) | ((w >> 16) & 0x7000)) | (w & 0x80008000)
    return [h & M32 for h in (hx, hy, hz, hw)]


def _words():
    g = np.random.default_rng(17)
    ws = [int(v) for v in g.integers(0, 1 << 32, size=3000, dtype=np.uint64)]
    # every code in every column position
    for code in range(16):
        for pos in range(8):
            ws.append((0x0 << 0) | (code << (4 * pos)))
            ws.append(0x88888888 ^ ((code ^ 0x8) << (4 * pos)))
    return ws + [0, M32, 0x76543210, 0xFEDCBA98]


def test_gemv_signed_bytes(oracle_lib):
    t = _tables()
    val = [oracle_lib.e2m1_to_f64(c) for c in range(16)]
    sb = lambda b: b - 256 if b >= 128 else b  # noqa: E731
    for w in _words():
        cols = [(w >> (4 * j)) & 0xF for j in range(8)]
        lo, hi = _x8_i8(t, w)
        got = [None] * 8
        for i in range(4):
            got[2 * i] = sb((lo >> (8 * i)) & 0xFF)
            got[2 * i + 1] = sb((hi >> (8 * i)) & 0xFF)
        assert got == [2 * val[c] for c in cols], hex(w)


def test_tensor_arm_fp16_pairs(oracle_lib):
    t = _tables()
    val = [oracle_lib.e2m1_to_f64(c) for c in range(16)]
    order = [0, 4, 1, 5, 2, 6, 3, 7]
    for w in _words():
        cols = [(w >> (4 * j)) & 0xF for j in range(8)]
        halves = []
        for h in _x8_f16(t, w):
            halves += [h & 0xFFFF, h >> 16]
        f = np.array(halves, dtype=np.uint16).view(np.float16).astype(np.float64)
        want = np.array([2 * val[cols[c]] for c in order])
        assert np.array_equal(f, want) and np.array_equal(np.signbit(f), np.signbit(want)), hex(w)
