"""Seeded synthetic inputs for the routed MoE layer.

This module only draws random numbers and encodes them in the storage formats
the layer consumes: bf16 and fp16 bit patterns, and int4 nibbles packed two per
byte.  It holds none of the layer's arithmetic (no dot product, routing,
dispatch, MLP or combine), so both sides of a parity test -- the fp64 oracle
and the CUDA path -- can draw the same inputs from here without sharing code.

Distributions follow the workloads the layer is measured on:

* hidden rows x and residual r: bf16 ~ N(0, 1)
* router rows W_r and the shared-expert gate vector g: bf16 ~ N(0, 0.02)
* expert weights: nibbles uniform in 0..15 (value = nibble - 8, the offset-binary
  int4 of colibri PR #418, "Correctness"), packed two per byte along K with the
  even column in the low nibble; one fp16 scale per 32 K-columns drawn as
  |N(0, 0.01)| + 1e-3 (the grouped scales of colibri PR #418, "Grouped scales in
  the Vulkan kernels", at group size 32)
* MXFP4 expert weights (the fmt=7 format of colibri PR #418's Kimi K3 tier): the same
  uniform nibbles read as e2m1 codes, one ue8m0 exponent per 32 K-columns drawn uniform in
  119..122 (scales 2^-8 .. 2^-5, weights of about the int4 sets' magnitude)
* given router logits (router-only sweeps): bf16 of N(0, 1) * 2

Every tensor draws from its own PCG64 stream keyed by (seed, tag, ...), and
hidden rows / logit rows draw one stream per row, keyed by (seed, tag, row,
attempt), so that a test can redraw a single row without disturbing the rest.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional

import numpy as np

# stream tags
TAG_X, TAG_R, TAG_WR, TAG_G, TAG_LOGITS = 1, 2, 3, 4, 5
TAG_GATE, TAG_UP, TAG_DOWN = 10, 11, 12
TAG_SH_GATE, TAG_SH_UP, TAG_SH_DOWN = 20, 21, 22
SCALE_GROUP = 32


def rng(seed: int, *tags: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([int(seed), *map(int, tags)])))


def bf16_bits(a) -> np.ndarray:
    """Round float32 values to bf16 (round to nearest, ties to even); return the bit patterns."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


def bf16_to_f32(bits) -> np.ndarray:
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


def f16_bits(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float32).astype(np.float16).view(np.uint16)


def f16_to_f32(bits) -> np.ndarray:
    return np.ascontiguousarray(bits, dtype=np.uint16).view(np.float16).astype(np.float32)


# ----------------------------------------------------------------------------- weights

FMT_INT4, FMT_MXFP4 = "int4", "mxfp4"
MXFP4_EXP_RANGE = (119, 122)  # ue8m0 exponents drawn uniform in this closed range


@dataclass
class Q4:
    """One 4-bit matrix per expert: q [n_mat][rows][K/2] uint8 (two codes per byte, the even
    column in the low nibble) and s [n_mat][rows][K/32]: fp16 bits for int4, ue8m0 exponent
    bytes for mxfp4."""
    q: np.ndarray
    s: np.ndarray
    fmt: str = FMT_INT4

    @property
    def rows(self) -> int:
        return self.q.shape[-2]

    @property
    def K(self) -> int:
        return self.q.shape[-1] * 2


def draw_q4(seed: int, tag: int, n_mat: int, rows: int, K: int) -> Q4:
    if K % SCALE_GROUP:
        raise ValueError("K must be a multiple of 32")
    g = rng(seed, tag)
    nbytes = n_mat * rows * (K // 2)
    # raw 64-bit outputs of the stream: every bit uniform, so every nibble is uniform in 0..15
    raw = g.bit_generator.random_raw((nbytes + 7) // 8).view(np.uint8)
    q = raw[:nbytes].reshape(n_mat, rows, K // 2).copy()
    s = f16_bits(np.abs(g.normal(0.0, 0.01, size=(n_mat, rows, K // SCALE_GROUP))) + 1e-3)
    return Q4(q, s)


def draw_mxfp4(seed: int, tag: int, n_mat: int, rows: int, K: int) -> Q4:
    """MXFP4 matrix: uniform e2m1 codes (the same stream as draw_q4's nibbles) and ue8m0
    exponents uniform in MXFP4_EXP_RANGE."""
    if K % SCALE_GROUP:
        raise ValueError("K must be a multiple of 32")
    g = rng(seed, tag)
    nbytes = n_mat * rows * (K // 2)
    raw = g.bit_generator.random_raw((nbytes + 7) // 8).view(np.uint8)
    q = raw[:nbytes].reshape(n_mat, rows, K // 2).copy()
    lo, hi = MXFP4_EXP_RANGE
    e8 = g.integers(lo, hi + 1, size=(n_mat, rows, K // SCALE_GROUP), dtype=np.uint8)
    return Q4(q, e8, FMT_MXFP4)


def draw_mat(fmt: str, seed: int, tag: int, n_mat: int, rows: int, K: int) -> Q4:
    if fmt == FMT_INT4:
        return draw_q4(seed, tag, n_mat, rows, K)
    if fmt == FMT_MXFP4:
        return draw_mxfp4(seed, tag, n_mat, rows, K)
    raise ValueError(f"unknown weight format {fmt!r}")


@dataclass
class Experts:
    E: int
    H: int
    I: int
    gate: Q4   # [E][I][H/2]
    up: Q4     # [E][I][H/2]
    down: Q4   # [E][H][I/2]

    @property
    def fmt(self) -> str:
        return self.gate.fmt


@dataclass
class Shared:
    I_sh: int
    gate: Q4   # [1][I_sh][H/2]
    up: Q4
    down: Q4   # [1][H][I_sh/2]
    g: Optional[np.ndarray]  # bf16 bits [H], or None for an ungated shared expert

    @property
    def fmt(self) -> str:
        return self.gate.fmt


def draw_experts(seed: int, E: int, H: int, I: int, fmt: str = FMT_INT4) -> Experts:
    return Experts(E, H, I,
                   draw_mat(fmt, seed, TAG_GATE, E, I, H),
                   draw_mat(fmt, seed, TAG_UP, E, I, H),
                   draw_mat(fmt, seed, TAG_DOWN, E, H, I))


def draw_shared(seed: int, H: int, I_sh: int, gated: bool = True, fmt: str = FMT_INT4) -> Shared:
    g = bf16_bits(rng(seed, TAG_G).normal(0.0, 0.02, size=H)) if gated else None
    return Shared(I_sh,
                  draw_mat(fmt, seed, TAG_SH_GATE, 1, I_sh, H),
                  draw_mat(fmt, seed, TAG_SH_UP, 1, I_sh, H),
                  draw_mat(fmt, seed, TAG_SH_DOWN, 1, H, I_sh),
                  g)


def draw_router(seed: int, E: int, H: int) -> np.ndarray:
    return bf16_bits(rng(seed, TAG_WR).normal(0.0, 0.02, size=(E, H)))


# ----------------------------------------------------------------------------- activations

def draw_x_row(seed: int, t: int, H: int, attempt: int = 0) -> np.ndarray:
    return bf16_bits(rng(seed, TAG_X, t, attempt).normal(0.0, 1.0, size=H))


def draw_x(seed: int, T: int, H: int, attempts: Optional[dict] = None) -> np.ndarray:
    """Hidden rows bf16 [T, H]; ``attempts`` maps a row to the redraw index it uses."""
    attempts = attempts or {}
    out = np.empty((T, H), dtype=np.uint16)
    for t in range(T):
        out[t] = draw_x_row(seed, t, H, attempts.get(t, 0))
    return out


def draw_residual(seed: int, T: int, H: int) -> np.ndarray:
    return bf16_bits(rng(seed, TAG_R).normal(0.0, 1.0, size=(T, H)))


def draw_logit_row(seed: int, t: int, E: int, attempt: int = 0) -> np.ndarray:
    return bf16_bits(rng(seed, TAG_LOGITS, t, attempt).normal(0.0, 1.0, size=E) * 2.0)


def draw_logits(seed: int, T: int, E: int, attempts: Optional[dict] = None) -> np.ndarray:
    attempts = attempts or {}
    out = np.empty((T, E), dtype=np.uint16)
    for t in range(T):
        out[t] = draw_logit_row(seed, t, E, attempts.get(t, 0))
    return out


def set_bias_channel(x: np.ndarray, W_r: np.ndarray, bias: np.ndarray) -> None:
    """Make column 0 of every hidden row a constant 1.0 and column 0 of router row e the value
    ``bias[e]`` (both stored as bf16), so that expert e's logit carries an extra ``bias[e]``.
    This is how the skewed-popularity workload is built; the biases themselves are an input."""
    x[:, 0] = bf16_bits(np.float32(1.0))
    W_r[:, 0] = bf16_bits(np.asarray(bias, dtype=np.float32))


def zipf_bias(E: int, s: float, H: int) -> np.ndarray:
    """Router bias for a Zipf(s)-like expert popularity: expert e gets -s * sigma * ln(e + 1),
    sigma = 0.02 * sqrt(H) the spread of a router logit (router rows ~N(0, 0.02), x ~N(0, 1)),
    expert 0 the most popular.  At H=256, E=8, k=2 the slot shares come out near Zipf(1.1)'s
    (0.38 0.23 0.15 0.08 0.07 0.04 0.03 0.03 against 0.40 0.19 0.12 0.09 0.07 0.06 0.05 0.04)."""
    sigma = 0.02 * np.sqrt(H)
    return (-s * sigma * np.log(np.arange(E, dtype=np.float64) + 1.0)).astype(np.float32)


ONE_BF16 = 0x3F80  # bf16 bits of 1.0, the bias channel's hidden value


# ----------------------------------------------------------------------------- workloads

@dataclass
class Workload:
    name: str
    T: int
    H: int
    I: int
    E: int
    k: int
    I_sh: int = 0
    zipf: float = 0.0  # > 0: skewed popularity through the bias channel (set_bias_channel)
    gated_shared: bool = True
    residual: bool = True
    seed: int = 0
    fmt: str = FMT_INT4     # routed experts' weight format
    sh_fmt: str = FMT_INT4  # shared expert's weight format
    notes: str = ""
    extra: dict = field(default_factory=dict)


WORKLOADS = {
    # tiny layer: T=4, H=256, I=128, E=8, k=2, no shared expert
    "tiny": Workload("tiny", 4, 256, 128, 8, 2),
    # Qwen3-30B-A3B-shaped decode layer
    "qwen3_30b_decode_t1": Workload("qwen3_30b_decode_t1", 1, 2048, 768, 128, 8),
    "qwen3_30b_decode_t4": Workload("qwen3_30b_decode_t4", 4, 2048, 768, 128, 8),
    "qwen3_30b_decode_t16": Workload("qwen3_30b_decode_t16", 16, 2048, 768, 128, 8),
    # GLM-class large-expert decode layer, K-expert 6144 -> 2048 -> 6144
    "glm_decode_k8_t1": Workload("glm_decode_k8_t1", 1, 6144, 2048, 256, 8),
    "glm_decode_k8_t8": Workload("glm_decode_k8_t8", 8, 6144, 2048, 256, 8),
    "glm_decode_k32_t1": Workload("glm_decode_k32_t1", 1, 6144, 2048, 256, 32),
    "glm_decode_k32_t8": Workload("glm_decode_k32_t8", 8, 6144, 2048, 256, 32),
    # Qwen1.5-MoE-A2.7B-shaped prefill layer with a sigmoid-gated shared expert
    "qwen15_prefill_t512": Workload("qwen15_prefill_t512", 512, 2048, 1408, 60, 4, I_sh=5632),
    "qwen15_prefill_t4096": Workload("qwen15_prefill_t4096", 4096, 2048, 1408, 60, 4, I_sh=5632),
    # tiny-layer shape at T=8192 with skewed (Zipf-like) expert popularity
    "tiny_zipf_t8192": Workload("tiny_zipf_t8192", 8192, 256, 128, 8, 2, zipf=1.1),
    # MXFP4 routed experts (the int4 shared expert kept, as in colibri PR #418's Kimi K3 tier)
    "qwen3_30b_decode_t16_mxfp4": Workload("qwen3_30b_decode_t16_mxfp4", 16, 2048, 768, 128, 8,
                                           fmt=FMT_MXFP4),
    "qwen15_prefill_t4096_mxfp4": Workload("qwen15_prefill_t4096_mxfp4", 4096, 2048, 1408, 60, 4,
                                           I_sh=5632, fmt=FMT_MXFP4),
}


@dataclass
class LayerInputs:
    wl: Workload
    x: np.ndarray                 # bf16 bits [T, H]
    residual: Optional[np.ndarray]
    W_r: np.ndarray               # bf16 bits [E, H]
    experts: Experts
    shared: Optional[Shared]


def draw_layer(wl: Workload, x_attempts: Optional[dict] = None) -> LayerInputs:
    s = wl.seed
    ex = draw_experts(s, wl.E, wl.H, wl.I, wl.fmt)
    sh = draw_shared(s, wl.H, wl.I_sh, wl.gated_shared, wl.sh_fmt) if wl.I_sh else None
    x = draw_x(s, wl.T, wl.H, x_attempts)
    W_r = draw_router(s, wl.E, wl.H)
    if wl.zipf > 0:
        set_bias_channel(x, W_r, zipf_bias(wl.E, wl.zipf, wl.H))
    return LayerInputs(wl, x, draw_residual(s + 1, wl.T, wl.H) if wl.residual else None, W_r, ex, sh)
