"""Seeded synthetic inputs for the fp32 matrix product and NCHW convolution.

This module only draws numbers: it holds none of the product or convolution
arithmetic, so the CUDA path and the CPU oracle can both take their inputs
from it without sharing any of the computation they are compared on.

Generator: SplitMix64 used as a counter-based stream. Element ``i`` of stream
``(seed, stream)`` is ``mix64(seed * 2**32 + stream * 2**48 + (i + 1) * GOLDEN)``
(all arithmetic modulo 2**64), with ``mix64`` the SplitMix64 finaliser
(Steele, Lea and Flood, "Fast splittable pseudorandom number generators",
OOPSLA 2014). Uniform floats take the top 24 bits; normals use Box-Muller in
float64 on two uniforms, then round once to float32.

Workload recipes (shapes, distributions and the special cells) follow the
five benchmark configurations of this library's documentation: a small
strided product with IEEE special cells, the 4096-cube product, an
LLM-prefill-shaped product and its ragged variant, the ResNet-50 stage-1
3x3 and 1x1 convolutions, and a grouped, strided, dilated convolution with
non-finite weights.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
BASE_SEED = 0x0DDC0FFEE


def _mix64(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def raw_u64(seed: int, stream: int, count: int, offset: int = 0) -> np.ndarray:
    """``count`` 64-bit words of stream ``(seed, stream)`` starting at ``offset``."""
    with np.errstate(over="ignore"):
        base = np.uint64((seed * (1 << 32) + stream * (1 << 48)) & 0xFFFFFFFFFFFFFFFF)
        idx = np.arange(offset + 1, offset + count + 1, dtype=np.uint64)
        return _mix64(base + idx * GOLDEN)


def uniform(seed: int, stream: int, shape, lo: float, hi: float) -> np.ndarray:
    """float32 values ``lo + (hi - lo) * u`` with ``u = top24 / 2**24`` in [0, 1)."""
    n = int(np.prod(shape)) if len(shape) else 1
    u = (raw_u64(seed, stream, n) >> np.uint64(40)).astype(np.float64) / float(1 << 24)
    return (lo + (hi - lo) * u).astype(np.float32).reshape(shape)


def normal(seed: int, stream: int, shape, mean: float, std: float) -> np.ndarray:
    """float32 draws of N(mean, std**2) (``std`` is the standard deviation)."""
    n = int(np.prod(shape)) if len(shape) else 1
    m = (n + 1) // 2
    w = raw_u64(seed, stream, 2 * m)
    u1 = ((w[0::2] >> np.uint64(11)).astype(np.float64) + 1.0) / float(1 << 53)  # (0, 1]
    u2 = (w[1::2] >> np.uint64(11)).astype(np.float64) / float(1 << 53)          # [0, 1)
    r = np.sqrt(-2.0 * np.log(u1))
    z = np.empty(2 * m, dtype=np.float64)
    z[0::2] = r * np.cos(2.0 * math.pi * u2)
    z[1::2] = r * np.sin(2.0 * math.pi * u2)
    return (mean + std * z[:n]).astype(np.float32).reshape(shape)


def choose_distinct(seed: int, stream: int, population: int, count: int) -> np.ndarray:
    """``count`` distinct indices in ``[0, population)``, seeded (rejection of repeats)."""
    if count > population:
        raise ValueError("count exceeds population")
    out: list[int] = []
    seen: set[int] = set()
    offset = 0
    while len(out) < count:
        words = raw_u64(seed, stream, 4 * count + 8, offset)
        offset += len(words)
        for wv in words:
            v = int(wv % np.uint64(population))
            if v not in seen:
                seen.add(v)
                out.append(v)
                if len(out) == count:
                    break
    return np.array(out, dtype=np.int64)


def bits_to_f32(bits) -> np.ndarray:
    return np.array(bits, dtype=np.uint32).view(np.float32)


# IEEE special values planted in the small strided product: quiet NaN,
# +inf, -inf, a subnormal, negative zero, then the cycle again.
SPECIAL_CELL_BITS = [0x7FC00000, 0x7F800000, 0xFF800000, None, 0x80000000,
                     0x7FC00000, 0x7F800000, None]
SUBNORMAL_1EM40 = np.float32(1e-40)


def special_cell_values() -> np.ndarray:
    vals = []
    for b in SPECIAL_CELL_BITS:
        vals.append(SUBNORMAL_1EM40 if b is None else bits_to_f32([b])[0])
    return np.array(vals, dtype=np.float32)


@dataclass
class GemmCase:
    """A row-major product problem laid out in padded buffers.

    ``A`` is ``m x lda`` (columns ``k..lda-1`` are padding), ``B`` is
    ``k x ldb`` and ``C`` is ``m x ldc``; the padding holds sentinels
    (NaN in the operands, a recognisable pattern in ``C``) so reads or
    writes outside the used region show up in the result.
    """
    name: str
    m: int
    n: int
    k: int
    lda: int
    ldb: int
    ldc: int
    A: np.ndarray  # shape (max(m,1), lda) float32
    B: np.ndarray  # shape (max(k,1), ldb)
    C_init: np.ndarray  # shape (max(m,1), ldc), sentinel-filled
    special: dict = field(default_factory=dict)


C_SENTINEL_BITS = 0x7FBADBAD  # a signalling-NaN pattern no kernel produces


def _padded(rows: int, ld: int, used_cols: int, body: np.ndarray, pad_bits: int) -> np.ndarray:
    buf = np.empty((max(rows, 1), max(ld, 1)), dtype=np.float32)
    buf.view(np.uint32)[:] = np.uint32(pad_bits)
    if rows and used_cols:
        buf[:rows, :used_cols] = body
    return buf


def make_gemm(name: str, m: int, n: int, k: int, lda: int | None = None,
              ldb: int | None = None, ldc: int | None = None, seed: int = 0,
              dist_a=("uniform", -1.0, 1.0), dist_b=("uniform", -1.0, 1.0),
              special_cells: int = 0) -> GemmCase:
    lda = k if lda is None else lda
    ldb = n if ldb is None else ldb
    ldc = n if ldc is None else ldc
    s = BASE_SEED + seed

    def draw(stream, shape, dist):
        kind, p, q = dist
        if kind == "uniform":
            return uniform(s, stream, shape, p, q)
        if kind == "normal":
            return normal(s, stream, shape, p, q)
        if kind == "int":
            r = raw_u64(s, stream, int(np.prod(shape)))
            return (np.int64(p) + (r % np.uint64(q - p + 1)).astype(np.int64)).astype(np.float32).reshape(shape)
        raise ValueError(kind)

    a = draw(1, (m, k), dist_a) if m and k else np.zeros((m, k), np.float32)
    b = draw(2, (k, n), dist_b) if k and n else np.zeros((k, n), np.float32)
    special = {}
    if special_cells and m and n and k:
        vals = special_cell_values()[:special_cells]
        na = special_cells // 2
        ia = choose_distinct(s, 3, m * k, na)
        ib = choose_distinct(s, 4, k * n, special_cells - na)
        a.reshape(-1)[ia] = vals[:na]
        b.reshape(-1)[ib] = vals[na:]
        special = {"A_cells": ia.tolist(), "B_cells": ib.tolist()}
    A = _padded(m, lda, k, a, 0x7FC00000)
    B = _padded(k, ldb, n, b, 0x7FC00000)
    C = _padded(m, ldc, 0, np.zeros((0, 0), np.float32), C_SENTINEL_BITS)
    return GemmCase(name, m, n, k, lda, ldb, ldc, A, B, C, special)


@dataclass
class ConvCase:
    name: str
    N: int
    Cin: int
    H: int
    W: int
    Cout: int
    G: int
    KH: int
    KW: int
    stride: int
    pad: int
    dil: int
    x: np.ndarray  # (N, Cin, H, W) float32
    w: np.ndarray  # (Cout, Cin/G, KH, KW) float32
    special: dict = field(default_factory=dict)


def make_conv(name: str, N: int, Cin: int, H: int, W: int, Cout: int, G: int,
              KH: int, KW: int, stride: int, pad: int, dil: int, seed: int = 0,
              dist_x=("uniform", 0.0, 1.0), dist_w=("normal", 0.0, 0.1),
              nonfinite_weights: int = 0) -> ConvCase:
    s = BASE_SEED + seed
    cg = Cin // G if G else 0

    def draw(stream, shape, dist):
        kind, p, q = dist
        if int(np.prod(shape)) == 0:
            return np.zeros(shape, np.float32)
        if kind == "uniform":
            return uniform(s, stream, shape, p, q)
        if kind == "normal":
            return normal(s, stream, shape, p, q)
        if kind == "int":
            r = raw_u64(s, stream, int(np.prod(shape)))
            return (np.int64(p) + (r % np.uint64(q - p + 1)).astype(np.int64)).astype(np.float32).reshape(shape)
        raise ValueError(kind)

    x = draw(1, (N, Cin, H, W), dist_x)
    w = draw(2, (Cout, cg, KH, KW), dist_w)
    special = {}
    if nonfinite_weights and w.size:
        idx = choose_distinct(s, 3, w.size, nonfinite_weights)
        bits = np.where(np.arange(len(idx)) % 2 == 0, 0x7F800000, 0x7FC00000).astype(np.uint32)
        if len(idx) > 1:
            bits[1] = 0xFFC00001  # a NaN with sign and payload set
        w.reshape(-1).view(np.uint32)[idx] = bits
        special = {"w_cells": idx.tolist()}
    return ConvCase(name, N, Cin, H, W, Cout, G, KH, KW, stride, pad, dil, x, w, special)


# The five benchmark workloads (sizes, distributions, seeds).
def workload_gemm_small_strided(with_k0: bool = False) -> GemmCase:
    if with_k0:
        return make_gemm("gemm_67x53_k0", 67, 53, 0, lda=3, ldb=58, ldc=54, seed=0)
    return make_gemm("gemm_67x53x300_strided", 67, 53, 300, lda=303, ldb=58, ldc=54,
                     seed=0, special_cells=8)


def workload_gemm_4096() -> GemmCase:
    return make_gemm("gemm_4096^3", 4096, 4096, 4096, seed=1,
                     dist_a=("normal", 0.0, 1.0), dist_b=("normal", 0.0, 1.0))


def workload_gemm_prefill(ragged: bool = False) -> GemmCase:
    if ragged:
        return make_gemm("gemm_prefill_509x11005x4096", 509, 11005, 4096, lda=4096,
                         ldb=11005, ldc=11005, seed=3,
                         dist_a=("normal", 0.0, 1.0), dist_b=("normal", 0.0, 0.02))
    return make_gemm("gemm_prefill_512x11008x4096", 512, 11008, 4096, seed=2,
                     dist_a=("normal", 0.0, 1.0), dist_b=("normal", 0.0, 0.02))


def workload_conv3x3() -> ConvCase:
    return make_conv("conv3x3_n32_c64_56", 32, 64, 56, 56, 64, 1, 3, 3, 1, 1, 1, seed=4,
                     dist_x=("uniform", 0.0, 1.0), dist_w=("normal", 0.0, math.sqrt(2.0 / 576)))


def workload_conv1x1() -> ConvCase:
    return make_conv("conv1x1_n32_c256to64_56", 32, 256, 56, 56, 64, 1, 1, 1, 1, 0, 1, seed=5,
                     dist_x=("uniform", 0.0, 1.0), dist_w=("normal", 0.0, math.sqrt(2.0 / 256)))


def workload_conv_grouped() -> ConvCase:
    return make_conv("conv_g32_s2_d2_n16_c256_28", 16, 256, 28, 28, 256, 32, 3, 3, 2, 1, 2, seed=6,
                     dist_x=("uniform", -1.0, 1.0), dist_w=("normal", 0.0, 0.1),
                     nonfinite_weights=18)


# Widened workloads (not among the five above): a depthwise layer of
# MobileNet-like shape and a one-token product with the prefill weights.
def workload_conv_depthwise() -> ConvCase:
    return make_conv("conv_dw3x3_n32_c256_56", 32, 256, 56, 56, 256, 256, 3, 3, 1, 1, 1, seed=7,
                     dist_x=("uniform", 0.0, 1.0), dist_w=("normal", 0.0, math.sqrt(2.0 / 9)))


def workload_gemm_decode() -> GemmCase:
    return make_gemm("gemm_decode_1x11008x4096", 1, 11008, 4096, seed=8,
                     dist_a=("normal", 0.0, 1.0), dist_b=("normal", 0.0, 0.02))


def workload_conv_late3x3() -> ConvCase:
    """A late ResNet-50 layer at batch 1: 512 -> 512 channels, 3x3, 7x7 (49 output pixels)."""
    return make_conv("conv_late3x3_n1_c512_7", 1, 512, 7, 7, 512, 1, 3, 3, 1, 1, 1, seed=10,
                     dist_x=("uniform", 0.0, 1.0), dist_w=("normal", 0.0, math.sqrt(2.0 / 4608)))
