"""Planted mistakes in the oracle must be caught by its pins.

Each mutant is a copy of oracle/om_oracle.c with one plausible error
(a fused multiply-add in exact mode, a reversed or reordered sum, a skipped
padding product, a wrong group offset, a dropped term, a missing NaN
canonicalisation, a transposed operand), compiled on the CPU into a temporary
library. The golden pins and the brute-force model must reject every one.
"""
import ctypes
import json
import os
import subprocess

import numpy as np
import pytest

import oracle
from tests import ieee_ref

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(os.path.dirname(HERE), "oracle", "om_oracle.c")

MUTANTS = {
    "fma_in_exact": ("    float prod = a * b;                /* rounded to binary32 */\n"
                     "    return acc + prod;                 /* rounded to binary32 */",
                     "    return fmaf(a, b, acc);"),
    "unfused_in_fast": ("        return fmaf(a, b, acc);        /* one rounding: round(a*b + acc) */",
                        "        { float t = a * b; return acc + t; }"),
    "reversed_k": ("            for (int64_t p = 0; p < k; ++p) {\n                acc = add_term(acc, A[i * lda + p], B[p * ldb + j], mode);",
                   "            for (int64_t p = k - 1; p >= 0; --p) {\n                acc = add_term(acc, A[i * lda + p], B[p * ldb + j], mode);"),
    "dropped_last_term": ("            for (int64_t p = 0; p < k; ++p) {\n                acc = add_term(acc, A[i * lda + p], B[p * ldb + j], mode);",
                          "            for (int64_t p = 0; p + 1 < k; ++p) {\n                acc = add_term(acc, A[i * lda + p], B[p * ldb + j], mode);"),
    "transposed_b_index": ("acc = add_term(acc, A[i * lda + p], B[p * ldb + j], mode);",
                           "acc = add_term(acc, A[i * lda + p], B[j * ldb + p], mode);"),
    "no_nan_canonical": ("    if (isnan(acc)) {", "    if (0) {"),
    "start_minus_zero": ("            float acc = +0.0f;\n            for (int64_t p = 0; p < k; ++p) {",
                         "            float acc = -0.0f;\n            for (int64_t p = 0; p < k; ++p) {"),
    "conv_kx_before_ky": ("                        for (int64_t ky = 0; ky < KH; ++ky) {\n                            for (int64_t kx = 0; kx < KW; ++kx) {\n                                const int64_t iy = oy * sH - pT + ky * dH;\n                                const int64_t ix = ox * sW - pL + kx * dW;\n                                float v",
                          "                        for (int64_t kx = 0; kx < KW; ++kx) {\n                            for (int64_t ky = 0; ky < KH; ++ky) {\n                                const int64_t iy = oy * sH - pT + ky * dH;\n                                const int64_t ix = ox * sW - pL + kx * dW;\n                                float v"),
    "conv_skip_padding_taps": ("                                const float wt = w[((oc * cin_g + c) * KH + ky) * KW + kx];\n                                acc = add_term(acc, wt, v, mode);",
                               "                                const float wt = w[((oc * cin_g + c) * KH + ky) * KW + kx];\n                                if (iy >= 0 && iy < H && ix >= 0 && ix < W) acc = add_term(acc, wt, v, mode);"),
    "conv_wrong_group": ("v = x[((n * Cin + g * cin_g + c) * H + iy) * W + ix];",
                         "v = x[((n * Cin + c) * H + iy) * W + ix];"),
    "conv_pad_sign": ("                                const int64_t iy = oy * sH - pT + ky * dH;\n                                const int64_t ix = ox * sW - pL + kx * dW;\n                                float v",
                      "                                const int64_t iy = oy * sH + pT + ky * dH;\n                                const int64_t ix = ox * sW - pL + kx * dW;\n                                float v"),
    "out_dim_off_by_one": ("    return num / stride + 1;", "    return (num + 1) / stride + 1;"),
    "epilogue_relu_before_residual": (
        "        if (res) v = v + res[o];\n        if (activation == 1 && !(v > 0.0f) && !isnan(v)) v = +0.0f;",
        "        if (activation == 1 && !(v > 0.0f) && !isnan(v)) v = +0.0f;\n        if (res) v = v + res[o];"),
    "epilogue_bias_plus_residual_first": (
        "        if (bias) v = v + bias[(o / plane) % channels];\n        if (res) v = v + res[o];",
        "        if (bias && res) v = v + (bias[(o / plane) % channels] + res[o]);\n        else if (bias) v = v + bias[(o / plane) % channels];\n        else if (res) v = v + res[o];"),
    "epilogue_relu_drops_nan": ("!(v > 0.0f) && !isnan(v)", "!(v > 0.0f)"),
    "f64_mag_without_fabs": ("t = t + fabs(prod);", "t = t + prod;"),
    "f64_gemm_dropped_last_term": (
        "            for (int64_t p = 0; p < k; ++p) {\n                const double prod",
        "            for (int64_t p = 0; p + 1 < k; ++p) {\n                const double prod"),
    "f64_conv_wrong_group": ("v = x[((n * Cin + g * cin_g + c) * H + iy) * W + ix];\n                                }\n                                const double",
                             "v = x[((n * Cin + c) * H + iy) * W + ix];\n                                }\n                                const double"),
}


def _build(tmp_path, name, old, new):
    src = open(SRC).read()
    assert src.count(old) >= 1, name
    mutated = src.replace(old, new)
    c = tmp_path / f"{name}.c"
    so = tmp_path / f"{name}.so"
    c.write_text(mutated)
    subprocess.run(["gcc", *oracle.CFLAGS, str(c), "-o", str(so), "-lm"], check=True,
                   capture_output=True)
    L = ctypes.CDLL(str(so))
    i64, vp, ci = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int
    L.oracle_gemm_f32.argtypes = [i64, i64, i64, vp, i64, vp, i64, vp, i64, ci, ci]
    L.oracle_conv2d_f32.argtypes = [i64] * 16 + [vp, vp, vp, ci, ci]
    L.oracle_conv_out_dim.argtypes = [i64] * 6
    L.oracle_conv_out_dim.restype = i64
    L.oracle_epilogue_f32.argtypes = [i64, i64, i64, vp, vp, vp, ci]
    L.oracle_epilogue_f32.restype = None
    L.oracle_gemm_f64.argtypes = [i64, i64, i64, vp, i64, vp, i64, vp, vp, i64, ci]
    L.oracle_gemm_f64.restype = None
    L.oracle_conv2d_f64.argtypes = [i64] * 16 + [vp, vp, vp, vp, ci]
    L.oracle_conv2d_f64.restype = None
    return L


def _slack(a: np.ndarray) -> np.ndarray:
    """A copy of ``a`` at the start of a much larger zeroed buffer, so a
    mutant that indexes past the end reads zeros instead of foreign memory."""
    buf = np.zeros(a.size + 4096, np.float32)
    buf[:a.size] = a.reshape(-1)
    return buf


def _gemm(L, A, B, mode):
    m, k = A.shape
    n = B.shape[1]
    Ab, Bb = _slack(A), _slack(B)
    C = np.zeros(m * n + 4096, np.float32)
    L.oracle_gemm_f32(m, n, k, Ab.ctypes.data, k, Bb.ctypes.data, n, C.ctypes.data, n, mode, 1)
    return C[:m * n].view(np.uint32).reshape(m, n)


def _pins_pass(L) -> bool:
    g = json.load(open(os.path.join(HERE, "golden", "gemm_pins.json")))
    for mode, key in ((0, "exact_bits"), (1, "fast_bits")):
        for pin in g["pins"]:
            A = np.array(pin["A_bits"], np.uint32).view(np.float32)
            B = np.array(pin["B_bits"], np.uint32).view(np.float32)
            if _gemm(L, A, B, mode).tolist() != pin[key]:
                return False
        rng = np.random.default_rng(99 + mode)
        A = rng.standard_normal((3, 6)).astype(np.float32)
        B = rng.standard_normal((6, 2)).astype(np.float32)
        if _gemm(L, A, B, mode).tolist() != ieee_ref.gemm_bits(A, B, mode).tolist():
            return False
    c = json.load(open(os.path.join(HERE, "golden", "conv_pins.json")))
    for pin in c["pins"]:
        s = pin["shape"]
        x = _slack(np.array(pin["x_bits"], np.uint32).view(np.float32))
        w = _slack(np.array(pin["w_bits"], np.uint32).view(np.float32))
        oh = L.oracle_conv_out_dim(s["H"], s["KH"], s["stride"], s["pad"], s["pad"], s["dil"])
        ow = L.oracle_conv_out_dim(s["W"], s["KW"], s["stride"], s["pad"], s["pad"], s["dil"])
        if s["N"] * s["Cout"] * oh * ow != len(pin["exact_bits"]):
            return False
        y = np.zeros(len(pin["exact_bits"]) + 4096, np.float32)
        L.oracle_conv2d_f32(s["N"], s["Cin"], s["H"], s["W"], s["Cout"], s["G"], s["KH"], s["KW"],
                            s["stride"], s["stride"], s["pad"], s["pad"], s["pad"], s["pad"],
                            s["dil"], s["dil"], x.ctypes.data, w.ctypes.data, y.ctypes.data, 0, 1)
        if y[:len(pin["exact_bits"])].view(np.uint32).tolist() != pin["exact_bits"]:
            return False
    e = json.load(open(os.path.join(HERE, "golden", "epilogue_pins.json")))
    for pin in e["pins"]:
        y = np.array(pin["y"], np.float32)
        shape = pin.get("shape", [1, len(pin["y"])])
        channels = shape[1]
        plane = int(np.prod(shape[2:])) if len(shape) > 2 else 1
        bias = pin["bias"]
        if bias is not None and "shape" not in pin:
            bias = bias * channels
        b = None if bias is None else np.array(bias, np.float32)
        r = None if pin["res"] is None else np.array(pin["res"], np.float32)
        L.oracle_epilogue_f32(y.size, plane, channels, y.ctypes.data,
                              None if b is None else b.ctypes.data,
                              None if r is None else r.ctypes.data, pin["act"])
        if y.view(np.uint32).tolist() != pin["out_bits"]:
            return False
    if not _f64_pins_pass(L):
        return False
    for cs in c["out_dims"]["cases"]:
        if L.oracle_conv_out_dim(cs["size"], cs["k"], cs["stride"], cs["pad"], cs["pad"], cs["dil"]) != cs["out"]:
            return False
    return True


def _f64_pins_pass(L) -> bool:
    """The binary64 companions on small integers of both signs: exact sums."""
    rng = np.random.default_rng(5)
    A = rng.integers(-9, 10, (4, 7))
    B = rng.integers(-9, 10, (7, 3))
    Ab, Bb = _slack(A.astype(np.float32)), _slack(B.astype(np.float32))
    ref = np.zeros(12 + 4096)
    mag = np.zeros(12 + 4096)
    L.oracle_gemm_f64(4, 3, 7, Ab.ctypes.data, 7, Bb.ctypes.data, 3, ref.ctypes.data,
                      mag.ctypes.data, 3, 1)
    if not (np.array_equal(ref[:12].reshape(4, 3), A @ B)
            and np.array_equal(mag[:12].reshape(4, 3), np.abs(A) @ np.abs(B))):
        return False
    # grouped convolution, 2 images, 4 -> 4 channels in 2 groups, 3x3, pad 1
    x = rng.integers(-4, 5, (2, 4, 5, 5))
    w = rng.integers(-4, 5, (4, 2, 3, 3))
    xp = np.zeros((2, 4, 7, 7), np.int64)
    xp[:, :, 1:6, 1:6] = x
    want = np.zeros((2, 4, 5, 5), np.int64)
    want_mag = np.zeros((2, 4, 5, 5), np.int64)
    for oc in range(4):
        g = oc // 2
        for c in range(2):
            for ky in range(3):
                for kx in range(3):
                    win = xp[:, g * 2 + c, ky:ky + 5, kx:kx + 5]
                    want[:, oc] += w[oc, c, ky, kx] * win
                    want_mag[:, oc] += abs(w[oc, c, ky, kx]) * np.abs(win)
    xb, wb = _slack(x.astype(np.float32)), _slack(w.astype(np.float32))
    ref = np.zeros(200 + 4096)
    mag = np.zeros(200 + 4096)
    L.oracle_conv2d_f64(2, 4, 5, 5, 4, 2, 3, 3, 1, 1, 1, 1, 1, 1, 1, 1, xb.ctypes.data,
                        wb.ctypes.data, ref.ctypes.data, mag.ctypes.data, 1)
    return (np.array_equal(ref[:200].reshape(want.shape), want)
            and np.array_equal(mag[:200].reshape(want.shape), want_mag))


def test_unmutated_copy_passes(tmp_path):
    L = _build(tmp_path, "identity", "int oracle_abi_version", "int oracle_abi_version")
    assert _pins_pass(L)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(tmp_path, name):
    old, new = MUTANTS[name]
    L = _build(tmp_path, name, old, new)
    assert not _pins_pass(L), f"pins did not catch the planted mistake {name}"
