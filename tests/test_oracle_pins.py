"""Pins for the CPU oracle, against facts fixed outside the oracle itself.

Each test ties the oracle to something it does not compute: hand-derived
closed forms from the pages' rules (tests/golden), an independent exact
rational model of binary32 arithmetic (brute force on tiny inputs), integer
arithmetic, a textbook correlation routine, an explicit im2col built with
numpy, and the accuracy bound of sequential summation.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
from implicit_gemm_convolution_gb300 import synth
from tests import ieee_ref

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
U = 2.0 ** -24


def bits(a):
    return np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)


def test_selfcheck_and_version():
    L = oracle.lib()
    assert L.oracle_selfcheck() == 0
    assert L.oracle_abi_version() == 1


# --- the rational model itself is pinned to numpy's binary32 rounding ------
def test_ieee_ref_rounding_matches_float32_conversion():
    rng = np.random.default_rng(7)
    vals = np.concatenate([rng.standard_normal(300) * 10.0 ** rng.integers(-45, 39, 300),
                           [1e-46, 3e-45, 1.5e-45, 3.4028235e38, 3.4028236e38, 1e39]])
    from fractions import Fraction
    for v in vals:
        with np.errstate(over="ignore"):
            want = float(np.float32(v))
        got = ieee_ref.round_f32(Fraction(float(v)))
        assert got == want or (got == 0 and want == 0), (v, got, want)


@pytest.mark.parametrize("mode", [oracle.EXACT, oracle.FAST])
def test_golden_gemm_pins(mode):
    d = json.load(open(os.path.join(GOLDEN, "gemm_pins.json")))
    key = "exact_bits" if mode == oracle.EXACT else "fast_bits"
    for pin in d["pins"]:
        A = np.array(pin["A_bits"], np.uint32).view(np.float32)
        B = np.array(pin["B_bits"], np.uint32).view(np.float32)
        C = oracle.gemm(A, B, mode)
        assert bits(C).tolist() == pin[key], pin["name"]
        # the independent rational model agrees with the hand derivation too
        assert ieee_ref.gemm_bits(A, B, mode).tolist() == pin[key], pin["name"]


@pytest.mark.parametrize("mode", [oracle.EXACT, oracle.FAST])
def test_golden_conv_pins(mode):
    d = json.load(open(os.path.join(GOLDEN, "conv_pins.json")))
    key = "exact_bits" if mode == oracle.EXACT else "fast_bits"
    for pin in d["pins"]:
        s = pin["shape"]
        x = np.array(pin["x_bits"], np.uint32).view(np.float32).reshape(s["N"], s["Cin"], s["H"], s["W"])
        w = np.array(pin["w_bits"], np.uint32).view(np.float32).reshape(
            s["Cout"], s["Cin"] // s["G"], s["KH"], s["KW"])
        y = oracle.conv2d(x, w, s["stride"], s["pad"], s["dil"], s["G"], mode)
        assert bits(y).reshape(-1).tolist() == pin[key], pin["name"]


def test_golden_out_dims():
    d = json.load(open(os.path.join(GOLDEN, "conv_pins.json")))
    for c in d["out_dims"]["cases"]:
        got = oracle.conv_out_dim(c["size"], c["k"], c["stride"], c["pad"], c["pad"], c["dil"])
        assert got == c["out"], c


def test_out_dims_match_torch_shapes():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(3)
    for _ in range(200):
        size, k = int(rng.integers(1, 20)), int(rng.integers(1, 6))
        s, p, d = int(rng.integers(1, 4)), int(rng.integers(0, 3)), int(rng.integers(1, 3))
        want_pos = size + 2 * p - d * (k - 1) - 1 >= 0
        got = oracle.conv_out_dim(size, k, s, p, p, d)
        if not want_pos:
            assert got == 0
            continue
        y = torch.nn.functional.conv2d(torch.zeros(1, 1, size, size), torch.zeros(1, 1, k, k),
                                       stride=s, padding=p, dilation=d)
        assert got == y.shape[-1]


# --- brute force on tiny inputs against the rational model -----------------
@pytest.mark.parametrize("mode", [oracle.EXACT, oracle.FAST])
def test_brute_force_tiny_gemm(mode):
    rng = np.random.default_rng(11 + mode)
    for m in range(0, 4):
        for n in range(0, 4):
            for k in range(0, 5):
                A = (rng.standard_normal((m, k)) * 2.0 ** rng.integers(-3, 4, (m, k))).astype(np.float32)
                B = (rng.standard_normal((k, n)) * 2.0 ** rng.integers(-3, 4, (k, n))).astype(np.float32)
                C = oracle.gemm(A, B, mode)
                assert bits(C).tolist() == ieee_ref.gemm_bits(A, B, mode).tolist(), (m, n, k)


@pytest.mark.parametrize("mode", [oracle.EXACT, oracle.FAST])
def test_brute_force_specials(mode):
    rng = np.random.default_rng(21 + mode)
    pool = np.array([np.nan, np.inf, -np.inf, 0.0, -0.0, 1e-40, -1e-40, 1.0, -1.0, 3e38,
                     1.5, -2.75, 1e-30, 7.0], np.float32)
    for _ in range(60):
        m, n, k = (int(v) for v in rng.integers(1, 4, 3))
        A = rng.choice(pool, (m, k)).astype(np.float32)
        B = rng.choice(pool, (k, n)).astype(np.float32)
        C = oracle.gemm(A, B, mode)
        assert bits(C).tolist() == ieee_ref.gemm_bits(A, B, mode).tolist()


def test_modes_differ_only_by_fusion_on_random_sums():
    # With tie-free random data the fused and unfused sums generally differ
    # somewhere; if they never did, one of the modes would not be doing its job.
    rng = np.random.default_rng(5)
    A = rng.standard_normal((16, 64)).astype(np.float32)
    B = rng.standard_normal((64, 16)).astype(np.float32)
    e = oracle.gemm(A, B, oracle.EXACT)
    f = oracle.gemm(A, B, oracle.FAST)
    assert (bits(e) != bits(f)).any()
    assert bits(e[:2, :2]).tolist() == ieee_ref.gemm_bits(A[:2], B[:, :2], 0).tolist()
    assert bits(f[:2, :2]).tolist() == ieee_ref.gemm_bits(A[:2], B[:, :2], 1).tolist()


# --- closed forms ----------------------------------------------------------
@pytest.mark.parametrize("mode", [oracle.EXACT, oracle.FAST])
def test_k_zero_gives_plus_zero(mode):
    case = synth.workload_gemm_small_strided(with_k0=True)
    C = case.C_init.copy()
    oracle.gemm_raw(case.m, case.n, 0, case.A, case.lda, case.B, case.ldb, C, case.ldc, mode)
    assert (bits(C)[:, :case.n] == 0).all()
    assert (bits(C)[:, case.n:] == synth.C_SENTINEL_BITS).all()


@pytest.mark.parametrize("mode", [oracle.EXACT, oracle.FAST])
def test_k_one_is_rounded_product(mode):
    rng = np.random.default_rng(2)
    a = rng.standard_normal((9, 1)).astype(np.float32)
    b = rng.standard_normal((1, 7)).astype(np.float32)
    want = (a.astype(np.float32) * b.astype(np.float32)).astype(np.float32)  # numpy binary32 multiply
    assert bits(oracle.gemm(a, b, mode)).tolist() == bits(want).tolist()


@pytest.mark.parametrize("mode", [oracle.EXACT, oracle.FAST])
def test_identity_right_factor(mode):
    rng = np.random.default_rng(4)
    A = rng.standard_normal((13, 29)).astype(np.float32)
    A[0, 0] = -0.0  # -0 * 1 = -0, +0 + -0 = +0: the identity gives +0 there
    C = oracle.gemm(A, np.eye(29, dtype=np.float32), mode)
    want = A.copy()
    want[0, 0] = 0.0
    assert bits(C).tolist() == bits(want).tolist()


@pytest.mark.parametrize("mode", [oracle.EXACT, oracle.FAST])
def test_small_integers_are_exact(mode):
    # |values| <= 2^7 and k*max|ab| < 2^24: every product and partial sum is exact.
    rng = np.random.default_rng(8)
    A = rng.integers(-64, 65, (31, 47))
    B = rng.integers(-64, 65, (47, 23))
    C = oracle.gemm(A.astype(np.float32), B.astype(np.float32), mode)
    assert (C.astype(np.int64) == A @ B).all()


def test_transposed_operands_are_distinguished():
    rng = np.random.default_rng(9)
    A = rng.integers(-8, 9, (5, 7)).astype(np.float32)
    B = rng.integers(-8, 9, (7, 3)).astype(np.float32)
    C = oracle.gemm(A, B)
    assert (C == (A.astype(np.int64) @ B.astype(np.int64))).all()
    # the strided entry point reads A with lda and B with ldb, not the other way
    Ap = np.full((5, 10), np.nan, np.float32); Ap[:, :7] = A
    Bp = np.full((7, 6), np.nan, np.float32); Bp[:, :3] = B
    Cp = np.full((5, 4), 123.0, np.float32)
    oracle.gemm_raw(5, 3, 7, Ap, 10, Bp, 6, Cp, 4, oracle.EXACT)
    assert (Cp[:, :3] == C).all() and (Cp[:, 3] == 123.0).all()


@pytest.mark.parametrize("mode", [oracle.EXACT, oracle.FAST])
def test_sequential_sum_error_bound(mode):
    # |c - exact| <= k * u * sum|a_p b_p| (+1e-30 for the subnormal range).
    rng = np.random.default_rng(12)
    for (m, n, k) in [(8, 8, 1000), (4, 5, 4096), (3, 3, 17)]:
        A = rng.standard_normal((m, k)).astype(np.float32)
        B = rng.standard_normal((k, n)).astype(np.float32)
        C = oracle.gemm(A, B, mode).astype(np.float64)
        ref, mag = oracle.gemm_f64(A, B)
        assert (np.abs(C - ref) <= k * U * mag + 1e-30).all()


def test_thread_count_does_not_change_bits():
    case = synth.make_gemm("t", 37, 41, 129, seed=10)
    outs = []
    for t in (1, 3, 8):
        C = case.C_init.copy()
        oracle.gemm_raw(case.m, case.n, case.k, case.A, case.lda, case.B, case.ldb, C, case.ldc, 0, t)
        outs.append(bits(C).copy())
    assert all((o == outs[0]).all() for o in outs)


# --- the strided workload: padding never read, never written ---------------
@pytest.mark.parametrize("mode", [oracle.EXACT, oracle.FAST])
def test_strided_workload_padding(mode):
    case = synth.workload_gemm_small_strided()
    C = case.C_init.copy()
    oracle.gemm_raw(case.m, case.n, case.k, case.A, case.lda, case.B, case.ldb, C, case.ldc, mode)
    assert (bits(C)[:, case.n:] == synth.C_SENTINEL_BITS).all()
    used = C[:, :case.n]
    # NaN padding in A and B would poison every output if it were read
    assert np.isfinite(used).mean() > 0.5
    dense = oracle.gemm(case.A[:, :case.k], case.B[:, :case.n], mode)
    assert bits(used).tolist() == bits(dense).tolist()
    assert ((bits(used) == 0x7FC00000) | ~np.isnan(used)).all()


# --- convolution ------------------------------------------------------------
def im2col(x, KH, KW, stride, pad, dil, groups):
    """Explicit patch matrix per (image, group), rows ordered (c, ky, kx); numpy only."""
    N, Cin, H, W = x.shape
    cg = Cin // groups
    OH = (H + 2 * pad - dil * (KH - 1) - 1) // stride + 1
    OW = (W + 2 * pad - dil * (KW - 1) - 1) // stride + 1
    xp = np.zeros((N, Cin, H + 2 * pad, W + 2 * pad), np.float32)
    xp[:, :, pad:pad + H, pad:pad + W] = x
    cols = np.zeros((N, groups, cg * KH * KW, OH * OW), np.float32)
    for c in range(cg):
        for ky in range(KH):
            for kx in range(KW):
                r = (c * KH + ky) * KW + kx
                win = xp[:, :, ky * dil: ky * dil + stride * (OH - 1) + 1: stride,
                         kx * dil: kx * dil + stride * (OW - 1) + 1: stride]
                for g in range(groups):
                    cols[:, g, r, :] = win[:, g * cg + c].reshape(N, -1)
    return cols, OH, OW


CONV_SHAPES = [
    # N, Cin, H, W, Cout, G, KH, KW, s, p, d
    (2, 3, 7, 6, 4, 1, 3, 3, 1, 1, 1),
    (1, 4, 9, 9, 6, 2, 3, 2, 2, 1, 2),
    (2, 8, 5, 5, 8, 8, 3, 3, 1, 2, 1),
    (1, 6, 11, 4, 3, 3, 1, 1, 1, 0, 1),
    (3, 2, 4, 9, 5, 1, 2, 3, 3, 0, 1),
]


@pytest.mark.parametrize("shape", CONV_SHAPES)
@pytest.mark.parametrize("mode", [oracle.EXACT, oracle.FAST])
def test_conv_equals_gemm_over_explicit_im2col(shape, mode):
    N, Cin, H, W, Cout, G, KH, KW, s, p, d = shape
    case = synth.make_conv("t", N, Cin, H, W, Cout, G, KH, KW, s, p, d, seed=31,
                           dist_x=("uniform", -1.0, 1.0), dist_w=("normal", 0.0, 1.0))
    y = oracle.conv2d(case.x, case.w, s, p, d, G, mode)
    cols, OH, OW = im2col(case.x, KH, KW, s, p, d, G)
    cog = Cout // G
    wm = case.w.reshape(G, cog, -1)
    for n in range(N):
        for g in range(G):
            yg = oracle.gemm(wm[g], cols[n, g], mode).reshape(cog, OH, OW)
            assert bits(y[n, g * cog:(g + 1) * cog]).tolist() == bits(yg).tolist()


def test_conv_small_integers_match_correlate2d():
    signal = pytest.importorskip("scipy.signal")
    rng = np.random.default_rng(17)
    x = rng.integers(-5, 6, (2, 3, 8, 7)).astype(np.float32)
    w = rng.integers(-5, 6, (4, 3, 3, 3)).astype(np.float32)
    y = oracle.conv2d(x, w, 1, 0, 1, 1)
    for n in range(2):
        for oc in range(4):
            want = sum(signal.correlate2d(x[n, c].astype(np.int64), w[oc, c].astype(np.int64), "valid")
                       for c in range(3))
            assert (y[n, oc].astype(np.int64) == want).all()


def test_conv_small_integers_match_torch_conv2d():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(18)
    for (N, Cin, H, W, Cout, G, KH, KW, s, p, d) in CONV_SHAPES:
        x = rng.integers(-4, 5, (N, Cin, H, W)).astype(np.float32)
        w = rng.integers(-4, 5, (Cout, Cin // G, KH, KW)).astype(np.float32)
        y = oracle.conv2d(x, w, s, p, d, G)
        t = torch.nn.functional.conv2d(torch.from_numpy(x).double(), torch.from_numpy(w).double(),
                                       stride=s, padding=p, dilation=d, groups=G)
        assert np.array_equal(y.astype(np.float64), t.numpy())


@pytest.mark.parametrize("mode", [oracle.EXACT, oracle.FAST])
def test_conv_1x1_is_gemm_on_input_planes(mode):
    case = synth.make_conv("t", 2, 12, 5, 7, 9, 1, 1, 1, 1, 0, 1, seed=40,
                           dist_x=("normal", 0.0, 1.0), dist_w=("normal", 0.0, 1.0))
    y = oracle.conv2d(case.x, case.w, 1, 0, 1, 1, mode)
    for n in range(2):
        g = oracle.gemm(case.w.reshape(9, 12), case.x[n].reshape(12, -1), mode)
        assert bits(y[n].reshape(9, -1)).tolist() == bits(g).tolist()


@pytest.mark.parametrize("mode", [oracle.EXACT, oracle.FAST])
def test_conv_error_bound(mode):
    case = synth.make_conv("t", 2, 16, 9, 9, 8, 2, 3, 3, 1, 1, 1, seed=41,
                           dist_x=("normal", 0.0, 1.0), dist_w=("normal", 0.0, 1.0))
    y = oracle.conv2d(case.x, case.w, 1, 1, 1, 2, mode).astype(np.float64)
    ref, mag = oracle.conv2d_f64(case.x, case.w, 1, 1, 1, 2)
    k = 8 * 9
    assert (np.abs(y - ref) <= k * U * mag + 1e-30).all()


def test_grouped_workload_nonfinite_weights_reach_outputs():
    case = synth.workload_conv_grouped()
    # a cut-down copy of the grouped workload keeps every non-finite weight
    x = case.x[:2]
    y = oracle.conv2d(x, case.w, case.stride, case.pad, case.dil, case.G)
    yb = bits(y)
    nan = np.isnan(y)
    assert nan.any()
    assert (yb[nan] == 0x7FC00000).all()
    bad_oc = sorted({i // (case.w[0].size) for i in case.special["w_cells"]})
    # an infinite weight makes every output of its channel infinite or NaN
    assert (~np.isfinite(y[:, bad_oc])).all()
    # every output of an output channel holding a NaN weight is NaN (padding taps included)
    nan_w_oc = sorted({i // case.w[0].size for i in case.special["w_cells"]
                       if np.isnan(case.w.reshape(-1)[i])})
    assert nan[:, nan_w_oc].all()


def test_f64_companions_are_exact_sums_on_small_integers():
    """The binary64 companions behind every error bound: with small integers
    of both signs each product and partial sum is exact in binary64, so ref
    must equal the integer sum of a*b and mag the integer sum of |a*b|
    (a missing absolute value, a dropped term or a transposed index fails)."""
    rng = np.random.default_rng(19)
    A = rng.integers(-9, 10, (6, 11))
    B = rng.integers(-9, 10, (11, 5))
    ref, mag = oracle.gemm_f64(A.astype(np.float32), B.astype(np.float32))
    assert np.array_equal(ref, (A @ B).astype(np.float64))
    assert np.array_equal(mag, (np.abs(A) @ np.abs(B)).astype(np.float64))
    assert (mag > np.abs(ref)).any()  # cancellation present, so |.| matters
    for (N, Cin, H, W, Cout, G, KH, KW, s, p, d) in CONV_SHAPES:
        x = rng.integers(-4, 5, (N, Cin, H, W))
        w = rng.integers(-4, 5, (Cout, Cin // G, KH, KW))
        ref, mag = oracle.conv2d_f64(x.astype(np.float32), w.astype(np.float32), s, p, d, G)
        cols, OH, OW = im2col(x.astype(np.float32), KH, KW, s, p, d, G)
        cog = Cout // G
        wm = w.reshape(G, cog, -1)
        for n in range(N):
            for g in range(G):
                cg = cols[n, g].astype(np.int64)
                want = (wm[g] @ cg).reshape(cog, OH, OW)
                want_mag = (np.abs(wm[g]) @ np.abs(cg)).reshape(cog, OH, OW)
                assert np.array_equal(ref[n, g * cog:(g + 1) * cog], want.astype(np.float64))
                assert np.array_equal(mag[n, g * cog:(g + 1) * cog], want_mag.astype(np.float64))


def test_conv_thread_count_does_not_change_bits():
    case = synth.make_conv("t", 3, 8, 10, 10, 8, 2, 3, 3, 1, 1, 1, seed=42)
    ys = [bits(oracle.conv2d(case.x, case.w, 1, 1, 1, 2, 0, t)).copy() for t in (1, 4)]
    assert (ys[0] == ys[1]).all()


# --- output epilogue (bias, residual, ReLU) ---------------------------------
def test_golden_epilogue_pins():
    d = json.load(open(os.path.join(GOLDEN, "epilogue_pins.json")))
    for pin in d["pins"]:
        y = np.array(pin["y"], np.float32)
        if "shape" in pin:
            y = y.reshape(pin["shape"])
        else:
            y = y.reshape(1, -1)
        bias = None if pin["bias"] is None else np.array(pin["bias"], np.float32)
        res = None if pin["res"] is None else np.array(pin["res"], np.float32).reshape(y.shape)
        if bias is not None and "shape" not in pin:
            bias = np.full(y.shape[1], bias[0], np.float32)
        out = oracle.epilogue(y, bias, res, pin["act"])
        assert bits(out).reshape(-1).tolist() == pin["out_bits"], pin["name"]


def test_epilogue_matches_rational_model():
    rng = np.random.default_rng(33)
    y = (rng.standard_normal((6, 7)) * 10).astype(np.float32)
    bias = (rng.standard_normal(7) * 10).astype(np.float32)
    res = (rng.standard_normal((6, 7)) * 10).astype(np.float32)
    out = oracle.epilogue(y, bias, res, oracle.RELU)
    for i in range(6):
        for j in range(7):
            v = ieee_ref.add(ieee_ref.add(float(y[i, j]), float(bias[j])), float(res[i, j]))
            v = v if (v > 0 or math.isnan(v)) else 0.0
            assert bits(out)[i, j] == ieee_ref.canonical_bits(v)


def test_epilogue_on_conv_equals_torch_with_integers():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(34)
    x = rng.integers(-3, 4, (2, 4, 6, 6)).astype(np.float32)
    w = rng.integers(-3, 4, (6, 4, 3, 3)).astype(np.float32)
    b = rng.integers(-20, 21, 6).astype(np.float32)
    r = rng.integers(-20, 21, (2, 6, 6, 6)).astype(np.float32)
    y = oracle.epilogue(oracle.conv2d(x, w, 1, 1, 1, 1), b, r, oracle.RELU)
    t = torch.nn.functional.conv2d(torch.from_numpy(x).double(), torch.from_numpy(w).double(),
                                   torch.from_numpy(b).double(), padding=1)
    t = torch.relu(t + torch.from_numpy(r).double())
    assert np.array_equal(y.astype(np.float64), t.numpy())
