"""GPU parity of the matrix-vector kernels against the oracle, bit for bit.

Products with at most 8 rows or 8 columns, and 1x1 convolutions over 1x1
inputs of at most 8 images, take the matrix-vector kernels by default; the
16-byte copy path (rows 16-byte aligned) and the 4-byte path are both
covered, with ragged k and strip tails.
"""
import numpy as np
import pytest

import implicit_gemm_convolution_gb300 as om
import oracle
from implicit_gemm_convolution_gb300 import synth
from tests.gpu_util import (assert_bits_equal, bits, forced_config, guarded_output,
                            guards_intact, to_dev)

pytestmark = pytest.mark.gpu

MODES = [(oracle.EXACT, "exact"), (oracle.FAST, "fast")]


@pytest.fixture(scope="module", autouse=True)
def built():
    om.build()
    om.lib()
    oracle.build()


def run_gemm(case, name, cfg=None):
    import torch
    A, B = to_dev(case.A), to_dev(case.B)
    buf, C = guarded_output(case.C_init)
    with forced_config("OM_FORCE_GEMM_CFG", cfg):
        st = om.gemm_raw(case.m, case.n, case.k, A.data_ptr(), case.lda, B.data_ptr(), case.ldb,
                         C.data_ptr(), case.ldc, name)
    assert st == 0, om.STATUS_NAMES.get(st, st)
    torch.cuda.synchronize()
    assert om.device_status() == 0
    assert guards_intact(buf), "write outside C"
    return C.cpu().numpy().reshape(case.C_init.shape)


def want_gemm(case, mode):
    want = case.C_init.copy()
    oracle.gemm_raw(case.m, case.n, case.k, case.A, case.lda, case.B, case.ldb, want, case.ldc,
                    mode, oracle.default_threads())
    return want


def specials(m, n, k):
    """Seeded NaN/inf/-0/subnormal cells, two in A and two in B, when both have room."""
    return 4 if min(m * k, k * n) >= 2 else 0


def ld_variants(cols):
    """A leading dimension that is a multiple of 4 (16-byte rows) and one that is not."""
    aligned = (cols + 3) // 4 * 4
    return [aligned, aligned + 1]


# (m, n, k): at most 8 rows, column strips with ragged tails, k ragged
# against the stages, k below one stage
FEW_ROWS = [(1, 1, 1), (1, 300, 70), (2, 7, 31), (3, 1000, 300), (5, 129, 1), (8, 64, 33),
            (8, 4097, 65), (6, 190, 1000),
            # more 128-column strips than SMs: some blocks stream two strips
            (2, 20000, 70)]
# (m, n, k): at most 8 columns
FEW_COLS = [(300, 1, 33), (1000, 1, 300), (65, 8, 33), (129, 3, 64), (70, 2, 1), (200, 5, 1001)]


@pytest.mark.parametrize("shape", FEW_ROWS)
@pytest.mark.parametrize("mode,name", MODES)
def test_few_rows(shape, mode, name):
    m, n, k = shape
    for ldb in ld_variants(n):
        case = synth.make_gemm("gv", m, n, k, lda=k + 3, ldb=ldb, ldc=n + 1,
                               seed=m * 11 + n * 5 + k + ldb,
                               special_cells=specials(m, n, k))
        got = run_gemm(case, name)
        assert_bits_equal(got, want_gemm(case, mode), f"{shape} ldb={ldb}")
        assert (bits(got)[:, n:] == synth.C_SENTINEL_BITS).all()


@pytest.mark.parametrize("shape", FEW_COLS)
@pytest.mark.parametrize("mode,name", MODES)
def test_few_columns(shape, mode, name):
    m, n, k = shape
    for lda in ld_variants(k):
        case = synth.make_gemm("gv", m, n, k, lda=lda, ldb=n + 2, ldc=n + 1,
                               seed=m * 13 + n * 3 + k + lda,
                               special_cells=specials(m, n, k))
        got = run_gemm(case, name)
        assert_bits_equal(got, want_gemm(case, mode), f"{shape} lda={lda}")


@pytest.mark.parametrize("mode,name", MODES)
def test_decode_shaped_product(mode, name):
    # one token times the prefill workload's weight matrix (4096 x 11008)
    case = synth.make_gemm("decode", 1, 11008, 4096, seed=42, dist_a=("normal", 0, 1),
                           dist_b=("normal", 0, 0.02))
    assert_bits_equal(run_gemm(case, name), want_gemm(case, mode), "1 x 11008 x 4096")


@pytest.mark.parametrize("mode,name", MODES)
def test_decode_workload_full_size(mode, name):
    # the benchmark's decode line: its own seeded operands, whole output
    case = synth.workload_gemm_decode()
    assert_bits_equal(run_gemm(case, name), want_gemm(case, mode), "decode workload")


@pytest.mark.parametrize("mode,name", MODES)
def test_forced_gemv_on_a_wide_product_falls_back(mode, name):
    case = synth.make_gemm("gv", 40, 50, 20, seed=3)
    assert_bits_equal(run_gemm(case, name, cfg=5), want_gemm(case, mode), "forced gemv 40x50")


@pytest.mark.parametrize("mode,name", MODES)
def test_few_rows_epilogue(mode, name):
    m, n, k = 3, 333, 130
    rng = np.random.default_rng(9)
    A = rng.standard_normal((m, k)).astype(np.float32)
    B = rng.standard_normal((k, n)).astype(np.float32)
    bias = rng.standard_normal(n).astype(np.float32)
    bias[[3, 40]] = [np.inf, np.nan]
    res = (rng.standard_normal((m, n)) * 3).astype(np.float32)
    want = oracle.epilogue(oracle.gemm(A, B, mode), bias, res, oracle.RELU)
    got = om.gemm_ex(to_dev(A), to_dev(B), to_dev(bias), to_dev(res), "relu", mode=name)
    assert_bits_equal(got.cpu().numpy(), want, "gemv epilogue rows")
    At = np.ascontiguousarray(B.T)  # 333 x 130 times 130 x 3
    Bt = np.ascontiguousarray(A.T)
    bias3 = bias[:m].copy()
    res_t = np.ascontiguousarray(res.T)
    want_t = oracle.epilogue(oracle.gemm(At, Bt, mode), bias3, res_t, oracle.RELU)
    got_t = om.gemm_ex(to_dev(At), to_dev(Bt), to_dev(bias3), to_dev(res_t), "relu", mode=name)
    assert_bits_equal(got_t.cpu().numpy(), want_t, "gemv epilogue columns")


# 1x1 convolutions over 1x1 inputs: N, Cin, Cout, G
FC = [(1, 64, 100, 1), (3, 5, 7, 1), (8, 260, 96, 2), (2, 2048, 1000, 1), (5, 12, 18, 3)]


@pytest.mark.parametrize("shape", FC)
@pytest.mark.parametrize("mode,name", MODES)
def test_1x1_conv_over_1x1_input(shape, mode, name):
    import torch
    N, Cin, Cout, G = shape
    c = synth.make_conv("fc", N, Cin, 1, 1, Cout, G, 1, 1, 1, 0, 1, seed=N + Cin + Cout,
                        dist_x=("uniform", -1, 1), dist_w=("normal", 0, 0.3))
    want = oracle.conv2d(c.x, c.w, 1, 0, 1, G, mode, oracle.default_threads())
    x, w = to_dev(c.x), to_dev(c.w)
    for cfg in (None, 3):
        with forced_config("OM_FORCE_CONV_CFG", cfg):
            got = om.conv2d(x, w, groups=G, mode=name)
            assert_bits_equal(got.cpu().numpy(), want, f"fc {shape} cfg={cfg}")
            wp = om.pack_conv_weights(w, G)
            got_p = om.conv2d_packed(x, wp, tuple(w.shape), groups=G, mode=name)
            assert_bits_equal(got_p.cpu().numpy(), want, f"fc packed {shape} cfg={cfg}")
    rng = np.random.default_rng(N * Cout)
    bias = rng.standard_normal(Cout).astype(np.float32)
    res = rng.standard_normal((N, Cout, 1, 1)).astype(np.float32)
    want_ep = oracle.epilogue(want, bias, res, oracle.RELU)
    got_ep = om.conv2d_ex(x, w, groups=G, bias=to_dev(bias), residual=to_dev(res),
                          activation="relu", mode=name)
    assert_bits_equal(got_ep.cpu().numpy(), want_ep, f"fc epilogue {shape}")
    torch.cuda.synchronize()
    assert om.device_status() == 0
