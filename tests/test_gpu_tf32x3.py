"""OM_MODE_TF32X3: the tensor-core tolerance mode (tcgen05, three-product TF32
split). It is not bit-exact; it must stay within the documented bound
|C - C_exact| <= 1e-5 * sqrt(k) * sum_p |a_p| |b_p| for finite exact results.
"""
import math

import numpy as np
import pytest

import implicit_gemm_convolution_gb300 as om
import oracle
from implicit_gemm_convolution_gb300 import synth
from tests.gpu_util import bits, guarded_output, guards_intact, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    om.build()
    om.lib()
    oracle.build()


def run_tf32x3(case):
    import torch
    A, B = to_dev(case.A), to_dev(case.B)
    buf, C = guarded_output(case.C_init)
    st = om.gemm_raw(case.m, case.n, case.k, A.data_ptr(), case.lda, B.data_ptr(), case.ldb,
                     C.data_ptr(), case.ldc, "tf32x3")
    assert st == 0, om.STATUS_NAMES.get(st, st)
    torch.cuda.synchronize()
    assert om.device_status() == 0
    assert guards_intact(buf)
    return C.cpu().numpy().reshape(case.C_init.shape)


def check_bound(got, case, rows=None):
    r0, r1 = rows if rows else (0, case.m)
    A = case.A[r0:r1, :case.k]
    B = case.B[:, :case.n]
    exact = oracle.gemm(A, B, oracle.EXACT, oracle.default_threads()).astype(np.float64)
    _, mag = oracle.gemm_f64(A, B, oracle.default_threads())
    g = got[r0:r1, :case.n].astype(np.float64)
    err = np.abs(g - exact)
    bound = 1e-5 * math.sqrt(max(case.k, 1)) * mag
    assert (err <= bound).all(), f"max err/bound {np.max(err / np.maximum(bound, 1e-300))}"
    return float(np.max(err / np.maximum(mag, 1e-300)))


@pytest.mark.parametrize("shape", [(128, 128, 32), (300, 520, 200), (1, 1, 1), (129, 257, 65),
                                   (640, 384, 1000), (77, 1000, 3)])
def test_bound_random(shape):
    m, n, k = shape
    case = synth.make_gemm("tc", m, n, k, seed=m + 3 * n + 7 * k, dist_a=("normal", 0, 1),
                           dist_b=("normal", 0, 1))
    got = run_tf32x3(case)
    rel = check_bound(got, case)
    # three products keep the error far below single-TF32 rounding (2^-11)
    assert rel < 2.0 ** -16
    assert (bits(got)[:, case.n:] == synth.C_SENTINEL_BITS).all()


def test_split_products_are_all_present():
    # a = 1 + ja*2^-20, b = 1 + jb*2^-20: hi = 1, lo = j*2^-20 exactly. With k = 1,
    # lo*hi + hi*lo + hi*hi = 1 + (ja+jb)*2^-20, which is also round(a*b): a dropped
    # or doubled product changes the bits.
    rng = np.random.default_rng(3)
    ja = rng.integers(1, 8, (130, 1))
    jb = rng.integers(1, 8, (1, 140))
    A = (1.0 + ja * 2.0 ** -20).astype(np.float32)
    B = (1.0 + jb * 2.0 ** -20).astype(np.float32)
    got = om.gemm(to_dev(A), to_dev(B), mode="tf32x3").cpu().numpy()
    want = (A.astype(np.float32) * B.astype(np.float32))
    assert np.array_equal(bits(got), bits(want))


def test_4096_cube_sampled_rows():
    case = synth.workload_gemm_4096()
    got = run_tf32x3(case)
    for r in [(0, 2), (2047, 2049), (4094, 4096)]:
        check_bound(got, case, r)


def test_prefill_sampled_rows():
    case = synth.workload_gemm_prefill(False)
    got = run_tf32x3(case)
    for r in [(0, 2), (510, 512)]:
        check_bound(got, case, r)


def test_nonfinite_inputs_give_nonfinite_outputs():
    rng = np.random.default_rng(5)
    A = rng.standard_normal((130, 70)).astype(np.float32)
    B = rng.standard_normal((70, 150)).astype(np.float32)
    A[3, 5] = np.inf
    A[7, 1] = np.nan
    B[2, 9] = -np.inf
    got = om.gemm(to_dev(A), to_dev(B), mode="tf32x3").cpu().numpy()
    exact = oracle.gemm(A, B, oracle.EXACT)
    nonfinite = ~np.isfinite(exact)
    assert nonfinite.any()
    assert (~np.isfinite(got[nonfinite])).all()
    assert (bits(got)[np.isnan(got)] == 0x7FC00000).all()
    fin = np.isfinite(exact)
    _, mag = oracle.gemm_f64(np.where(np.isfinite(A), A, 0), np.where(np.isfinite(B), B, 0))
    assert (np.abs(got[fin].astype(np.float64) - exact[fin]) <= 1e-5 * math.sqrt(70) * mag[fin]).all()


def test_k_zero_and_unaligned_operands():
    import torch
    C = torch.full((5, 6), 3.0, device="cuda")
    A = torch.zeros((5, 1), device="cuda")
    B = torch.zeros((1, 6), device="cuda")
    assert om.gemm_raw(5, 6, 0, A.data_ptr(), 1, B.data_ptr(), 6, C.data_ptr(), 6, "tf32x3") == 0
    torch.cuda.synchronize()
    assert (C.cpu().numpy().view(np.uint32) == 0).all()
    # lda = 67 is not a multiple of 4: TMA cannot fetch A, so the fast-mode CUDA-core
    # kernel computes the call; its bits equal fast mode's
    rng = np.random.default_rng(6)
    A = rng.standard_normal((64, 67)).astype(np.float32)
    B = rng.standard_normal((67, 64)).astype(np.float32)
    got = om.gemm(to_dev(A), to_dev(B), mode="tf32x3").cpu().numpy()
    assert np.array_equal(bits(got), bits(oracle.gemm(A, B, oracle.FAST)))
