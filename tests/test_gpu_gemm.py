"""GPU parity of om_gemm_f32 against the CPU oracle, bit for bit.

Every kernel configuration (forced through the test-only override) must
give the oracle's bits; the default dispatch is what the benchmark times.
"""
import functools

import numpy as np
import pytest

import implicit_gemm_convolution_gb300 as om
import oracle
from implicit_gemm_convolution_gb300 import synth
from tests.gpu_util import (assert_bits_equal, bits, forced_config, guarded_output,
                            guards_intact, sha, to_dev)

pytestmark = pytest.mark.gpu

MODES = [(oracle.EXACT, "exact"), (oracle.FAST, "fast")]
# naive, TMA 128x256, TMA 128x128, cp.async 128x128, TMA 128x256 one-lane,
# A by TMA and B by cp.async 128x256 and 128x128, default
CFGS = [0, 1, 2, 3, 4, 6, 7, None]


@pytest.fixture(scope="module", autouse=True)
def built():
    om.build()
    om.lib()
    oracle.build()


def run_case(case: synth.GemmCase, name: str, cfg=None):
    """Runs the padded-buffer problem; returns (C host copy, guards intact)."""
    import torch
    A, B = to_dev(case.A), to_dev(case.B)
    buf, C = guarded_output(case.C_init)
    with forced_config("OM_FORCE_GEMM_CFG", cfg):
        st = om.gemm_raw(case.m, case.n, case.k, A.data_ptr(), case.lda, B.data_ptr(), case.ldb,
                         C.data_ptr(), case.ldc, name)
    assert st == 0, om.STATUS_NAMES.get(st, st)
    torch.cuda.synchronize()
    assert om.device_status() == 0
    return C.cpu().numpy().reshape(case.C_init.shape), guards_intact(buf)


def oracle_case(case: synth.GemmCase, mode: int, rows=None):
    want = case.C_init.copy()
    if rows is None:
        oracle.gemm_raw(case.m, case.n, case.k, case.A, case.lda, case.B, case.ldb, want, case.ldc,
                        mode, oracle.default_threads())
        return want
    r0, r1 = rows
    sub = want[r0:r1].copy()
    oracle.gemm_raw(r1 - r0, case.n, case.k, case.A[r0:r1].copy(), case.lda, case.B, case.ldb, sub,
                    case.ldc, mode, oracle.default_threads())
    return sub


@pytest.mark.parametrize("cfg", CFGS)
@pytest.mark.parametrize("mode,name", MODES)
def test_strided_specials_workload(mode, name, cfg):
    case = synth.workload_gemm_small_strided()
    got, ok = run_case(case, name, cfg)
    assert ok, "write outside C"
    assert_bits_equal(got, oracle_case(case, mode), f"67x53x300 {name} cfg={cfg}")
    assert (bits(got)[:, case.n:] == synth.C_SENTINEL_BITS).all()


@pytest.mark.parametrize("cfg", CFGS)
@pytest.mark.parametrize("mode,name", MODES)
def test_k_zero(mode, name, cfg):
    case = synth.workload_gemm_small_strided(with_k0=True)
    got, ok = run_case(case, name, cfg)
    assert ok
    assert (bits(got)[:, :case.n] == 0).all()
    assert (bits(got)[:, case.n:] == synth.C_SENTINEL_BITS).all()


TILED_SHAPES = [
    # several tiles in each direction plus ragged tails (m, n, k)
    (300, 520, 200), (129, 257, 65), (256, 512, 64), (1, 1, 1), (1, 300, 70), (300, 1, 33),
    (127, 255, 31), (260, 700, 1),
]


@pytest.mark.parametrize("shape", TILED_SHAPES)
@pytest.mark.parametrize("cfg", CFGS)
@pytest.mark.parametrize("mode,name", MODES)
def test_tiled_shapes(shape, mode, name, cfg):
    m, n, k = shape
    case = synth.make_gemm("t", m, n, k, seed=m * 7 + n * 3 + k, dist_a=("normal", 0, 1),
                           dist_b=("normal", 0, 1))
    got, ok = run_case(case, name, cfg)
    assert ok
    assert_bits_equal(got, oracle_case(case, mode), f"{shape} {name} cfg={cfg}")


@pytest.mark.parametrize("mode,name", MODES)
def test_random_strided_sweep(mode, name):
    # sizes 0..70 in each dimension with random leading-dimension padding
    rng = np.random.default_rng(1234 + mode)
    for trial in range(40):
        m, n, k = (int(v) for v in rng.integers(0, 71, 3))
        lda, ldb, ldc = k + int(rng.integers(0, 5)), n + int(rng.integers(0, 5)), n + int(rng.integers(0, 5))
        case = synth.make_gemm("sweep", m, n, k, lda=lda, ldb=ldb, ldc=ldc, seed=5000 + trial,
                               special_cells=int(rng.integers(0, 3)) * 2)
        if m == 0 or n == 0:
            continue
        for cfg in (None, 3):
            got, ok = run_case(case, name, cfg)
            assert ok
            assert_bits_equal(got, oracle_case(case, mode), f"sweep {m}x{n}x{k} cfg={cfg}")


@pytest.mark.parametrize("mode,name", MODES)
def test_special_values_everywhere(mode, name):
    rng = np.random.default_rng(77)
    pool = np.array([np.nan, np.inf, -np.inf, 0.0, -0.0, 1e-40, -1e-40, 1.0, -1.0, 3e38, 1.5],
                    np.float32)
    A = rng.choice(pool, (130, 40)).astype(np.float32)
    B = rng.choice(pool, (40, 260)).astype(np.float32)
    want = oracle.gemm(A, B, mode)
    for cfg in CFGS:
        with forced_config("OM_FORCE_GEMM_CFG", cfg):
            got = om.gemm(to_dev(A), to_dev(B), mode=name).cpu().numpy()
        assert_bits_equal(got, want, f"specials cfg={cfg}")


@pytest.mark.parametrize("mode,name", MODES)
def test_4096_cube_sampled_rows(mode, name):
    """The benchmark workload in the benchmark's launch configuration; the
    oracle computes a sample of whole rows (first, last and seeded)."""
    import torch
    case = synth.workload_gemm_4096()
    A, B = to_dev(case.A), to_dev(case.B)
    C = om.gemm(A, B, mode=name)
    torch.cuda.synchronize()
    got = C.cpu().numpy()
    rows = [(0, 4), (4092, 4096), (1357, 1361), (2048, 2050)]
    for r0, r1 in rows:
        assert_bits_equal(got[r0:r1], oracle_case(case, mode, (r0, r1)), f"4096^3 rows {r0}:{r1}")
    # repeatable bit for bit
    C2 = om.gemm(A, B, mode=name)
    assert sha(C2.cpu().numpy()) == sha(got)


@functools.lru_cache(maxsize=2)
def _prefill(ragged):
    return synth.workload_gemm_prefill(ragged)


@pytest.mark.parametrize("use_ws", [False, True])
@pytest.mark.parametrize("ragged", [False, True])
@pytest.mark.parametrize("mode,name", MODES)
def test_prefill_sampled_rows(mode, name, ragged, use_ws):
    """The prefill product (512 x 11008 x 4096) and its ragged variant
    (509 x 11005, B and C rows not 16-byte aligned) with the benchmark's
    inputs (A ~ N(0, 1), B ~ N(0, 0.02)), through the plain and the
    workspace entry points in both modes; sampled whole rows against the
    oracle, guard bands around C."""
    import torch
    case = _prefill(ragged)
    A, B = to_dev(case.A), to_dev(case.B)
    buf, C = guarded_output(case.C_init)
    ws = om.new_workspace() if use_ws else None
    st = om.gemm_raw(case.m, case.n, case.k, A.data_ptr(), case.lda, B.data_ptr(), case.ldb,
                     C.data_ptr(), case.ldc, name, workspace=ws)
    assert st == 0
    torch.cuda.synchronize()
    assert om.device_status() == 0
    assert guards_intact(buf)
    got = C.cpu().numpy().reshape(case.C_init.shape)
    for r0, r1 in [(0, 2), (case.m - 2, case.m), (255, 257), (127, 129)]:
        assert_bits_equal(got[r0:r1], oracle_case(case, mode, (r0, r1)),
                          f"prefill {case.m}x{case.n} {name} ws={use_ws} rows {r0}")


def test_config_independence_hash():
    case = synth.make_gemm("h", 333, 517, 250, seed=99, dist_a=("normal", 0, 1), dist_b=("normal", 0, 1))
    for mode, name in MODES:
        hashes = {sha(run_case(case, name, cfg)[0]) for cfg in CFGS}
        assert len(hashes) == 1, name


def test_fast_mode_error_bound_4096_rows():
    case = synth.workload_gemm_4096()
    import torch
    C = om.gemm(to_dev(case.A), to_dev(case.B), mode="fast")
    torch.cuda.synchronize()
    got = C.cpu().numpy()[:2].astype(np.float64)
    ref, mag = oracle.gemm_f64(case.A[:2], case.B, oracle.default_threads())
    assert (np.abs(got - ref) <= case.k * 2.0 ** -24 * mag + 1e-30).all()


# ---- balanced schedule (om_gemm_f32_ws): k-block continuation across CTAs
WS_SHAPES = [
    # (m, n, k): more tiles than SMs, not whole rounds, so the last rounds are split
    (2048, 2560, 1000), (4096, 4096, 4096), (1300, 5000, 333), (640, 7700, 64),
    (512, 11008, 4096),
]


@pytest.mark.parametrize("shape", WS_SHAPES)
@pytest.mark.parametrize("mode,name", MODES)
def test_workspace_schedule_is_bit_identical(shape, mode, name):
    import torch
    m, n, k = shape
    case = synth.make_gemm("ws", m, n, k, seed=m + n + k, dist_a=("normal", 0, 1),
                           dist_b=("normal", 0, 1))
    A, B = to_dev(case.A), to_dev(case.B)
    ws = om.new_workspace()
    plain = om.gemm(A, B, mode=name).cpu().numpy()
    for cfg in (None, 2, 4):
        with forced_config("OM_FORCE_GEMM_CFG", cfg):
            C = torch.full((m, n), float("nan"), device="cuda")
            om.gemm(A, B, out=C, mode=name, workspace=ws)
            assert_bits_equal(C.cpu().numpy(), plain, f"ws vs plain {shape} cfg={cfg}")
    torch.cuda.synchronize()
    assert om.device_status() == 0
    for r0 in (0, m // 2, m - 1):
        assert_bits_equal(plain[r0:r0 + 1], oracle_case(case, mode, (r0, r0 + 1)), f"rows {r0}")


@pytest.mark.parametrize("mode,name", MODES)
def test_workspace_with_specials_and_padding(mode, name):
    # strided operands (4-byte producer) and IEEE specials through the balanced schedule
    import torch
    case = synth.make_gemm("wsp", 1500, 3000, 200, lda=203, ldb=3001, ldc=3003, seed=77,
                           special_cells=8)
    A, B = to_dev(case.A), to_dev(case.B)
    buf, C = guarded_output(case.C_init)
    ws = om.new_workspace()
    st = om.gemm_raw(case.m, case.n, case.k, A.data_ptr(), case.lda, B.data_ptr(), case.ldb,
                     C.data_ptr(), case.ldc, name, workspace=ws)
    assert st == 0
    torch.cuda.synchronize()
    assert guards_intact(buf)
    got = C.cpu().numpy().reshape(case.C_init.shape)
    assert (bits(got)[:, case.n:] == synth.C_SENTINEL_BITS).all()
    plain, ok = run_case(case, name)
    assert_bits_equal(got, plain, "ws vs plain strided")
    for r in sorted({case.special["A_cells"][0] // case.k, 0, case.m - 1}):
        assert_bits_equal(got[r:r + 1], oracle_case(case, mode, (r, r + 1)), f"row {r}")


def test_workspace_validation():
    import torch
    ws = om.new_workspace()
    A = torch.zeros((64, 64), device="cuda")
    C = torch.zeros((64, 64), device="cuda")
    L = om.lib()
    args = (64, 64, 64, A.data_ptr(), 64, A.data_ptr(), 64, C.data_ptr(), 64, 0)
    assert L.om_gemm_f32_ws(*args, None, 4096, None) == 2
    assert L.om_gemm_f32_ws(*args, ws.data_ptr(), 16, None) == 1
    assert L.om_gemm_f32_ws(*args, ws.data_ptr() + 4, 8192, None) == 7
    assert L.om_gemm_f32_ws(*args, C.data_ptr(), 16384, None) == 3  # workspace inside C
    assert om.workspace_bytes() == 4096
