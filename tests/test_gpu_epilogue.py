"""Fused output epilogue (bias, then residual, then ReLU) on the GPU against
the oracle's epilogue applied to the oracle's product or convolution, bit for
bit, in every kernel configuration and both schedules."""
import numpy as np
import pytest

import implicit_gemm_convolution_gb300 as om
import oracle
from implicit_gemm_convolution_gb300 import synth
from tests.gpu_util import assert_bits_equal, forced_config, to_dev

pytestmark = pytest.mark.gpu

MODES = [(oracle.EXACT, "exact"), (oracle.FAST, "fast")]


@pytest.fixture(scope="module", autouse=True)
def built():
    om.build()
    om.lib()
    oracle.build()


def _specials(a, rng, count):
    pool = np.array([np.nan, np.inf, -np.inf, -0.0, 1e-40], np.float32)
    idx = rng.choice(a.size, count, replace=False)
    a.reshape(-1)[idx] = pool[np.arange(count) % len(pool)]
    return a


@pytest.mark.parametrize("shape", [(300, 520, 200), (1300, 5000, 333), (67, 53, 7)])
@pytest.mark.parametrize("act", [None, "relu"])
@pytest.mark.parametrize("mode,name", MODES)
def test_gemm_epilogue(shape, act, mode, name):
    import torch
    m, n, k = shape
    rng = np.random.default_rng(m + n + k)
    case = synth.make_gemm("ep", m, n, k, seed=m * 3 + n, dist_a=("normal", 0, 1),
                           dist_b=("normal", 0, 1))
    A, B = case.A[:, :k].copy(), case.B[:, :n].copy()
    bias = _specials(rng.standard_normal(n).astype(np.float32), rng, 3)
    res = _specials((rng.standard_normal((m, n)) * 4).astype(np.float32), rng, 5)
    want = oracle.epilogue(oracle.gemm(A, B, mode, oracle.default_threads()), bias, res,
                           0 if act is None else oracle.RELU)
    dA, dB, db, dr = to_dev(A), to_dev(B), to_dev(bias), to_dev(res)
    ws = om.new_workspace()
    for cfg in (None, 0, 1, 2, 3):
        for workspace in (None, ws):
            with forced_config("OM_FORCE_GEMM_CFG", cfg):
                got = om.gemm_ex(dA, dB, db, dr, act, mode=name, workspace=workspace)
            assert_bits_equal(got.cpu().numpy(), want, f"gemm ep {shape} cfg={cfg} ws={workspace is not None}")
    # bias only / residual only
    want_b = oracle.epilogue(oracle.gemm(A, B, mode, oracle.default_threads()), bias, None, 0)
    assert_bits_equal(om.gemm_ex(dA, dB, db, None, None, mode=name).cpu().numpy(), want_b, "bias only")
    torch.cuda.synchronize()
    assert om.device_status() == 0


CONVS = [
    (2, 16, 12, 12, 64, 1, 3, 3, 1, 1, 1),
    (4, 32, 9, 11, 96, 2, 1, 1, 1, 0, 1),
    (3, 24, 6, 10, 40, 2, 1, 1, 1, 0, 1),
    (2, 16, 14, 14, 16, 16, 3, 3, 1, 1, 1),
    (2, 16, 12, 16, 16, 16, 3, 3, 1, 1, 1),
    (1, 8, 13, 13, 8, 8, 3, 3, 2, 1, 2),
    # the row-segment kernel's shape (forced below as configuration 6)
    (2, 8, 8, 28, 64, 1, 3, 3, 1, 1, 1),
    # small groups (the direct kernel and the TMA window kernel, configurations 2 and 7)
    (2, 32, 12, 16, 48, 8, 3, 3, 2, 1, 2),
]


@pytest.mark.parametrize("shape", CONVS)
@pytest.mark.parametrize("mode,name", MODES)
def test_conv_epilogue(shape, mode, name):
    N, Cin, H, W, Cout, G, KH, KW, s, p, d = shape
    rng = np.random.default_rng(sum(shape))
    c = synth.make_conv("ep", *shape, seed=sum(shape) + 1, dist_x=("uniform", -1, 1),
                        dist_w=("normal", 0, 0.5))
    conv = oracle.conv2d(c.x, c.w, s, p, d, G, mode, oracle.default_threads())
    bias = _specials(rng.standard_normal(Cout).astype(np.float32), rng, 2)
    res = _specials(rng.standard_normal(conv.shape).astype(np.float32), rng, 4)
    want = oracle.epilogue(conv, bias, res, oracle.RELU)
    x, w, db, dr = to_dev(c.x), to_dev(c.w), to_dev(bias), to_dev(res)
    wp = om.pack_conv_weights(w, G)
    ws = om.new_workspace()
    for cfg in (None, 0, 1, 2, 6, 7):
        for workspace in (None, ws):
            for packed in (False, True):
                with forced_config("OM_FORCE_CONV_CFG", cfg):
                    got = om.conv2d_ex(x, w, s, p, d, G, db, dr, "relu", mode=name,
                                       workspace=workspace, w_packed=wp if packed else None)
                assert_bits_equal(got.cpu().numpy(), want,
                                  f"conv ep {shape} cfg={cfg} ws={workspace is not None} packed={packed}")


@pytest.mark.parametrize("mode,name", MODES)
def test_conv3x3_workload_epilogue_balanced(mode, name):
    # the benchmark's 3x3 layer, residual block style: relu(conv + bias + identity)
    c = synth.workload_conv3x3()
    rng = np.random.default_rng(12)
    bias = rng.standard_normal(64).astype(np.float32) * 0.1
    res = c.x.copy()  # identity shortcut, same shape as y
    x, w = to_dev(c.x), to_dev(c.w)
    got = om.conv2d_ex(x, w, 1, 1, 1, 1, to_dev(bias), to_dev(res), "relu", mode=name,
                       workspace=om.new_workspace()).cpu().numpy()
    conv0 = oracle.conv2d(c.x[:1], c.w, 1, 1, 1, 1, mode, oracle.default_threads())
    want0 = oracle.epilogue(conv0, bias, res[:1], oracle.RELU)
    assert_bits_equal(got[:1], want0, "conv3x3 + bias + identity + relu, image 0")


def test_tf32x3_epilogue_within_bound():
    import math
    rng = np.random.default_rng(4)
    A = rng.standard_normal((300, 200)).astype(np.float32)
    B = rng.standard_normal((200, 520)).astype(np.float32)
    bias = rng.standard_normal(520).astype(np.float32)
    res = rng.standard_normal((300, 520)).astype(np.float32)
    got = om.gemm_ex(to_dev(A), to_dev(B), to_dev(bias), to_dev(res), None, mode="tf32x3").cpu().numpy()
    exact = oracle.epilogue(oracle.gemm(A, B, oracle.EXACT), bias, res, 0).astype(np.float64)
    _, mag = oracle.gemm_f64(A, B)
    # the product's bound plus the two epilogue roundings
    slack = 1e-5 * math.sqrt(200) * mag + 4 * 2.0 ** -24 * (np.abs(exact) + np.abs(res) + np.abs(bias))
    assert (np.abs(got.astype(np.float64) - exact) <= slack).all()


def test_epilogue_validation():
    import torch
    L = om.lib()
    A = torch.zeros((64, 64), device="cuda")
    C = torch.zeros((64, 64), device="cuda")
    b = torch.zeros(64, device="cuda")
    args = (64, 64, 64, A.data_ptr(), 64, A.data_ptr(), 64, C.data_ptr(), 64)
    assert L.om_gemm_f32_ex(*args, b.data_ptr(), None, 0, 7, 0, None, 0, None) == 1  # activation
    assert L.om_gemm_f32_ex(*args, None, C.data_ptr(), 64, 1, 0, None, 0, None) == 3  # residual = C
    assert L.om_gemm_f32_ex(*args, None, A.data_ptr(), 32, 1, 0, None, 0, None) == 1  # short ldr
