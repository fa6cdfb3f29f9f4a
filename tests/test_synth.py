"""The seeded input generator: determinism, distributions and workload shapes."""
import math

import numpy as np

from implicit_gemm_convolution_gb300 import synth


def test_splitmix64_known_values():
    # SplitMix64 with state 0: the first outputs of the reference generator
    # (Steele, Lea and Flood 2014; also java.util.SplittableRandom(0).nextLong()).
    got = synth.raw_u64(0, 0, 3)
    assert [int(v) for v in got] == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_deterministic_and_stream_separated():
    a = synth.uniform(5, 1, (100,), -1, 1)
    b = synth.uniform(5, 1, (100,), -1, 1)
    c = synth.uniform(5, 2, (100,), -1, 1)
    assert (a == b).all() and not (a == c).all()


def test_distributions():
    u = synth.uniform(1, 1, (200000,), -1.0, 1.0)
    assert u.min() >= -1.0 and u.max() < 1.0 and abs(u.mean()) < 0.01
    z = synth.normal(1, 2, (200001,), 0.0, 0.02)
    assert z.shape == (200001,) and abs(z.std() - 0.02) < 0.0005 and abs(z.mean()) < 0.0005


def test_workload_shapes_and_specials():
    g = synth.workload_gemm_small_strided()
    assert (g.m, g.n, g.k, g.lda, g.ldb, g.ldc) == (67, 53, 300, 303, 58, 54)
    assert g.A.shape == (67, 303) and g.B.shape == (300, 58) and g.C_init.shape == (67, 54)
    assert np.isnan(g.A[:, 300:]).all() and np.isnan(g.B[:, 53:]).all()
    used_a = g.A[:, :300].reshape(-1)[g.special["A_cells"]]
    used_b = g.B[:, :53].reshape(-1)[g.special["B_cells"]]
    vals = np.concatenate([used_a, used_b])
    assert np.isnan(vals).sum() == 2 and np.isposinf(vals).sum() == 2 and np.isneginf(vals).sum() == 1
    assert (vals.view(np.uint32) == 0x80000000).sum() == 1
    c = synth.workload_conv_grouped()
    assert c.w.shape == (256, 8, 3, 3) and len(c.special["w_cells"]) == 18
    wb = c.w.reshape(-1)
    assert (~np.isfinite(wb)).sum() == 18
    assert (wb.view(np.uint32) == 0xFFC00001).sum() == 1
    c3 = synth.workload_conv3x3()
    assert abs(float(c3.w.std()) - math.sqrt(2 / 576)) < 0.003
