"""Seeded random convolution shapes through every dispatch path, bit for bit
against the oracle: the default routing and each forced configuration (a
configuration that declines a shape falls back to another path, which must
give the same bits)."""
import numpy as np
import pytest

import implicit_gemm_convolution_gb300 as om
import oracle
from implicit_gemm_convolution_gb300 import synth
from tests.test_gpu_conv import MODES, run_conv, want_conv

pytestmark = pytest.mark.gpu


def random_shapes(seed, count):
    rng = np.random.default_rng(seed)
    out = []
    while len(out) < count:
        G = int(rng.choice([1, 1, 2, 4, 8]))
        cin_g = int(rng.choice([1, 2, 3, 4, 8, 16]))
        m = int(rng.choice([1, 2, 3, 4, 6, 8, 12, 16, 24, 64]))
        k = int(rng.choice([1, 3, 5]))
        s = int(rng.choice([1, 1, 2]))
        d = int(rng.choice([1, 1, 2]))
        p = int(rng.integers(0, k))
        H = int(rng.integers(3, 24))
        W = int(rng.choice([int(rng.integers(3, 24)), 4 * int(rng.integers(1, 8))]))
        N = int(rng.integers(1, 4))
        if (H + 2 * p - d * (k - 1) - 1) < 0 or (W + 2 * p - d * (k - 1) - 1) < 0:
            continue
        out.append((N, G * cin_g, H, W, G * m, G, k, k, s, p, d))
    return out


SHAPES = random_shapes(20261202, 64)


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("mode,name", MODES)
def test_random_shapes_every_path(shape, mode, name):
    c = synth.make_conv("fuzz", *shape, seed=sum(shape) + 77, dist_x=("uniform", -1, 1),
                        dist_w=("normal", 0, 0.5))
    want = want_conv(c, mode)
    for cfg in (None, 1, 2, 4, 5, 6, 7):
        assert_ok = run_conv(c, name, cfg)
        np.testing.assert_array_equal(assert_ok.view(np.uint32), want.view(np.uint32),
                                      err_msg=f"{shape} cfg={cfg}")
