"""A convolution chain (ResNet-50's layer pattern, scaled down) through the
fused epilogue, eagerly and replayed from a CUDA graph, against the oracle
run layer by layer: every buffer bit for bit."""
import numpy as np
import pytest

import implicit_gemm_convolution_gb300 as om
import oracle
from implicit_gemm_convolution_gb300 import chain
from tests.gpu_util import assert_bits_equal

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    om.build()
    om.lib()
    oracle.build()


def oracle_chain(layers, inputs, params, mode):
    buf = dict(inputs)
    for L in layers:
        w, b = params[L.name]
        y = oracle.conv2d(buf[L.src], w, L.stride, L.pad, 1, 1, mode, oracle.default_threads())
        buf[L.dst] = oracle.epilogue(y, b, buf[L.residual] if L.residual else None,
                                     oracle.RELU if L.relu else 0)
    return buf


@pytest.mark.parametrize("mode,name", [(oracle.EXACT, "exact"), (oracle.FAST, "fast")])
def test_scaled_resnet_chain_eager_and_graph(mode, name):
    import torch
    layers = chain.resnet50_convs(width_div=8, depth=(2, 1, 2, 1))
    shapes = chain.buffer_shapes(layers, 2, 64)
    params = chain.make_params(layers, seed=3)
    inputs = chain.make_inputs(shapes, seed=3)
    want = oracle_chain(layers, inputs, params, mode)
    ch = chain.ConvChain(layers, 2, 64, name, params=params, inputs=inputs)
    ch.run()
    torch.cuda.synchronize()
    for key in want:
        assert_bits_equal(ch.buf[key].cpu().numpy(), want[key], f"eager {key}")
    for key in want:
        if key not in inputs:
            ch.buf[key].fill_(float("nan"))
    g = ch.capture()
    for key in want:
        if key not in inputs:
            ch.buf[key].fill_(float("nan"))
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    for key in want:
        assert_bits_equal(ch.buf[key].cpu().numpy(), want[key], f"graph {key}")
    assert om.device_status() == 0


@pytest.mark.parametrize("mode,name", [(oracle.EXACT, "exact"), (oracle.FAST, "fast")])
def test_full_resnet50_chain_224_batch1(mode, name):
    """The benchmark's chain at full size (ResNet-50's 53 convolutions,
    224 x 224, batch 1, the benchmark's seeded weights and inputs), eagerly
    and from the CUDA graph the benchmark replays: every activation buffer,
    the last one included, bit for bit against the oracle."""
    import torch
    layers = chain.resnet50_convs()
    shapes = chain.buffer_shapes(layers, 1, 224)
    params = chain.make_params(layers)
    inputs = chain.make_inputs(shapes)
    want = oracle_chain(layers, inputs, params, mode)
    ch = chain.ConvChain(layers, 1, 224, name, params=params, inputs=inputs)
    ch.run()
    torch.cuda.synchronize()
    for key in want:
        assert_bits_equal(ch.buf[key].cpu().numpy(), want[key], f"eager {key}")
    g = ch.capture()
    for key in want:
        if key not in inputs:
            ch.buf[key].fill_(float("nan"))
    g.replay()
    torch.cuda.synchronize()
    for key in want:
        assert_bits_equal(ch.buf[key].cpu().numpy(), want[key], f"graph {key}")
    assert om.device_status() == 0
    last = layers[-1].dst
    assert np.isfinite(want[last]).all() and (want[last] > 0).any()
