"""The ResNet-50 convolution list the chain benchmark runs (host only)."""
from implicit_gemm_convolution_gb300 import chain


def test_resnet50_layer_list():
    layers = chain.resnet50_convs()
    shapes = chain.buffer_shapes(layers, 1, 224)
    assert len(layers) == 53
    assert shapes["stem_out"] == (1, 64, 112, 112) and shapes["s1_in"] == (1, 64, 56, 56)
    assert shapes["x3"] == (1, 256, 56, 56) and shapes["x7"] == (1, 512, 28, 28)
    assert shapes["x13"] == (1, 1024, 14, 14) and shapes["x16"] == (1, 2048, 7, 7)
    # about 4.1 G multiply-adds for the convolutions at 224 x 224
    assert 8.0e9 < chain.layer_flops(layers, shapes) < 8.4e9
