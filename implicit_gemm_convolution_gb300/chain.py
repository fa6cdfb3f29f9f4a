"""Convolution chains: a network's convolutions back to back, each with the
fused output epilogue, run eagerly through the C ABI or replayed from a CUDA
graph (one graph launch for the whole chain instead of one host call per
layer).

The pages time "the convolution chain" of ResNet-50 at 224 x 224, batch 1
(the matrix-product and convolution kernels page, "Measuring exact against
fast"; the fast-mode convolution page, "Layout of the work"). Their layer list
is not on the pages; `resnet50_convs` writes it from the published
architecture: a 7 x 7 stride-2 stem, then bottleneck blocks (1 x 1 reduce,
3 x 3, 1 x 1 expand, with a 1 x 1 projection on the first block of a stage)
in stages of 3, 4, 6 and 3 blocks with 64, 128, 256 and 512 middle channels,
the stride of a downsampling block on its 3 x 3 convolution (the v1.5
variant). The max pool after the stem is not a convolution and is not run:
stage 1 reads its own input buffer. Each block ends with
relu(conv + bias + shortcut); the other layers with relu(conv + bias); the
projection with conv + bias.

Everything here is argument marshalling and buffer bookkeeping: every layer is
one call of om_conv2d_f32_ex.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np

from . import synth


@dataclass(frozen=True)
class ConvLayer:
    name: str
    src: str                 # activation buffer read
    dst: str                 # activation buffer written
    cin: int
    cout: int
    k: int
    stride: int
    pad: int
    residual: str | None     # buffer added before the activation (same shape as dst)
    relu: bool


def resnet50_convs(width_div: int = 1, depth=(3, 4, 6, 3)) -> list[ConvLayer]:
    """The 53 convolutions of ResNet-50 (v1.5) in execution order; channel
    counts divided by ``width_div`` and stage depths ``depth`` for scaled-down
    test chains."""
    c = lambda v: max(1, v // width_div)
    layers = [ConvLayer("stem", "image", "stem_out", 3, c(64), 7, 2, 3, None, True)]
    cin, src, bi = c(64), "s1_in", 0
    for si, (blocks, mid) in enumerate(zip(depth, (64, 128, 256, 512))):
        for b in range(blocks):
            stride = 2 if (si > 0 and b == 0) else 1
            out = f"x{bi + 1}"
            pre = f"st{si + 1}b{b + 1}"
            layers.append(ConvLayer(f"{pre}_reduce", src, f"{pre}_a", cin, c(mid), 1, 1, 0, None, True))
            layers.append(ConvLayer(f"{pre}_3x3", f"{pre}_a", f"{pre}_b", c(mid), c(mid), 3, stride, 1,
                                    None, True))
            shortcut = src
            if b == 0:
                layers.append(ConvLayer(f"{pre}_proj", src, f"{pre}_p", cin, c(4 * mid), 1, stride, 0,
                                        None, False))
                shortcut = f"{pre}_p"
            layers.append(ConvLayer(f"{pre}_expand", f"{pre}_b", out, c(mid), c(4 * mid), 1, 1, 0,
                                    shortcut, True))
            cin, src, bi = c(4 * mid), out, bi + 1
    return layers


def out_hw(hw: int, k: int, stride: int, pad: int) -> int:
    return (hw + 2 * pad - k) // stride + 1


def buffer_shapes(layers: list[ConvLayer], batch: int, image_hw: int) -> dict[str, tuple]:
    """NCHW shape of every activation buffer. The stage-1 input has the
    shape the stem's max pool would give (stem output halved)."""
    shapes = {"image": (batch, layers[0].cin, image_hw, image_hw)}
    for L in layers:
        if L.src == "s1_in" and "s1_in" not in shapes:
            stem = shapes["stem_out"]
            shapes["s1_in"] = (batch, stem[1], out_hw(stem[2], 3, 2, 1), out_hw(stem[3], 3, 2, 1))
        n, ci, h, w = shapes[L.src]
        assert ci == L.cin, L.name
        shapes[L.dst] = (n, L.cout, out_hw(h, L.k, L.stride, L.pad), out_hw(w, L.k, L.stride, L.pad))
    return shapes


def layer_flops(layers: list[ConvLayer], shapes: dict[str, tuple]) -> float:
    return float(sum(2.0 * math.prod(shapes[L.dst]) * L.cin * L.k * L.k for L in layers))


def make_params(layers: list[ConvLayer], seed: int = 9) -> dict[str, tuple[np.ndarray, np.ndarray]]:
    """Seeded synthetic weights (He init, std sqrt(2 / fan-in)) and biases
    (N(0, 0.01)) per layer."""
    out = {}
    for i, L in enumerate(layers):
        w = synth.normal(seed, 100 + 2 * i, (L.cout, L.cin, L.k, L.k), 0.0,
                         math.sqrt(2.0 / (L.cin * L.k * L.k)))
        b = synth.normal(seed, 101 + 2 * i, (L.cout,), 0.0, 0.01)
        out[L.name] = (w, b)
    return out


def make_inputs(shapes: dict[str, tuple], seed: int = 9) -> dict[str, np.ndarray]:
    """The chain's two external inputs, U[0, 1): the image and the stage-1 input."""
    return {"image": synth.uniform(seed, 1, shapes["image"], 0.0, 1.0),
            "s1_in": synth.uniform(seed, 2, shapes["s1_in"], 0.0, 1.0)}


class ConvChain:
    """Device buffers and the per-layer calls of one chain."""

    def __init__(self, layers: list[ConvLayer], batch: int, image_hw: int, mode: str,
                 params=None, inputs=None, device="cuda"):
        import torch
        from . import conv2d_ex
        self._conv2d_ex = conv2d_ex
        self.layers, self.mode = layers, mode
        self.shapes = buffer_shapes(layers, batch, image_hw)
        params = params if params is not None else make_params(layers)
        inputs = inputs if inputs is not None else make_inputs(self.shapes)
        self.buf = {name: torch.empty(shape, dtype=torch.float32, device=device)
                    for name, shape in self.shapes.items()}
        for name, arr in inputs.items():
            self.buf[name].copy_(torch.from_numpy(arr))
        self.w = {n: torch.from_numpy(w).to(device) for n, (w, _) in params.items()}
        self.b = {n: torch.from_numpy(b).to(device) for n, (_, b) in params.items()}
        self.flops = layer_flops(layers, self.shapes)

    def run(self, stream=None):
        """One pass: every layer once, in order, on ``stream`` (default: the current one)."""
        for L in self.layers:
            self._conv2d_ex(self.buf[L.src], self.w[L.name], stride=L.stride, padding=L.pad,
                            bias=self.b[L.name],
                            residual=self.buf[L.residual] if L.residual else None,
                            activation="relu" if L.relu else None, out=self.buf[L.dst],
                            mode=self.mode, stream=stream)

    def capture(self):
        """A CUDA graph of one pass (captured after one eager warm-up pass)."""
        import torch
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            self.run()
        torch.cuda.current_stream().wait_stream(side)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            self.run()
        return g
