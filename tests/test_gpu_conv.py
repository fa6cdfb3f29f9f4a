"""GPU parity of om_conv2d_f32 / om_conv2d_f32_packed against the oracle, bit for bit."""
import numpy as np
import pytest

import implicit_gemm_convolution_gb300 as om
import oracle
from implicit_gemm_convolution_gb300 import synth
from tests.gpu_util import (assert_bits_equal, forced_config, guarded_output, guards_intact, sha,
                            to_dev)

pytestmark = pytest.mark.gpu

MODES = [(oracle.EXACT, "exact"), (oracle.FAST, "fast")]
# naive, implicit GEMM, direct small-group, few-pixel, 1x1 columns, row
# segments, small-group TMA window, default
CFGS = [0, 1, 2, 4, 5, 6, 7, None]


@pytest.fixture(scope="module", autouse=True)
def built():
    om.build()
    om.lib()
    oracle.build()


def run_conv(c: synth.ConvCase, name, cfg=None, packed=False, workspace=None):
    import torch
    x, w = to_dev(c.x), to_dev(c.w)
    OH = oracle.conv_out_dim(c.H, c.KH, c.stride, c.pad, c.pad, c.dil)
    OW = oracle.conv_out_dim(c.W, c.KW, c.stride, c.pad, c.pad, c.dil)
    init = np.zeros((c.N, c.Cout, OH, OW), np.float32)
    init.view(np.uint32)[:] = 0x7FBADBAD
    buf, y = guarded_output(init)
    with forced_config("OM_FORCE_CONV_CFG", cfg):
        if packed:
            wp = om.pack_conv_weights(w, c.G)
            args = (c.N, c.Cin, c.H, c.W, c.Cout, c.G, c.KH, c.KW, c.stride, c.pad, c.dil,
                    x.data_ptr(), wp.data_ptr(), y.data_ptr(), om.MODES[name])
            if workspace is None:
                st = om.lib().om_conv2d_f32_packed(*args, None)
            else:
                st = om.lib().om_conv2d_f32_packed_ws(*args, workspace.data_ptr(), 4096, None)
        else:
            args = (c.N, c.Cin, c.H, c.W, c.Cout, c.G, c.KH, c.KW, c.stride, c.pad, c.dil,
                    x.data_ptr(), w.data_ptr(), y.data_ptr(), om.MODES[name])
            if workspace is None:
                st = om.lib().om_conv2d_f32(*args, None)
            else:
                st = om.lib().om_conv2d_f32_ws(*args, workspace.data_ptr(), 4096, None)
    assert st == 0, om.STATUS_NAMES.get(st, st)
    torch.cuda.synchronize()
    assert om.device_status() == 0
    assert guards_intact(buf), "write outside y"
    return y.cpu().numpy().reshape(init.shape)


def want_conv(c, mode, images=None):
    x = c.x if images is None else c.x[images[0]:images[1]]
    return oracle.conv2d(x, c.w, c.stride, c.pad, c.dil, c.G, mode, oracle.default_threads())


SMALL = [
    # N, Cin, H, W, Cout, G, KH, KW, s, p, d
    (2, 3, 7, 6, 4, 1, 3, 3, 1, 1, 1),
    (1, 4, 9, 9, 6, 2, 3, 2, 2, 1, 2),
    (2, 8, 5, 5, 8, 8, 3, 3, 1, 2, 1),
    (1, 6, 11, 4, 3, 3, 1, 1, 1, 0, 1),
    (3, 2, 4, 9, 5, 1, 2, 3, 3, 0, 1),
    (2, 16, 12, 12, 64, 1, 3, 3, 1, 1, 1),
    (3, 32, 10, 10, 96, 2, 1, 1, 1, 0, 1),
    (2, 40, 13, 11, 70, 1, 3, 3, 2, 1, 1),
    (1, 3, 30, 30, 16, 1, 7, 7, 2, 3, 1),
    (4, 64, 7, 7, 128, 1, 3, 3, 1, 1, 1),
    # 1x1 stride 1 unpadded with pixel counts a multiple of 4 (the input
    # planes are B, copied 16 bytes at a time): ragged channels and columns,
    # images straddling column tiles
    (2, 20, 6, 6, 24, 1, 1, 1, 1, 0, 1),
    (5, 37, 12, 12, 40, 1, 1, 1, 1, 0, 1),
    # 1x1 that must not take that copy: 25 pixels, stride 2
    (2, 33, 5, 5, 8, 1, 1, 1, 1, 0, 1),
    (2, 12, 8, 8, 16, 1, 1, 1, 2, 0, 1),
    # K = 9216 taps: the tap table would not fit in shared memory beside the
    # stages, so the per-element gather runs
    (1, 1024, 6, 5, 8, 1, 3, 3, 1, 1, 1),
    # depthwise and small groups (the direct kernel's shapes): multiplier 1,
    # 2 and 3, a 5x5 dilated kernel, 32 channels per group
    (2, 32, 15, 15, 32, 32, 3, 3, 1, 1, 1),
    (1, 16, 20, 20, 32, 16, 3, 3, 2, 1, 1),
    (2, 24, 9, 9, 72, 24, 5, 5, 1, 2, 2),
    (2, 64, 10, 10, 64, 2, 3, 3, 1, 1, 1),
    # depthwise 3x3 / 5x5 with stride 1 and 2 (the register-run kernel): ragged
    # rows of 8 outputs, paddings 0-2, several row bands in one plane
    (3, 16, 17, 23, 16, 16, 3, 3, 2, 1, 1),
    (2, 24, 19, 13, 24, 24, 5, 5, 1, 2, 1),
    (2, 12, 21, 30, 12, 12, 5, 5, 2, 2, 1),
    (1, 8, 7, 7, 8, 8, 3, 3, 1, 0, 1),
    (1, 4, 300, 260, 4, 4, 3, 3, 1, 1, 1),
    # depthwise with "same" padding, output rows a multiple of 8 (one TMA copy
    # of the band's window): bands of 16 rows on a 112 x 112 plane, stride 2,
    # 5 x 5, and a 16-column plane
    (1, 8, 112, 112, 8, 8, 3, 3, 1, 1, 1),
    (2, 6, 112, 112, 6, 6, 3, 3, 2, 1, 1),
    (2, 4, 40, 40, 4, 4, 5, 5, 1, 2, 1),
    (2, 4, 40, 48, 4, 4, 5, 5, 2, 2, 1),
    (3, 16, 24, 16, 16, 16, 3, 3, 1, 1, 1),
    # rows a multiple of 4 floats (16-byte window copies and stores)
    (2, 8, 20, 32, 8, 8, 5, 5, 2, 2, 1),
    (2, 8, 30, 64, 8, 8, 3, 3, 2, 1, 1),
    # few output pixels, many output channels (the few-pixel kernel with 2 and
    # 4 channels per thread; a 9 x 9 window per channel, so an odd-sized
    # chunk window before the weights)
    (2, 9, 7, 7, 512, 1, 3, 3, 1, 1, 1),
    (4, 9, 7, 7, 512, 1, 3, 3, 1, 1, 1),
    (1, 300, 7, 7, 64, 1, 3, 3, 1, 1, 1),
    (8, 40, 7, 7, 1024, 1, 1, 1, 1, 0, 1),
    # the row-segment kernel's shapes (stride 1; 3x3 padding 1 or 1x1
    # unpadded; 64-channel blocks; output rows of 14, 28, 56 and 112 pixels):
    # a ragged last input-channel stage, two and four channel blocks, two
    # groups, rows spanning 1, 2 and 4 per warp task (and a 3x1 kernel, which
    # it declines)
    (2, 16, 28, 28, 64, 1, 3, 3, 1, 1, 1),
    (3, 37, 28, 28, 128, 1, 3, 3, 1, 1, 1),
    (2, 24, 16, 56, 64, 1, 1, 1, 1, 0, 1),
    (1, 16, 4, 112, 128, 2, 3, 3, 1, 1, 1),
    (2, 8, 30, 28, 64, 1, 3, 1, 1, 0, 1),
    (4, 20, 14, 14, 256, 1, 1, 1, 1, 0, 1),
    (2, 72, 8, 56, 64, 1, 3, 3, 1, 1, 1),
    (2, 37, 8, 56, 64, 1, 1, 1, 1, 0, 1),
    # the small-group TMA window kernel's shapes (input rows a multiple of 4
    # floats): 1, 2, 4, 6, 12 and 16 channels per group (4, 8 and 16 channel
    # slots); 1x1, 3x3, 5x5; stride 2 with dilation 2; paddings 0, 4 and 5
    # (window origins 0, -4 and -8 columns); several bands with a short last
    # one; a 248-pixel output row
    (2, 32, 16, 16, 32, 8, 3, 3, 1, 1, 1),
    (2, 24, 12, 20, 48, 8, 3, 3, 2, 1, 2),
    (1, 64, 20, 24, 64, 4, 3, 3, 1, 1, 1),
    (2, 16, 12, 12, 48, 4, 5, 5, 1, 2, 1),
    (3, 12, 8, 8, 6, 3, 1, 1, 1, 0, 1),
    (2, 8, 9, 16, 4, 4, 3, 3, 2, 0, 1),
    (1, 32, 40, 40, 48, 16, 3, 3, 1, 1, 1),
    (1, 8, 10, 12, 8, 2, 3, 3, 1, 4, 1),
    (1, 6, 7, 8, 6, 3, 3, 3, 2, 5, 2),
    (2, 16, 6, 248, 16, 4, 3, 3, 1, 1, 1),
]


@pytest.mark.parametrize("shape", SMALL)
@pytest.mark.parametrize("cfg", CFGS)
@pytest.mark.parametrize("mode,name", MODES)
def test_small_convs(shape, mode, name, cfg):
    c = synth.make_conv("t", *shape, seed=sum(shape), dist_x=("uniform", -1, 1),
                        dist_w=("normal", 0, 0.5))
    assert_bits_equal(run_conv(c, name, cfg), want_conv(c, mode), f"{shape} {name} cfg={cfg}")


@pytest.mark.parametrize("shape", SMALL[:6])
@pytest.mark.parametrize("mode,name", MODES)
def test_packed_equals_unpacked(shape, mode, name):
    c = synth.make_conv("t", *shape, seed=3 + sum(shape))
    a = run_conv(c, name, None, packed=False)
    b = run_conv(c, name, None, packed=True)
    assert sha(a) == sha(b)
    assert_bits_equal(a, want_conv(c, mode))


@pytest.mark.parametrize("mode,name", MODES)
def test_padding_taps_with_nonfinite_weights(mode, name):
    c = synth.make_conv("t", 2, 4, 6, 6, 4, 1, 3, 3, 1, 1, 1, seed=8)
    c.w[1, 2, 0, 0] = np.inf
    c.w[3, 0, 2, 2] = np.nan
    for cfg in CFGS:
        assert_bits_equal(run_conv(c, name, cfg), want_conv(c, mode), f"nonfinite cfg={cfg}")


@pytest.mark.parametrize("mode,name", MODES)
def test_padding_taps_with_nonfinite_weights_row_kernel(mode, name):
    # a shape the row-segment kernel takes: non-finite weights on taps that
    # meet the zero border the window copy writes
    c = synth.make_conv("t", 2, 8, 14, 28, 64, 1, 3, 3, 1, 1, 1, seed=18)
    c.w[5, 2, 0, 0] = np.inf
    c.w[17, 7, 2, 2] = np.nan
    c.w[63, 0, 1, 0] = -np.inf
    for cfg in (6, None):
        assert_bits_equal(run_conv(c, name, cfg), want_conv(c, mode), f"nonfinite rows cfg={cfg}")


@pytest.mark.parametrize("mode,name", MODES)
def test_grouped_strided_dilated_workload(mode, name):
    c = synth.workload_conv_grouped()
    for cfg in CFGS:
        assert_bits_equal(run_conv(c, name, cfg), want_conv(c, mode), f"grouped cfg={cfg}")


@pytest.mark.parametrize("mode,name", MODES)
def test_conv3x3_workload_sampled_images(mode, name):
    c = synth.workload_conv3x3()
    got = run_conv(c, name)
    for n0 in (0, 31):
        assert_bits_equal(got[n0:n0 + 1], want_conv(c, mode, (n0, n0 + 1)), f"conv3x3 image {n0}")


@pytest.mark.parametrize("mode,name", MODES)
def test_depthwise_workload_sampled_images(mode, name):
    # the benchmark's depthwise line (TMA window ring kernel), first and last image
    c = synth.workload_conv_depthwise()
    got = run_conv(c, name)
    for n0 in (0, 31):
        assert_bits_equal(got[n0:n0 + 1], want_conv(c, mode, (n0, n0 + 1)), f"depthwise image {n0}")


@pytest.mark.parametrize("mode,name", MODES)
def test_late3x3_workload_full_size(mode, name):
    # the benchmark's batch-1 7x7 layer (column kernel), whole output
    c = synth.workload_conv_late3x3()
    assert_bits_equal(run_conv(c, name), want_conv(c, mode), "late 3x3 workload")


@pytest.mark.parametrize("mode,name", MODES)
def test_conv1x1_workload_sampled_images(mode, name):
    c = synth.workload_conv1x1()
    got = run_conv(c, name)
    for n0 in (0, 17):
        assert_bits_equal(got[n0:n0 + 1], want_conv(c, mode, (n0, n0 + 1)), f"conv1x1 image {n0}")


def test_empty_input_channels_give_plus_zero():
    import torch
    x = torch.zeros((2, 0, 5, 5), device="cuda")
    w = torch.zeros((3, 0, 3, 3), device="cuda")
    y = torch.full((2, 3, 5, 5), 7.0, device="cuda")
    st = om.lib().om_conv2d_f32(2, 0, 5, 5, 3, 1, 3, 3, 1, 1, 1, x.data_ptr(), w.data_ptr(),
                                y.data_ptr(), 0, None)
    assert st == 0
    torch.cuda.synchronize()
    assert (y.cpu().numpy().view(np.uint32) == 0).all()


# ---- balanced schedule (om_conv2d_f32_ws): k-block continuation across CTAs
@pytest.mark.parametrize("which", ["conv3x3", "conv1x1", "grouped"])
@pytest.mark.parametrize("mode,name", MODES)
def test_workspace_schedule_is_bit_identical(which, mode, name):
    c = {"conv3x3": synth.workload_conv3x3, "conv1x1": synth.workload_conv1x1,
         "grouped": synth.workload_conv_grouped}[which]()
    ws = om.new_workspace()
    plain = run_conv(c, name, 0)  # the direct kernel
    for cfg in (None, 1):
        assert_bits_equal(run_conv(c, name, cfg, workspace=ws), plain, f"{which} ws cfg={cfg}")
    got = run_conv(c, name, None, packed=True, workspace=ws)
    assert_bits_equal(got, plain, f"{which} packed ws")
    assert_bits_equal(got[:1], want_conv(c, mode, (0, 1)), f"{which} image 0 vs oracle")


@pytest.mark.parametrize("mode,name", MODES)
def test_workspace_odd_geometry(mode, name):
    # ragged columns, K = 81 (not a multiple of 32 or 4: 4-byte weight path), 3 groups
    c = synth.make_conv("t", 20, 27, 33, 31, 96, 3, 3, 3, 1, 1, 1, seed=90,
                        dist_x=("uniform", -1, 1), dist_w=("normal", 0, 0.3))
    ws = om.new_workspace()
    want = want_conv(c, mode)
    for cfg in (None, 1):
        assert_bits_equal(run_conv(c, name, cfg, workspace=ws), want, f"odd ws cfg={cfg}")


@pytest.mark.parametrize("mode,name", MODES)
def test_1x1_input_not_16_byte_aligned(mode, name):
    # the same 1x1 geometry with x starting 4 bytes past a 16-byte boundary
    import torch
    c = synth.make_conv("t", 3, 24, 8, 8, 32, 1, 1, 1, 1, 0, 1, seed=7,
                        dist_x=("uniform", -1, 1), dist_w=("normal", 0, 0.5))
    xbuf = torch.zeros(c.x.size + 4, dtype=torch.float32, device="cuda")
    xbuf[1:1 + c.x.size] = to_dev(c.x).reshape(-1)
    x = xbuf[1:1 + c.x.size]
    assert x.data_ptr() % 16 == 4
    w = to_dev(c.w)
    y = torch.empty((c.N, c.Cout, c.H, c.W), device="cuda")
    st = om.lib().om_conv2d_f32(c.N, c.Cin, c.H, c.W, c.Cout, c.G, 1, 1, 1, 0, 1, x.data_ptr(),
                                w.data_ptr(), y.data_ptr(), om.MODES[name], None)
    assert st == 0
    torch.cuda.synchronize()
    assert_bits_equal(y.cpu().numpy(), want_conv(c, mode), "misaligned 1x1")


# Shapes with enough output pixels that the direct small-group kernel
# (forced as configuration 2) gives each thread 4 (depthwise; 8 channels per
# group) or 2 (4 channels) pixels; by default the TMA window kernel takes the
# grouped ones.
DIRECT_WIDE = [
    (4, 64, 56, 56, 64, 64, 3, 3, 1, 1, 1),
    (4, 128, 48, 48, 256, 64, 3, 3, 1, 1, 1),
    (8, 64, 56, 56, 256, 32, 3, 3, 1, 1, 1),
]


@pytest.mark.parametrize("shape", DIRECT_WIDE)
@pytest.mark.parametrize("cfg", [2, None])
@pytest.mark.parametrize("mode,name", MODES)
def test_direct_kernel_several_pixels_per_thread(shape, mode, name, cfg):
    c = synth.make_conv("t", *shape, seed=sum(shape) + 5, dist_x=("uniform", -1, 1),
                        dist_w=("normal", 0, 0.5))
    assert_bits_equal(run_conv(c, name, cfg), want_conv(c, mode), f"direct {shape} cfg={cfg}")


# Larger shapes of the small-group TMA window kernel: 4 and 8 channel
# slots per thread, 16-channel groups in two blocks of 8, several bands per
# plane, 1x1 / 3x3 / 5x5, stride and dilation 1 or 2.
GROUP_WIDE = [
    (8, 64, 30, 28, 64, 16, 3, 3, 1, 1, 1),
    (32, 64, 40, 40, 64, 8, 3, 3, 2, 1, 1),
    (4, 64, 36, 36, 128, 8, 5, 5, 1, 2, 1),
    (8, 64, 32, 64, 32, 16, 1, 1, 1, 0, 1),
    (4, 64, 36, 36, 128, 8, 3, 3, 1, 2, 2),
    (20, 96, 26, 28, 96, 24, 3, 3, 2, 1, 2),
    (64, 64, 40, 40, 64, 8, 3, 3, 2, 1, 1),
    (16, 128, 32, 64, 128, 16, 1, 1, 1, 0, 1),
    (8, 64, 36, 36, 128, 16, 5, 5, 1, 2, 1),
]


@pytest.mark.parametrize("shape", GROUP_WIDE)
@pytest.mark.parametrize("cfg", [7, None])
@pytest.mark.parametrize("mode,name", MODES)
def test_group_window_kernel_wide_shapes(shape, mode, name, cfg):
    c = synth.make_conv("t", *shape, seed=sum(shape) + 9, dist_x=("uniform", -1, 1),
                        dist_w=("normal", 0, 0.5))
    assert_bits_equal(run_conv(c, name, cfg), want_conv(c, mode), f"group window {shape} cfg={cfg}")


@pytest.mark.parametrize("mode,name", MODES)
def test_group_window_kernel_packed_weights_and_unaligned_input(mode, name):
    # packed weights (rows padded to 4 floats) through the TMA window kernel,
    # and the same layer with x 4 bytes past a 16-byte boundary (the copy
    # kernel takes it): identical bits
    import torch
    c = synth.make_conv("t", 3, 36, 14, 16, 48, 4, 3, 3, 2, 1, 2, seed=21, dist_x=("uniform", -1, 1),
                        dist_w=("normal", 0, 0.5))
    want = want_conv(c, mode)
    assert_bits_equal(run_conv(c, name, None, packed=True), want, "packed, group window")
    xbuf = torch.zeros(c.x.size + 4, dtype=torch.float32, device="cuda")
    xbuf[1:1 + c.x.size] = to_dev(c.x).reshape(-1)
    x = xbuf[1:1 + c.x.size]
    assert x.data_ptr() % 16 == 4
    w = to_dev(c.w)
    y = torch.empty(want.shape, device="cuda")
    st = om.lib().om_conv2d_f32(c.N, c.Cin, c.H, c.W, c.Cout, c.G, c.KH, c.KW, c.stride, c.pad, c.dil,
                                x.data_ptr(), w.data_ptr(), y.data_ptr(), om.MODES[name], None)
    assert st == 0
    torch.cuda.synchronize()
    assert_bits_equal(y.cpu().numpy(), want, "misaligned group layer")


# The small-group TMA window kernel at its box limits: 256 input channels per
# group (the box's channel extent), a 256-column box, a band of one row of
# 248 output pixels, and many bands per plane.
GROUP_LIMITS = [
    (1, 512, 6, 8, 16, 2, 1, 1, 1, 0, 1),
    (1, 8, 5, 252, 8, 2, 1, 1, 1, 0, 1),
    (2, 16, 3, 248, 16, 4, 3, 3, 1, 1, 1),
    (1, 8, 300, 12, 8, 2, 3, 3, 1, 1, 1),
]


@pytest.mark.parametrize("shape", GROUP_LIMITS)
@pytest.mark.parametrize("mode,name", MODES)
def test_group_window_kernel_limits(shape, mode, name):
    c = synth.make_conv("t", *shape, seed=sum(shape) + 31, dist_x=("uniform", -1, 1),
                        dist_w=("normal", 0, 0.5))
    for cfg in (7, None):
        assert_bits_equal(run_conv(c, name, cfg), want_conv(c, mode), f"group limits {shape} cfg={cfg}")
