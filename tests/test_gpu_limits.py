"""Maximum sizes: operands whose offsets do not fit in 32 bits.

Each case puts elements more than 2^31 floats apart (leading dimensions or
image strides), so that any 32-bit index arithmetic in a kernel would read or
write the wrong place. Inputs are drawn on the device by torch's generator;
expected values come from the oracle on small crops copied back from those
same buffers (every output depends only on its own row of A and column of B,
or on its own input window). Several GB per case; skipped when the device
has less than 40 GB free.
"""
import numpy as np
import pytest

import implicit_gemm_convolution_gb300 as om
import oracle
from tests.gpu_util import assert_bits_equal, forced_config

pytestmark = pytest.mark.gpu

SENT = -12345.0


@pytest.fixture(scope="module", autouse=True)
def built():
    import torch
    om.build()
    om.lib()
    oracle.build()
    free, _ = torch.cuda.mem_get_info()
    if free < 40 * (1 << 30):
        pytest.skip("less than 40 GB of device memory free")


def _release():
    import torch
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


@pytest.mark.parametrize("mode,name", [(oracle.EXACT, "exact"), (oracle.FAST, "fast")])
def test_gemm_rows_more_than_2_31_floats_apart(mode, name):
    """A few rows (matrix-vector kernel) with lda = 2^31 + 8."""
    import torch
    m, n, k = 2, 100, 50
    lda = (1 << 31) + 8
    g = torch.Generator(device="cuda").manual_seed(11)
    A = torch.empty((m - 1) * lda + k, dtype=torch.float32, device="cuda")
    A[:k] = torch.rand(k, generator=g, device="cuda") - 0.5
    A[lda:lda + k] = torch.rand(k, generator=g, device="cuda") - 0.5
    B = torch.rand((k, n), generator=g, device="cuda") - 0.5
    C = torch.full((m, n), SENT, device="cuda")
    st = om.gemm_raw(m, n, k, A.data_ptr(), lda, B.data_ptr(), n, C.data_ptr(), n, name)
    assert st == 0, om.STATUS_NAMES.get(st, st)
    a = np.stack([A[:k].cpu().numpy(), A[lda:lda + k].cpu().numpy()])
    want = oracle.gemm(a, B.cpu().numpy(), mode)
    assert_bits_equal(C.cpu().numpy(), want, "lda = 2^31 + 8")
    assert om.device_status() == 0
    del A, B, C
    _release()


@pytest.mark.parametrize("mode,name", [(oracle.EXACT, "exact"), (oracle.FAST, "fast")])
def test_gemm_tiles_with_output_rows_2_31_floats_apart(mode, name):
    """The tiled kernel with ldc = 2^24 + 4: row 129 of C starts past 2^31 floats;
    the padding columns of sampled rows keep their sentinel."""
    import torch
    m, n, k = 130, 20, 32
    ldc = (1 << 24) + 4
    g = torch.Generator(device="cuda").manual_seed(12)
    A = torch.rand((m, k), generator=g, device="cuda") - 0.5
    B = torch.rand((k, n), generator=g, device="cuda") - 0.5
    C = torch.full(((m - 1) * ldc + n + 4,), SENT, device="cuda")
    for cfg in (None, 1, 3):
        with forced_config("OM_FORCE_GEMM_CFG", cfg):
            st = om.gemm_raw(m, n, k, A.data_ptr(), k, B.data_ptr(), n, C.data_ptr(), ldc, name)
        assert st == 0, om.STATUS_NAMES.get(st, st)
        rows = [0, 1, 64, 127, 128, 129]
        got = np.stack([C[r * ldc:r * ldc + n + 4].cpu().numpy() for r in rows])
        want = oracle.gemm(A.cpu().numpy()[rows], B.cpu().numpy(), mode)
        assert_bits_equal(got[:, :n], want, f"ldc = 2^24 + 4 cfg={cfg}")
        assert (got[:, n:] == SENT).all(), "padding column written"
    assert om.device_status() == 0
    del A, B, C
    _release()


@pytest.mark.parametrize("mode,name", [(oracle.EXACT, "exact"), (oracle.FAST, "fast")])
def test_conv_1x1_images_more_than_2_31_floats_apart(mode, name):
    """1x1 convolution over two images of 2 x 32000 x 32000 (x: 4.1e9 floats)."""
    import torch
    N, Cin, H, W, Cout = 2, 2, 32000, 32000, 1
    g = torch.Generator(device="cuda").manual_seed(13)
    x = torch.rand((N, Cin, H, W), generator=g, device="cuda")
    w = torch.rand((Cout, Cin, 1, 1), generator=g, device="cuda") - 0.5
    for cfg in (None, 1):
        with forced_config("OM_FORCE_CONV_CFG", cfg):
            y = om.conv2d(x, w, mode=name)
        for n, r, c in ((0, 0, 0), (1, 31999, 31992), (1, 12345, 6000)):
            crop = x[n:n + 1, :, r:r + 1, c:c + 8].cpu().numpy()
            want = oracle.conv2d(crop, w.cpu().numpy(), 1, 0, 1, 1, mode)
            got = y[n:n + 1, :, r:r + 1, c:c + 8].cpu().numpy()
            assert_bits_equal(got, want, f"1x1 image {n} ({r}, {c}) cfg={cfg}")
        del y
    assert om.device_status() == 0
    del x, w
    _release()


@pytest.mark.parametrize("mode,name", [(oracle.EXACT, "exact"), (oracle.FAST, "fast")])
def test_conv_3x3_input_beyond_2_31_floats(mode, name):
    """3x3 pad-1 convolution over two 40000 x 40000 planes (x: 3.2e9 floats):
    the implicit GEMM takes its per-element gather (the window kernels do not
    take rows this long); interior and corner windows checked."""
    import torch
    N, Cin, H, W, Cout = 2, 1, 40000, 40000, 1
    g = torch.Generator(device="cuda").manual_seed(14)
    x = torch.rand((N, Cin, H, W), generator=g, device="cuda") - 0.5
    w = torch.rand((Cout, Cin, 3, 3), generator=g, device="cuda") - 0.5
    wn = w.cpu().numpy()
    for cfg in (None, 1):
        with forced_config("OM_FORCE_CONV_CFG", cfg):
            y = om.conv2d(x, w, padding=1, mode=name)
        # interior: the crop holds the whole window, no padding needed
        for n, r, c in ((1, 20000, 30000), (1, 39000, 123)):
            crop = x[n:n + 1, :, r - 1:r + 2, c - 1:c + 9].cpu().numpy()
            want = oracle.conv2d(crop, wn, 1, 0, 1, 1, mode)
            assert_bits_equal(y[n:n + 1, :, r:r + 1, c:c + 8].cpu().numpy(), want,
                              f"3x3 interior image {n} ({r}, {c}) cfg={cfg}")
        # top-left corner of the second image: the crop padded like the plane
        crop = x[1:2, :, 0:2, 0:9].cpu().numpy()
        want = oracle.conv2d(crop, wn, 1, 1, 1, 1, mode)[:, :, 0:1, 0:8]
        assert_bits_equal(y[1:2, :, 0:1, 0:8].cpu().numpy(), want, f"3x3 corner cfg={cfg}")
        del y
    assert om.device_status() == 0
    del x, w
    _release()
