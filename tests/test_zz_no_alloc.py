"""om_gemm_f32_no_alloc: the product for callers that may not allocate device
memory (framework plugins limited to pre-planned buffers, latency-critical
paths). Its scratch is a static device array inside the library, shared by
all calls, so two calls in a row must each give exactly the bits of the
workspace entry point om_gemm_f32_ws; a leftover flag from the first call
would break the second.

This file sorts last so that a run stopping at the first failure has run
every other test before it.
"""
import ctypes

import numpy as np
import pytest

import implicit_gemm_convolution_gb300 as om
from implicit_gemm_convolution_gb300 import synth

pytestmark = pytest.mark.gpu


def _no_alloc():
    L = om.lib()
    f = L.om_gemm_f32_no_alloc
    i64, vp = ctypes.c_int64, ctypes.c_void_p
    f.restype = ctypes.c_int
    f.argtypes = [i64, i64, i64, vp, i64, vp, i64, vp, i64, ctypes.c_int, vp]
    return f


def _balanced_tiles(m, n, sms):
    """Output tiles of the balanced schedule's 128 x 256 tile; the schedule
    splits k-stages across CTAs only when the tiles exceed the SMs and do not
    fill whole rounds of them."""
    tiles = ((m + 127) // 128) * ((n + 255) // 256)
    return tiles, tiles > sms and tiles % sms != 0


@pytest.mark.parametrize("mode", ["exact", "fast"])
def test_no_alloc_matches_workspace_entry_point_twice(mode):
    import torch
    om.build()
    fn = _no_alloc()
    ws = om.new_workspace()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    # more output tiles than SMs and not whole rounds: the shared flags are used
    shapes = [(1300, 5000, 333), (2048, 2560, 1000)]
    for call, (m, n, k) in enumerate(shapes):
        tiles, split = _balanced_tiles(m, n, sms)
        assert split, f"{m}x{n}: {tiles} tiles on {sms} SMs would not take the balanced schedule"
        case = synth.make_gemm("na", m, n, k, seed=700 + call, dist_a=("normal", 0, 1),
                               dist_b=("normal", 0, 1))
        A = torch.from_numpy(case.A).cuda()
        B = torch.from_numpy(case.B).cuda()
        C_ref = torch.full((m, n), float("nan"), device="cuda")
        C_plain = torch.full((m, n), float("nan"), device="cuda")
        C = torch.full((m, n), float("nan"), device="cuda")
        assert om.gemm_raw(m, n, k, A.data_ptr(), k, B.data_ptr(), n, C_ref.data_ptr(), n, mode,
                           workspace=ws) == 0
        # the plain entry point runs whole tiles only: a fault in the shared
        # balanced schedule could not hide behind it
        assert om.gemm_raw(m, n, k, A.data_ptr(), k, B.data_ptr(), n, C_plain.data_ptr(), n,
                           mode) == 0
        st = fn(m, n, k, A.data_ptr(), k, B.data_ptr(), n, C.data_ptr(), n, om.MODES[mode],
                torch.cuda.current_stream().cuda_stream)
        assert st == 0, om.STATUS_NAMES.get(st, st)
        torch.cuda.synchronize()
        assert om.device_status() == 0
        got = C.cpu().numpy().view(np.uint32)
        for name, ref in (("workspace", C_ref), ("plain", C_plain)):
            want = ref.cpu().numpy().view(np.uint32)
            assert np.array_equal(got, want), \
                f"call {call} vs {name}: {np.count_nonzero(got != want)} outputs differ"


def test_no_alloc_allocates_nothing():
    """After a first call on the device, further calls leave the device's free
    memory unchanged (no allocation, no release)."""
    import torch
    om.build()
    fn = _no_alloc()
    m, n, k = 1300, 5000, 333
    case = synth.make_gemm("na", m, n, k, seed=711, dist_a=("normal", 0, 1), dist_b=("normal", 0, 1))
    A = torch.from_numpy(case.A).cuda()
    B = torch.from_numpy(case.B).cuda()
    C = torch.empty((m, n), device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    assert fn(m, n, k, A.data_ptr(), k, B.data_ptr(), n, C.data_ptr(), n, 0, stream) == 0
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(5):
        assert fn(m, n, k, A.data_ptr(), k, B.data_ptr(), n, C.data_ptr(), n, 1, stream) == 0
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0, f"free device memory changed by {free0 - free1} bytes"
