"""Failure detection on the GPU without a fault.

A bounded device-side wait that nothing completes (an mbarrier phase, the
pipelines' wait; a flag nothing sets, the balanced schedule's continuation
wait) must give up after its short limit, record the timeout, and leave the
context usable: om_device_status reports OM_ERR_TIMEOUT once, and the next
product is still bit-exact.
"""
import numpy as np
import pytest

import implicit_gemm_convolution_gb300 as om
import oracle
from tests.gpu_util import assert_bits_equal, to_dev

pytestmark = pytest.mark.gpu

OM_ERR_TIMEOUT = 6


@pytest.fixture(scope="module", autouse=True)
def built():
    om.build()
    om.lib()
    oracle.build()


@pytest.mark.parametrize("which", [0, 1], ids=["mbarrier", "flag"])
def test_wait_runs_out_and_context_survives(which):
    import torch
    L = om.lib()
    assert om.device_status() == 0
    assert L.om_selftest_wait_timeout(which, 20, None) == 0
    assert om.device_status() == OM_ERR_TIMEOUT
    assert om.device_status() == 0  # reported once, then cleared
    rng = np.random.default_rng(which)
    A = rng.standard_normal((130, 70)).astype(np.float32)
    B = rng.standard_normal((70, 260)).astype(np.float32)
    for mode, name in ((oracle.EXACT, "exact"), (oracle.FAST, "fast")):
        got = om.gemm(to_dev(A), to_dev(B), mode=name, workspace=om.new_workspace())
        torch.cuda.synchronize()
        assert_bits_equal(got.cpu().numpy(), oracle.gemm(A, B, mode), f"after timeout {name}")
    assert om.device_status() == 0
