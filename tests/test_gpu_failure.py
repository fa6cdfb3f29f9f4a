"""Failure detection on the GPU without a fault.

A bounded device-side wait that nothing completes (an mbarrier phase, the
pipelines' wait; a flag nothing sets, the balanced schedule's continuation
wait) must give up after its short limit, record the timeout, and leave the
context usable: om_device_status reports OM_ERR_TIMEOUT once, and the next
product is still bit-exact. With a workspace the timeout is reported to that
workspace's status word alone: a product running at the same time on
another stream with its own workspace sees OM_OK.
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


@pytest.mark.parametrize("which", [0, 1], ids=["mbarrier", "flag"])
def test_timeout_reported_to_its_own_workspace_only(which):
    import torch
    L = om.lib()
    assert om.device_status() == 0
    ws_wait, ws_prod = om.new_workspace(), om.new_workspace()
    s_wait, s_prod = torch.cuda.Stream(), torch.cuda.Stream()
    rng = np.random.default_rng(10 + which)
    # enough output tiles that the product takes the balanced schedule
    m, n, k = 2048, 2560, 300
    A = rng.standard_normal((m, k)).astype(np.float32)
    B = rng.standard_normal((k, n)).astype(np.float32)
    Ad, Bd = to_dev(A), to_dev(B)
    torch.cuda.synchronize()
    st = L.om_selftest_wait_timeout_ws(which, 200, ws_wait.data_ptr(), om.workspace_bytes(),
                                       s_wait.cuda_stream)
    assert st == 0
    outs = []
    with torch.cuda.stream(s_prod):
        for _ in range(3):
            outs.append(om.gemm(Ad, Bd, mode="fast", workspace=ws_prod))
    assert om.workspace_status(ws_prod, s_prod) == 0
    assert om.workspace_status(ws_wait, s_wait) == OM_ERR_TIMEOUT
    assert om.workspace_status(ws_wait, s_wait) == 0  # reported once, then cleared
    assert om.device_status() == 0  # the device-wide words saw nothing
    torch.cuda.synchronize()
    want = oracle.gemm(A[:4], B, oracle.FAST)
    for C in outs:
        assert_bits_equal(C.cpu().numpy()[:4], want, "product beside the timed-out wait")


def test_workspace_status_validation():
    L = om.lib()
    ws = om.new_workspace()
    assert L.om_workspace_status(None, om.workspace_bytes(), None) == 2
    assert L.om_workspace_status(ws.data_ptr(), 16, None) == 1
    assert L.om_workspace_status(ws.data_ptr() + 4, om.workspace_bytes(), None) == 7
    assert L.om_workspace_status(ws.data_ptr(), om.workspace_bytes(), None) == 0
