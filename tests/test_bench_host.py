"""Host-side logic of bench.py: operand copies for the calls-in-a-row timing,
kernel source hashes and the recorded DRAM traffic lookup."""
import os

import pytest

import bench

L2 = 129e6


@pytest.mark.parametrize("nbytes", [1e3, 12.9e6, 103e6, 180e6, 206e6, 1e9])
def test_rotation_copies_are_the_fewest_that_evict_l2(nbytes):
    n = bench.rotation_copies(nbytes, L2)
    assert n >= 2
    # between two calls on one copy, the other copies' bytes pass through L2
    assert (n - 1) * nbytes >= 1.5 * L2 or n == 2
    if n > 2:
        assert (n - 2) * nbytes < 1.5 * L2


def test_source_hash_is_stable_and_kernel_specific():
    a = bench.kernel_source_hash("sgemm_tiled_kernel")
    assert a == bench.kernel_source_hash("sgemm_tiled_kernel")
    assert len(a) == 16 and int(a, 16) >= 0
    assert a != bench.kernel_source_hash("gemv_kernel")
    # a kernel not listed hashes every source file
    assert bench.kernel_source_hash("no_such_kernel") == bench.kernel_source_hash()


def test_recorded_traffic_follows_the_source_hash(tmp_path, monkeypatch):
    prof = tmp_path / "profiles"
    prof.mkdir()
    h = bench.kernel_source_hash("gemv_kernel")
    (prof / "dram_traffic.txt").write_text(
        "# kernel workload source_hash bytes\n"
        f"gemv_kernel gemm_decode_fast {h} 180224000\n"
        "gemv_kernel gemm_decode_exact 0000000000000000 180224000\n")
    real_hash = bench.kernel_source_hash
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_source_hash", lambda k="": h if k == "gemv_kernel" else real_hash(k))
    assert bench.recorded_traffic("gemv_kernel", "gemm_decode_fast") == 180224000
    assert bench.recorded_traffic("gemv_kernel", "gemm_decode_exact") is None  # stale capture
    assert bench.recorded_traffic("gemv_kernel", "no_such_workload") is None
    monkeypatch.setattr(bench, "ROOT", os.path.join(str(tmp_path), "missing"))
    assert bench.recorded_traffic("gemv_kernel", "gemm_decode_fast") is None
