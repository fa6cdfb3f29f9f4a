"""The multi-GPU path of the benchmark is replicas only: each rank runs its
own copy of the workload and the ranks exchange nothing but the timing.
This checks that host logic with two gloo ranks on the CPU."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, ms_by_rank, out):
    import sys
    import torch.distributed as dist
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        ms, gflops = bench.combine_ranks(ms_by_rank[rank], 2.0e9, world, dist, "cpu")
        out[rank] = (ms, gflops)
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2])
def test_replicas_take_the_slowest_rank(world):
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    out = manager.dict()
    ms_by_rank = [3.0, 5.0]
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, ms_by_rank, out))
             for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    for r in range(world):
        ms, gflops = out[r]
        assert ms == 5.0
        # two ranks' work (2 GFLOP each) over the slowest rank's 5 ms
        assert abs(gflops - 2 * 2.0e9 / 5e-3 / 1e9) < 1e-6


def test_single_rank_needs_no_process_group():
    import bench
    ms, gflops = bench.combine_ranks(4.0, 2.0e9, 1)
    assert ms == 4.0 and abs(gflops - 500.0) < 1e-9
