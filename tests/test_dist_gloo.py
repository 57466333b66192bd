"""The benchmark's multi-rank host logic on CPU ranks (gloo, world size 2).

Each rank times its own batch; the job's time is the slowest rank's, found
with an all-reduce MAX after a barrier, and the whole-job rate counts every
rank's rows.  No GPU and no data-path collective are involved.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import torch.distributed as dist

    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    assert bench.dist_env() == (rank, world, rank)
    bench.barrier(dist)
    mine = 100.0 + 50.0 * rank           # rank 1 is the slow one
    slowest = bench.max_over_ranks(mine, dist)
    ms_step, value = bench.aggregate(16384, world, 10, slowest)
    out[rank] = (slowest, ms_step, value)
    bench.barrier(dist)
    dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_two_gloo_ranks_report_the_slowest_rank():
    world = 2
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_rank_main, args=(world, _free_port(), out), nprocs=world, start_method="spawn", join=True)
    for r in range(world):
        slowest, ms_step, value = out[r]
        assert slowest == 150.0
        assert ms_step == 15.0
        assert value == pytest.approx(16384 * 2 * 10 / 0.150)


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(42.0, None) == 42.0
    assert bench.aggregate(100, 1, 4, 2.0) == (0.5, 100 * 4 / 0.002)
