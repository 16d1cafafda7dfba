"""The benchmark's multi-rank logic on CPU: two gloo ranks on 127.0.0.1.

Each rank runs its own copy of the workload (weak scaling, no data-path
collective); the job's time per step is the slowest rank's, and its throughput
counts every rank's units over that time.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def rank_main(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    assert bench.dist_env() == (rank, rank, world)
    # rank r took 2 + r ms per kernel step and 10 - r ms end to end
    ms, e2e = bench.slowest_rank([2.0 + rank, 10.0 - rank], "cpu")
    out[rank] = (ms, e2e, bench.job_rate(16384, world, ms))
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2])
def test_slowest_rank_and_job_rate(world):
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        mp.start_processes(rank_main, args=(world, free_port(), out), nprocs=world, join=True,
                           start_method="spawn")
        res = dict(out)
    for r in range(world):
        ms, e2e, rate = res[r]
        assert ms == 2.0 + (world - 1) and e2e == 10.0
        assert rate == pytest.approx(world * 16384 / ((2.0 + world - 1) / 1e3))


def test_single_process_is_local():
    import bench
    assert bench.slowest_rank([3.0, 4.0], "cpu") == [3.0, 4.0]
    assert bench.job_rate(1000, 1, 2.0) == pytest.approx(5e5)
