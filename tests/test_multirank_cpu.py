"""bench.py's multi-rank host logic on CPU: two gloo ranks (no GPU, no data-path collective).

Each rank runs its own full workload (independent heads, weak scaling); the job
time is the slowest rank's, and the whole-job rate counts every rank's work.
"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    r, w, lr = bench.dist_env()
    assert (r, w, lr) == (rank, world, rank)
    ms = [10.0, 25.0][rank]  # rank 1 is the slow one
    worst = bench.max_over_ranks(ms, torch.device("cpu"))
    out[rank] = worst
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2])
def test_max_over_ranks_and_aggregate_rate(world):
    import bench
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    mp.start_processes(_rank, args=(world, _free_port(), out), nprocs=world, start_method="spawn")
    assert dict(out) == {0: 25.0, 1: 25.0}
    # whole-job rate: 2 ranks x 1e12 FLOP each in 25 ms -> 80 TFLOP/s
    assert bench.whole_job_rate(1e12, 25.0, world, 1e12) == pytest.approx(80.0)
    assert bench.max_over_ranks(3.0, torch.device("cpu")) == 3.0  # single process: identity
