"""The multi-rank logic of bench.py (replicas only: no data-path collective) on two
gloo ranks on the CPU: every rank reports the slowest rank's time, and the job's
rate counts every rank's tokens."""
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


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    try:
        r, w, _ = bench.dist_env()
        assert (r, w) == (rank, world)
        slowest = bench.max_over_ranks(10.0 + 5.0 * rank)      # rank 1 is the slow one
        dist.barrier()
        out[rank] = slowest
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_slowest_time():
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    port = _free_port()
    mp.start_processes(_worker, args=(2, port, out), nprocs=2, start_method="spawn", join=True)
    assert dict(out) == {0: 15.0, 1: 15.0}


def test_whole_job_rate_counts_every_replica():
    import bench
    # 2 replicas x 4096 tokens x 10 steps in 20 ms (slowest rank)
    assert bench.whole_job_rate(4096, 2, 10, 20.0) == pytest.approx(4096 * 2 * 10 / 0.020)
    assert bench.max_over_ranks(3.5) == 3.5          # not distributed: the value itself
