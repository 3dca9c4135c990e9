"""The N > 1 path of bench.py on CPU: two gloo ranks, each timing its own copy of the
workload; the job's time is the slowest rank's and its throughput counts every rank's work."""
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
    try:
        import bench
        local_ms = [3.0, 5.5][rank]
        t = bench.max_over_ranks(local_ms, "cpu")
        out[rank] = t
        assert bench.dist_env() == (world, rank, 0)
    finally:
        dist.destroy_process_group()


def test_two_rank_max_and_job_throughput():
    world, port = 2, _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        assert out[0] == out[1] == 5.5
    import bench
    # two replicas of 1e12 flops in 5.5 ms each -> 2e12 / 5.5e-3 flops/s
    assert abs(bench.job_throughput(2, 1e12, 5.5) - 2e12 / 5.5e-3 / 1e12) < 1e-9
    assert bench.max_over_ranks(1.25, "cpu") == 1.25  # no process group: the local value
