"""World-size-2 check (gloo, CPU) of the multi-rank logic of bench.py: every rank times its own
replica, the job's time is the slowest rank's, and the value counts every rank's work."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = [120.0, 150.0][rank]
        dist.barrier()
        total = bench.max_over_ranks(local_ms, dist, "cpu")
        value = bench.whole_job_tflops(world, 1.0e12, 10, total)
        q.put((rank, total, value))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_ranks_take_max_time_and_sum_work():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for rank, total, value in res:
        assert total == 150.0
        assert value == pytest.approx(2 * 1.0e12 * 10 / 0.150 / 1e12)


def test_single_rank_is_identity():
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.whole_job_tflops(1, 2e12, 4, 1000.0) == pytest.approx(8.0)
