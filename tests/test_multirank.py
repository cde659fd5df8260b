"""bench.py's multi-GPU logic on CPU: every rank runs its own replica, the
job time is the slowest rank's, and the throughput counts every rank's work.
Two gloo ranks stand in for two GPUs (no kernel runs)."""
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


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        own = 1.0 + rank  # rank 1 is slower
        t = bench.max_over_ranks(own, dist, "cpu")
        out[rank] = (t, bench.job_throughput(world, 1e12, 10, t))
    finally:
        dist.destroy_process_group()


def test_two_rank_time_is_max_and_throughput_counts_all_ranks():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    for r in range(2):
        t, v = out[r]
        assert t == 2.0                  # the slower rank's time on every rank
        assert v == pytest.approx(2 * 1e12 * 10 / 2.0 / 1e12)


def test_single_process_passthrough():
    assert bench.max_over_ranks(3.5, None) == 3.5
    assert bench.job_throughput(1, 2e12, 5, 10.0) == pytest.approx(1.0)
