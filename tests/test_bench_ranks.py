"""The multi-rank host logic of bench.py on CPU: two gloo ranks, as torchrun
starts them (127.0.0.1 rendezvous).  Each rank runs its own replica, so the
only exchange is the all-reduce that gives every rank the job's time, the
largest per-rank time; the job's throughput counts every rank's tokens."""

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
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = [3.0, 5.0][rank]   # this rank's own timed region
        t = bench.job_time_ms(torch, ms, dist, torch.device("cpu"))
        out.put((rank, t, bench.job_tokens_per_s(10, 1, 4096, world, t)))
    finally:
        dist.destroy_process_group()


def test_job_time_is_the_largest_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(out.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [g[0] for g in got] == [0, 1]
    for _, t, value in got:
        assert t == 5.0
        assert value == pytest.approx(10 * 4096 * 2 / 5e-3)


def test_single_rank_needs_no_exchange():
    assert bench.job_time_ms(torch, 2.5, None, None) == 2.5
    assert bench.job_tokens_per_s(4, 1, 4096, 1, 2.0) == pytest.approx(4 * 4096 / 2e-3)
