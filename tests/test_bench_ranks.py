"""The N > 1 path of bench.py on the CPU (gloo, two ranks).

A batch-1 decode step does not shard, so N GPUs run N independent replicas.
The only exchange is the timing: every rank's time is reduced to the
slowest, and the job's tokens/s is N x steps over that time.  The
reference arm prints on rank 0 only; the other ranks exit without work.
"""
import argparse
import multiprocessing as mp
import os
import socket

import pytest

import bench


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, seconds, steps, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        t = bench.max_over_ranks(seconds[rank], world, "cpu")
        q.put((rank, t, bench.job_throughput(world, steps, t)))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_ranks_take_the_slowest_time_and_sum_the_tokens():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    seconds, steps = [3.0, 5.0], 200
    procs = [ctx.Process(target=_rank, args=(r, 2, port, seconds, steps, q)) for r in range(2)]
    for p in procs:
        p.start()
    try:
        got = sorted(q.get(timeout=120) for _ in procs)
    finally:
        for p in procs:
            p.join(timeout=60)
            if p.is_alive():
                p.kill()
    assert [p.exitcode for p in procs] == [0, 0]
    # both ranks see the slower rank's 5 s; the job decoded 2 x 200 tokens
    assert got == [(0, 5.0, 80.0), (1, 5.0, 80.0)]


def test_one_rank_needs_no_process_group():
    assert bench.max_over_ranks(2.5, 1, "cpu") == 2.5
    assert bench.job_throughput(1, 200, 0.5) == 400.0


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    monkeypatch.setenv("RANK", "1")
    args = argparse.Namespace(gpus=2, steps=1, warmup=0)
    assert bench.run_reference(args) == 0
    assert capsys.readouterr().out == ""
