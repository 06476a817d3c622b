"""The benchmark's multi-process path on CPU: two gloo ranks run the same barrier and
max-over-ranks reduction that bench.py runs under torchrun, and the whole-job rate divides the
units of every rank by the slowest rank's time.  The reference arm does its work on rank 0
only."""
import argparse
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


def _worker(rank, world, port, times, queue):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier(True)
        ms = bench.max_over_ranks(times[rank], True, torch.device("cpu"))
        bench.barrier(True)
        queue.put((rank, ms, bench.job_rate(3.0e9, world, ms, 1e9)))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time_and_sum_the_units():
    ctx = mp.get_context("spawn")
    queue = ctx.Queue()
    port = _free_port()
    times = [12.5, 20.0]                       # ms per step on rank 0 and rank 1
    procs = [ctx.Process(target=_worker, args=(r, 2, port, times, queue)) for r in range(2)]
    for p in procs:
        p.start()
    got = {}
    try:
        for _ in range(2):
            rank, ms, rate = queue.get(timeout=120)
            got[rank] = (ms, rate)
    finally:
        for p in procs:
            p.join(timeout=60)
            if p.is_alive():
                p.kill()
    assert all(p.exitcode == 0 for p in procs)
    for rank in (0, 1):
        ms, rate = got[rank]
        assert ms == 20.0                      # both ranks see the slowest rank's time
        assert rate == pytest.approx(3.0e9 * 2 / 20.0e-3 / 1e9)


def test_single_process_reduction_is_the_identity():
    assert bench.max_over_ranks(7.25, False, torch.device("cpu")) == 7.25
    assert bench.job_rate(1.0e9, 1, 2.0, 1e9) == pytest.approx(500.0)


def test_reference_arm_does_no_work_off_rank_zero(capsys):
    args = argparse.Namespace(workload=bench.HEADLINE, steps=1, warmup=1)
    assert bench.reference_arm(args, rank=1, world=2) == 0
    assert capsys.readouterr().out == ""
