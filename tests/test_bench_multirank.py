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


def test_reference_arm_prints_the_contract_line(capsys):
    """Rank 0 of the reference arm times the float64 oracle on a bounded sample of the headline
    workload and prints one JSON line with the arm's metric, unit and direction, its own CPU
    baseline and an end-to-end figure with no host-device copies."""
    import json
    args = argparse.Namespace(workload=bench.HEADLINE, steps=1, warmup=0)
    assert bench.reference_arm(args, rank=0, world=1) == 0
    lines = [l for l in capsys.readouterr().out.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC
    assert d["unit"] == "GB/s" and d["higher_is_better"] is True and d["steps"] == 1
    assert d["value"] > 0 and d["dtype"] == "f64"
    assert d["config"]["workload"] == bench.HEADLINE
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1
    assert d["e2e"] == {"value": d["value"], "unit": "GB/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
