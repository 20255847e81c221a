"""The bench's N-rank host logic on CPU with two gloo ranks (the path itself has no
exchange: each rank runs its own replica; the ranks only agree on the slowest time)."""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import bench

    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        got = bench.max_over_ranks([1.0 + rank, 10.0 - rank, 0.5 * rank], world, "cpu")
        args = type("A", (), {"steps": 1, "warmup": 0, "cpu_seconds": 0.1})()
        ref_line = bench.run_reference(args, rank) if rank != 0 else "rank0"
        out.put((rank, got, ref_line))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_time():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    results = dict((r, (g, l)) for r, g, l in (out.get(timeout=120) for _ in procs))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert results[0][0] == results[1][0] == [2.0, 10.0, 0.5]
    assert results[1][1] is None  # only rank 0 runs and prints the reference arm


def test_whole_job_rate_counts_every_rank():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.whole_job_rate(1020, 1, 1.0) == pytest.approx(1.02e6)
    assert bench.whole_job_rate(1020, 4, 1.0) == pytest.approx(4.08e6)
    assert bench.max_over_ranks([3.0, 4.0], 1, "cpu") == [3.0, 4.0]


def test_reference_arm_reports_the_steps_it_ran():
    """The reference arm's line states the warm-up and timed steps it actually ran: K
    timed steps of ms_per_step each fit inside the call's own wall time, and the rate
    is the step's tokens over that step time."""
    import time

    sys.path.insert(0, ROOT)
    import bench

    args = type("A", (), {"steps": 2, "warmup": 1, "cpu_seconds": 0.1})()
    t0 = time.perf_counter()
    line = bench.run_reference(args, 0)
    wall = time.perf_counter() - t0
    assert line["impl"] == "reference" and line["steps"] == 2 and line["warmup"] == 1
    assert line["steps"] * line["ms_per_step"] / 1e3 <= wall
    assert line["value"] == pytest.approx(bench.REF_TOKENS / (line["ms_per_step"] / 1e3), rel=1e-2)
    assert set(line["cpu_baseline"]["per_step_ms"]) == set(bench.ORACLE_STEPS)
    assert line["cpu_baseline"]["cores"] == 1 and line["cpu_baseline"]["nproc"] >= 1
