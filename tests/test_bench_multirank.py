"""The bench's multi-GPU arithmetic, run as world_size-2 gloo ranks on the CPU:
the attention path has no exchange step, so N GPUs are N independent replicas;
the bench takes the slowest rank's time and counts every rank's work."""
import io
import json
import os
import sys
from contextlib import redirect_stdout

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _worker(rank, world, port, ret):
    sys.path.insert(0, ROOT)
    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = 10.0 + 5.0 * rank  # rank 1 is the slower one
        slowest = bench.max_over_ranks(ms, "cpu")
        ret[rank] = (slowest, bench.whole_job_tflops(world, 1e12, 4, slowest))
    finally:
        dist.destroy_process_group()


def test_slowest_rank_and_whole_job_value_two_gloo_ranks():
    world = 2
    port = 29500 + (os.getpid() % 1000)
    mgr = mp.Manager()
    ret = mgr.dict()
    mp.start_processes(_worker, args=(world, port, ret), nprocs=world, start_method="spawn")
    for r in range(world):
        slowest, tflops = ret[r]
        assert slowest == 15.0
        assert tflops == pytest.approx(2 * 1e12 * 4 / 15e-3 / 1e12)


def test_single_process_value_is_its_own():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks(3.5, "cpu") == 3.5
    assert bench.whole_job_tflops(1, 2e12, 10, 20.0) == pytest.approx(1000.0)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench

    class Args:
        steps, warmup, gpus = 1, 0, 2

    monkeypatch.setenv("RANK", "1")
    buf = io.StringIO()
    with redirect_stdout(buf):
        assert bench.run_reference(Args()) == 0
    assert buf.getvalue() == ""  # no work, no line on the other ranks


def test_reference_arm_line_on_rank_zero(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench

    monkeypatch.setenv("RANK", "0")
    monkeypatch.setattr(bench, "WORKLOAD", dict(bench.WORKLOAD, N=256))  # a small head keeps this quick

    class Args:
        steps, warmup, gpus = 1, 0, 1

    buf = io.StringIO()
    with redirect_stdout(buf):
        assert bench.run_reference(Args()) == 0
    line = json.loads(buf.getvalue())
    assert line["impl"] == "reference" and line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["value"] > 0


def test_window_pair_count_against_the_mask():
    # The sliding-window side measurement counts FLOPs over the visible pairs;
    # the count must equal the number of (i, j) with i - W < j <= i.
    sys.path.insert(0, ROOT)
    import bench

    for N in (1, 5, 64, 130):
        for W in (1, 3, 64, 129, 200):
            brute = sum(1 for i in range(N) for j in range(N) if i - W < j <= i)
            assert bench.window_pairs(N, W) == brute, (N, W)
