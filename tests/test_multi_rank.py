"""The multi-GPU arrangement is replicas only: each rank runs its own
sequences and the ranks meet only to time the job.  These tests run that
host logic as world-size-2 gloo ranks on the CPU."""

import os
import socket
import subprocess
import sys

import pytest

from tests.conftest import ROOT


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import torch.distributed as dist

    sys.path.insert(0, ROOT)
    import bench

    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        mine = 10.0 * rank + 5.0  # per-rank timed total (ms)
        slowest = bench.max_over_ranks(mine, "cpu")
        out[rank] = (slowest, bench.whole_job_rate(100, world, slowest))
    finally:
        dist.destroy_process_group()


def test_replicas_report_the_slowest_rank_and_the_whole_job_rate():
    import torch.multiprocessing as mp

    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    assert out[0] == out[1]
    slowest, rate = out[0]
    assert slowest == 15.0
    assert rate == pytest.approx(2 * 100 / 0.015)


def test_single_process_needs_no_group():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks(3.5, "cpu") == 3.5
    assert bench.whole_job_rate(10, 1, 20.0) == pytest.approx(500.0)


def test_reference_arm_runs_on_rank_zero_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference"], env=env,
                       capture_output=True, text=True, timeout=120)
    assert r.returncode == 0
    assert r.stdout.strip() == ""
