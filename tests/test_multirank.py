"""Host logic of the multi-rank benchmark (one process per GPU, independent
replicas), run as two gloo ranks on the CPU: the slowest rank's time is the
job's time, throughput counts the work of every rank, ranks draw distinct
inputs, and only rank 0 runs and prints the reference arm."""
import os
import socket
import subprocess
import sys

import numpy as np
import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        elapsed = [12.5, 20.0][rank]                   # rank 1 is the slow one
        slowest = bench.max_over_ranks(elapsed)
        dist.barrier()
        out[rank] = (slowest, bench.job_tops(2.0 * 4096 * 10240 * 2560, 100, world, slowest))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_time_and_job_throughput():
    world = 2
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_rank_main, args=(world, _free_port(), out), nprocs=world, join=True)
        res = dict(out)
    assert res[0] == res[1]
    slowest, tops = res[0]
    assert slowest == 20.0
    assert tops == pytest.approx(2.0 * 4096 * 10240 * 2560 * 100 * 2 / 20e-3 / 1e12)


def test_single_rank_reduction_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.25) == 3.25
    assert bench.job_tops(1e12, 10, 1, 1000.0) == pytest.approx(10.0)


def test_ranks_draw_distinct_inputs():
    sys.path.insert(0, ROOT)
    import argparse

    import bench
    a = argparse.Namespace(M=4, N=16, K=64)
    x0, w0 = bench.make_host_inputs(a, 0, 2)
    x1, w1 = bench.make_host_inputs(a, 1, 2)
    assert not np.array_equal(x0[0], x1[0]) and not np.array_equal(w0[0], w1[0])
    assert not np.array_equal(x0[0], x0[1])            # rotating sets differ too
    x0b, _ = bench.make_host_inputs(a, 0, 2)
    assert np.array_equal(x0[0], x0b[0])               # and are reproducible


def test_reference_arm_runs_on_rank_zero_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "3", "--warmup", "3", "--M", "8", "--N", "64", "--K", "128"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""


def test_reference_arm_line_on_rank_zero():
    """The reference arm (the oracle on the host cores) prints one JSON line with
    the contract's keys, on the same metric as the GPU arm."""
    import json
    env = dict(os.environ, RANK="0", WORLD_SIZE="1", LOCAL_RANK="0")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "3", "--warmup", "3", "--M", "8", "--N", "64", "--K", "128"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "TOPS" and d["higher_is_better"] is True
    assert d["metric"].startswith("W8A8 linear TOPS") and d["value"] > 0
    assert d["steps"] == 3 and d["warmup"] == 3
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    e = d["e2e"]
    assert e["value"] == d["value"] and e["unit"] == d["unit"]
    assert e["h2d_bytes_per_step"] == 0 and e["d2h_bytes_per_step"] == 0
    assert d["config"]["workload"] == "W8A8 per-channel linear M=8 N=64 K=128"
