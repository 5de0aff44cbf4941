"""Host-side pieces of the benchmark, on the CPU: clock sampling and its
throttle-reason parsing (against a stand-in nvidia-smi that prints fixed
samples), the traffic record's attachment to the kernels' own sources, the
kernel-source hash ignoring comments, and the launch counts it reports."""
import os
import stat
import sys
import time

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def fake_smi(tmp_path, rows):
    """An executable named nvidia-smi that prints `rows` (CSV, no header), one
    every 50 ms, then waits to be terminated."""
    body = "\n".join(f"echo '{r}'; sleep 0.05" for r in rows)
    path = tmp_path / "nvidia-smi"
    path.write_text(f"#!/bin/sh\n{body}\nexec sleep 30\n")
    path.chmod(path.stat().st_mode | stat.S_IEXEC)
    return str(tmp_path)


def sample(monkeypatch, tmp_path, rows):
    monkeypatch.setenv("PATH", fake_smi(tmp_path, rows) + os.pathsep + os.environ["PATH"])
    c = bench.ClockSampler(0)
    c.mark(True)
    c.start()
    deadline = time.time() + 10
    while len(c.lines) < len(rows) and time.time() < deadline:
        time.sleep(0.05)
    c.mark(False)
    return c.stop()


def test_clock_sampler_median_and_no_reasons(monkeypatch, tmp_path):
    rows = [f"0, {mhz}, 2070, 900.0, 0x0, Not Active, Not Active, Not Active, Not Active"
            for mhz in (2070, 2055, 2070, 2040, 2070)]
    r = sample(monkeypatch, tmp_path, rows)
    assert r["sm_mhz"] == 2070 and r["sm_max_mhz"] == 2070
    assert r["reasons"] == [] and r["samples"] == 5 and r["in_timed_region"]


def test_clock_sampler_reports_throttle_reasons(monkeypatch, tmp_path):
    rows = ["0, 1980, 2070, 1390.0, 0x4, Not Active, Not Active, Not Active, Active",
            "0, 1700, 2070, 1400.0, 0x8, Active, Not Active, Not Active, Active",
            "0, 1900, 2070, 1395.0, 0x4, Not Active, Not Active, Not Active, Active"]
    r = sample(monkeypatch, tmp_path, rows)
    assert r["sm_mhz"] == 1900
    assert r["reasons"] == ["hw_slowdown", "sw_power_cap"]


def test_clock_sampler_without_nvidia_smi(monkeypatch, tmp_path):
    monkeypatch.setenv("PATH", str(tmp_path))
    c = bench.ClockSampler(0)
    c.start()
    assert c.stop() is None


def test_traffic_attaches_to_the_kernels_own_sources(monkeypatch, tmp_path):
    """A traffic record is used only while the hash of the kernel's own
    sources (comments ignored) matches the one it was taken on."""
    import json
    import shutil
    head = "W8A8 per-channel linear M=4096 N=10240 K=2560"
    srcs = ["gemm_pair.cu", "cider_device.cuh"]
    csrc = tmp_path / "w4a8_quantized_linear_gb300" / "csrc"
    csrc.mkdir(parents=True)
    for f in srcs:
        shutil.copy(os.path.join(bench.ROOT, "w4a8_quantized_linear_gb300", "csrc", f), csrc / f)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps({head: {
        "kernel_source_sha": bench.kernel_source_sha(tuple(srcs)), "sources": srcs,
        "dram_bytes_per_launch": 123}}))
    assert bench.ncu_traffic(head) == 123                 # recorded on the current source
    with open(csrc / "gemm_pair.cu", "a") as f:
        f.write("int one_more_line;\n")
    assert bench.ncu_traffic(head) is None                # any source change drops it
    assert bench.ncu_traffic("no such workload") is None


def test_kernel_source_hash_ignores_comments(tmp_path, monkeypatch):
    csrc = tmp_path / "w4a8_quantized_linear_gb300" / "csrc"
    csrc.mkdir(parents=True)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    (csrc / "k.cu").write_text("int f() {  // the answer\n  return 42;\n}\n")
    h1 = bench.kernel_source_sha(("k.cu",))
    (csrc / "k.cu").write_text("// a new comment\n\nint f() {  // the answer, reworded\n  return 42;\n}\n")
    assert bench.kernel_source_sha(("k.cu",)) == h1
    (csrc / "k.cu").write_text("int f() {\n  return 43;\n}\n")
    assert bench.kernel_source_sha(("k.cu",)) != h1


def test_launch_counts_follow_the_dispatch():
    pytest.importorskip("ctypes")
    try:
        from w4a8_quantized_linear_gb300 import library
        library()
    except Exception as e:
        pytest.skip(f"libcider.so not built: {e}")
    assert bench.library_path(4096, 10240, 2560, 0)[1] == 2           # quantize + pair GEMM
    assert bench.library_path(4096, 10240, 2560, 128)[1] == 2         # quantize + per-group GEMM
    assert bench.library_path(1, 10240, 2560, 0)[1] == 1              # fused GEMV
    assert bench.library_path(16, 10240, 2560, 0)[1] == 2             # quantize + GEMV
    assert bench.library_path(16, 2560, 10240, 0)[1] == 3             # + K slices and combine
    assert "pair" in bench.library_path(4096, 10240, 2560, 0)[0]
