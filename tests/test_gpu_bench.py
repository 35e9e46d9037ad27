"""bench.py's GPU arm end to end on the small workload: one JSON line with
every key of the contract (roofline, cpu_baseline, e2e with its copied
bytes, the launch count, clocks), and an end-to-end step through host
buffers that reproduces the device-resident step bit for bit, also with the
plain steps timed as CUDA-graph replays."""
from __future__ import annotations

import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("layout,graph", [("ht", False), ("ll", False), ("ht", True)])
def test_bench_line_on_the_small_workload(ep, layout, graph):
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--config", "tiny", "--steps", "5",
           "--warmup", "3", "--layout", layout] + (["--graph"] if graph else [])
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=900, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "roofline", "e2e", "gpu_launches", "clocks"):
        assert key in d, key
    assert d["n_gpus"] == 1 and d["steps"] == 5 and d["warmup"] == 3
    assert d["value"] > 0 and d["config"]["workload"] == "tiny"
    rf = d["roofline"]
    assert rf["bound"] == "hbm" and rf["unit"] == "GB/s" and rf["peak"] > 0
    assert rf["frac"] == pytest.approx(rf["achieved"] / rf["peak"])
    e2e = d["e2e"]
    T, H, K = 512, 256, 4
    assert e2e["h2d_bytes_per_step"] == T * K * 8 + T * K * 4 + T * H * 2
    assert e2e["d2h_bytes_per_step"] == T * H * 2
    assert e2e["check"] == "out matches the device-resident step"
    assert e2e["link"]["h2d_gbs"] > 0 and e2e["link"]["d2h_gbs"] > 0
    assert 0 < e2e["link_floor_ms"] and e2e["host_enqueue_ms_per_step"] > 0
    # the reported end-to-end step is the median of its timed passes
    assert len(e2e["passes_ms"]) == 3
    assert sorted(e2e["passes_ms"])[1] == pytest.approx(e2e["ms_per_step"], abs=1e-3)
    # one single-launch layout, dispatch and combine per step, in every timed pass
    assert d["passes"]["n"] >= 1 and d["passes"]["steps_each"] == 5
    assert d["passes"]["ms_min"] <= d["ms_per_step"] <= d["passes"]["ms_max"]
    assert d["gpu_launches"] == 3 * d["steps"] * d["passes"]["n"]
    assert "workloads" not in d  # only the default run carries the other workloads
    assert "sm_mhz" in d["clocks"] and "reasons" in d["clocks"]
    # per-kernel times: each kernel alone (roofline), and inside ordinary steps
    # the pages' own accounting, for context: T * H for the dispatch, one copy
    # per dispatched row for the combine
    pc = d["pages_convention"]
    assert pc["dispatch"]["bytes"] == T * H * 2
    assert pc["combine"]["bytes"] == d["config"]["recv_rows"] * H * 2
    assert pc["dispatch"]["per_rank_gbs"] == pytest.approx(pc["dispatch"]["aggregate_gbs"] / 4,
                                                           abs=0.1)
    kt = d["kernel_timing"]
    assert kt["steps"] == 5 and kt["in_step_ms_per_step"] > 0
    parts = sum(kt["in_step"][k + "_ms"] for k in ("layout", "dispatch", "combine"))
    assert parts == pytest.approx(kt["in_step_ms_per_step"], rel=0.02)
    assert all(d["kernels"][k]["ms"] > 0 for k in ("layout", "dispatch", "combine"))
    assert (d["config"].get("step_launch") == "cuda_graph_replay") == graph
    if layout == "ht":
        cb = d["cpu_baseline"]
        assert cb["kind"] == "oracle" and cb["value"] > 0 and cb["cores"] >= 1
        assert cb["host"]["nproc"] >= 1 and cb["host"]["model"]


def test_bench_workloads_block(ep):
    """The block of other workloads that the default run adds to its line,
    here with the decode FP8 workload beside the small one: each entry has
    its step, per-kernel fractions against the same peak, and a clock window."""
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--config", "tiny", "--steps", "5",
           "--warmup", "3", "--no-cpu-baseline", "--workloads", "--workload-list",
           "decode_fp8,tiny"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=900, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-3000:]
    d = json.loads([ln for ln in r.stdout.splitlines() if ln.startswith("{")][0])
    assert list(d["workloads"]) == ["decode_fp8"]
    w = d["workloads"]["decode_fp8"]
    assert w["ms_per_step"] > 0 and w["tokens_per_s"] == pytest.approx(4096 / (w["ms_per_step"] / 1e3))
    for k in ("dispatch", "combine"):
        assert w[k]["frac"] == pytest.approx(w[k]["gbs"] / d["peak_gbs"])
        # DRAM bytes per launch from the captures of the current kernels, near the
        # algorithmic bytes (short by what is still in L2 when the kernel ends)
        assert 0.7 * w[k]["bytes"] < w[k]["traffic"] <= 1.01 * w[k]["bytes"]
    assert w["l2"].startswith("flushed")  # x (58.7 MB) fits in L2
    assert w["clocks"]["samples"] >= 1 and w["dtype"] == "e4m3+bf16"
    assert w["step_launch"] == "eager"  # only a step that fits in L2 replays as a graph


def test_bench_sharded_line_under_torchrun(ep):
    """The sharded form's bench line, one rank (NCCL, world size 1: the
    all-to-all is a copy to itself)."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "1",
           "--master-addr", "127.0.0.1", "--master-port", "29633", os.path.join(ROOT, "bench.py"),
           "--sharded", "--config", "decode_fp8", "--steps", "3", "--warmup", "3"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=900, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-3000:]
    d = json.loads([ln for ln in r.stdout.splitlines() if ln.startswith("{")][0])
    assert d["n_gpus"] == 1 and d["value"] > 0 and d["config"]["parallelism"] == "ep1 sharded"
    assert d["config"]["tokens_per_rank"] == 128 and d["gpu_launches"] > 0
