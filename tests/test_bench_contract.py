"""bench.py's output contract, checked on the CPU: the reference arm (the
oracle timed on the host) prints one JSON line with every required key, and
the roofline's algorithmic bytes are the per-unit figures times the units
(rows read and written), pinned here to the two workloads' published byte
counts."""
from __future__ import annotations

import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_the_contract_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--config", "tiny", "--steps", "1", "--warmup", "3"],
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference"
    assert d["steps"] == 1 and d["warmup"] == 3 and d["n_gpus"] == 1
    assert d["value"] > 0 and d["ms_per_step"] > 0 and d["higher_is_better"] is True
    assert d["config"]["workload"] == "tiny"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"]
    assert cb["host"]["nproc"] >= 1 and cb["host"]["model"]
    assert cb["sample"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_algorithmic_bytes_per_launch():
    sys.path.insert(0, ROOT)
    import bench
    from workloads import CONFIGS

    # skewed: T = 131072 tokens of 4096 bf16 channels, P = 514320 (token, rank) rows
    ab = bench.algorithmic_bytes(CONFIGS["skewed"], 514320)
    assert ab["dispatch"] == 131072 * 8192 + 514320 * 8192 == 5_287_051_264
    assert ab["combine"] == ab["dispatch"]
    # decode FP8: 4096 tokens x 7168 channels in, P = 29824 rows of E4M3 codes
    # plus 56 float32 scales out; combine reads P bf16 rows and writes 4096
    ab = bench.algorithmic_bytes(CONFIGS["decode_fp8"], 29824)
    assert ab["dispatch"] == 58_720_256 + 213_778_432 + 6_680_576 == 279_179_264
    assert ab["combine"] == 427_556_864 + 58_720_256 == 486_277_120


def test_whole_job_value_counts_every_replica():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.whole_job_tokens_per_s(131072, 4, 1.6) == pytest.approx(131072 * 4 / 1.6e-3)


def test_traffic_figures_belong_to_the_current_kernels():
    """Every entry of profiles/ncu_traffic.txt is keyed by a hash of its
    kernel's source files: a kernel edited since its capture would make the
    bench report roofline.traffic as null.  This keeps them in step."""
    sys.path.insert(0, ROOT)
    import bench
    for kernel in ("dispatch_kernel", "combine_kernel"):
        for workload in ("skewed", "dsv3_prefill", "mixtral", "decode_fp8",
                         "decode_fp8/ll", "dsv3_prefill/ll"):
            assert bench.load_traffic(kernel, workload) is not None, (kernel, workload)
