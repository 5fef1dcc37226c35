"""bench.py's JSON line on the GPU: one line, every key the benchmark contract names.

Runs the benchmark with few steps (and the CPU baseline skipped to keep it
short) and checks the line's structure: the headline metric and its units,
the roofline object of the dominant kernel (bound, achieved, peak, fraction,
DRAM traffic or null when a kernel changed since its ncu capture), the
end-to-end number with its copy volumes, the clocks record, the launch count
and the extra workloads.
"""
import json
import os
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def line():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    r = subprocess.run([sys.executable, "bench.py", "--steps", "3", "--warmup", "3", "--skip-cpu",
                        "--fill-seconds", "0"],
                       cwd=ROOT, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout[-2000:]
    return json.loads(lines[0])


def test_headline_keys(line):
    assert line["metric"].startswith("attention fwd+bwd TFLOP/s")
    assert line["unit"] == "TFLOP/s" and line["higher_is_better"] is True
    assert line["n_gpus"] == 1 and line["steps"] == 3 and line["warmup"] >= 3
    assert line["value"] > 0 and line["ms_per_step"] > 0
    assert line["dtype"] == "bf16" and line["data"] == "synthetic"
    assert line["scaling"] == "weak" and line["vs_baseline"] is None
    assert line["config"]["workload"].startswith("vit_l B16 H16 Lq1568 Lk1568 d64")
    assert line["gpu_launches"] == 4 * 3  # fwd + (pre, main, dq) per step
    assert 0 < line["useful_tflops"] < line["value"]


@pytest.mark.parametrize("key", ["roofline", "roofline_fwd"])
def test_roofline_object(line, key):
    roof = line[key]
    assert roof["bound"] == "tensor" and roof["unit"] == "TFLOP/s"
    assert roof["peak"] > 0 and roof["achieved"] > 0
    assert roof["frac"] == pytest.approx(roof["achieved"] / roof["peak"])
    assert "traffic" in roof and (roof["traffic"] is None or roof["traffic"] > 0)


def test_e2e_and_clocks(line):
    e2e = line["e2e"]
    assert e2e["unit"] == "TFLOP/s" and 0 < e2e["value"] <= line["value"]
    assert e2e["h2d_bytes_per_step"] > 0 and e2e["d2h_bytes_per_step"] > 0
    clocks = line["clocks"]
    assert {"sm_mhz", "sm_max_mhz", "reasons"} <= set(clocks)
    assert line["cpu_baseline"] is None  # skipped here; bench.py times it by default


def test_extra_workloads(line):
    for key in ("merge", "cross", "varlen", "gqa", "temporal", "spatial", "fp8", "vit_b",
                "long_video"):
        assert key in line, key
    assert line["merge"]["bound"] == "hbm" and line["merge"]["value"] > 0
    assert line["long_video"]["fwd_bwd_tflops"] > 0 and line["vit_b"]["fwd_bwd_tflops"] > 0
