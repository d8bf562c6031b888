"""The benchmark's own line on a GPU: a short run of the step workload
prints one JSON line carrying every key of the contract, with the launches
counted, the roofline against the measured copy peak, the end-to-end figure
with its per-step host traffic, and the clocks sampled during the timed
region."""

import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_bench_line_carries_the_contract_keys():
    steps = 201  # one graph of 200 calls plus a graph of the remainder
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--quick", "--no-cpu",
                        "--steps", str(steps), "--warmup", "3"],
                       capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
              "gpu_launches", "e2e", "roofline", "clocks", "eager_us_per_call"):
        assert k in d, k
    assert d["unit"] == "us/call" and d["higher_is_better"] is False
    assert d["n_gpus"] == 1 and d["steps"] == steps and d["warmup"] == 3
    assert d["gpu_launches"] == steps
    assert d["value"] > 0 and abs(d["ms_per_step"] * 1000 - d["value"]) < 1e-2
    assert "workload" in d["config"] and "issue" in d["measurement"]
    e = d["e2e"]
    assert e["value"] > 0 and e["unit"] == d["unit"]
    assert e["h2d_bytes_per_step"] == 8 * 20480 * 2          # every rank's [1, W] shard
    assert e["d2h_bytes_per_step"] == 8 * 8 * 20480 * 2      # every rank's [1, V] row
    assert e["d2h_copy_of_outputs_alone_us"] > 0              # the host link's write rate
    rf = d["roofline"]
    assert rf["bound"] == "hbm" and rf["unit"] == "GB/s" and rf["peak"] > 0
    assert abs(rf["frac"] - rf["achieved"] / rf["peak"]) < 1e-3
    assert abs(rf["achieved"] - 10_813_440 / (d["value"] * 1e-6) / 1e9) < 0.02 * rf["achieved"]
    c = d["clocks"]
    assert "sm_mhz" in c and "sm_max_mhz" in c and "reasons" in c
