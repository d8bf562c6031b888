"""Host-side logic of bench.py, without a GPU: the algorithmic-byte formula,
the number of rotating input sets, the output check, the replica arithmetic,
the lookup of the profiled DRAM traffic, the graph split of the timed calls,
and the reference arm's JSON line (the CPU oracle runs without a GPU)."""

import hashlib
import json
import os

import pytest
import torch

import bench

S = -(1 << 31)  # the sentinel word as a signed int32
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_algorithmic_bytes_formula():
    # M * V * 2 * (1 + 4 * TP): shard read, then push, poll, output, re-arm per rank
    assert bench.algorithmic_bytes(8, 20480, 1) == 10_813_440
    assert bench.algorithmic_bytes(8, 20480, 64) == 64 * 10_813_440
    assert bench.algorithmic_bytes(2, 4, 1) == 1 * 8 * 2 * 9


def test_sets_exceed_twice_the_l2():
    for tp, W, M in [(8, 20480, 1), (8, 20480, 8), (2, 4096, 1), (16, 65536, 256)]:
        n = bench.sets_for(tp, W, M)
        per = M * tp * W * 2 * (1 + tp)
        assert n >= 3
        assert n * per >= 2 * bench.L2_BYTES


def test_check_concat_accepts_rewritten_concat_and_rejects_errors():
    tp, M, W = 3, 2, 8
    g = torch.Generator().manual_seed(0)
    shards = torch.randint(-30000, 30000, (tp, M, W), dtype=torch.int16, generator=g)
    shards.view(torch.int32)[0, 0, 1] = S  # a sentinel word in rank 0
    want = torch.cat([shards[r].view(torch.int32) for r in range(tp)], dim=1)
    want = torch.where(want == S, torch.zeros_like(want), want)
    outs = torch.stack([want.view(torch.int16)] * tp)
    bench.check_concat(torch, shards, outs, tp, "ok")
    outs[2].view(torch.int32)[1, 3] ^= 1
    with pytest.raises(SystemExit):
        bench.check_concat(torch, shards, outs, tp, "corrupted")
    outs = torch.stack([torch.cat([shards[r].view(torch.int32) for r in range(tp)], dim=1)
                        .view(torch.int16)] * tp)  # sentinel not rewritten
    with pytest.raises(SystemExit):
        bench.check_concat(torch, shards, outs, tp, "no rewrite")


def test_replica_arithmetic_single_process():
    ms_max, us = bench.replica_us_per_call(None, 4.0, 1000, 1, None)
    assert ms_max == 4.0 and us == pytest.approx(4.0)


def test_traffic_lookup_follows_the_kernel_hash():
    with open(bench.TRAFFIC_FILE) as f:
        d = json.load(f)
    with open(bench.KERNEL_SRC, "rb") as f:
        h = hashlib.sha256(f.read()).hexdigest()[:16]
    got = bench.traffic_from_profile("tp8_w20480_m1")
    if d["kernel_sha256_16"] == h:
        assert got == d["per_launch_dram_bytes"]["tp8_w20480_m1"]
    else:
        assert got is None  # counters of another kernel source are not reported
    assert bench.traffic_from_profile("no_such_workload") is None


def test_graph_split_issues_exactly_the_steps():
    """The timed step's calls are replays of a graph of up to 200 calls plus
    one graph of the remainder: together exactly `steps` calls."""
    for steps in (1, 3, 199, 200, 201, 1000, 1001, 4321):
        n, reps, rem = bench.graph_split(steps)
        assert 1 <= n <= 200 and 0 <= rem < n
        assert n * reps + rem == steps
    assert bench.graph_split(1000) == (200, 5, 0)
    assert bench.graph_split(50) == (50, 1, 0)


def _run_bench(args, env_extra=None):
    import subprocess
    import sys
    env = dict(os.environ)
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        env.pop(k, None)
    env.update(env_extra or {})
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py")] + args, env=env,
                          capture_output=True, text=True, timeout=600)


def test_reference_arm_prints_the_contract_line():
    """The reference arm (the CPU oracle on the step workload) prints one JSON
    line with the contract's keys, on the same config, metric and unit."""
    r = _run_bench(["--impl", "reference", "--steps", "3", "--warmup", "3"])
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    assert d["metric"] == bench.METRIC and d["unit"] == "us/call"
    assert d["higher_is_better"] is False and d["scaling"] == "weak"
    assert d["steps"] == 3 and d["warmup"] == 3 and d["n_gpus"] == 1
    assert d["config"] == bench.workload_config()
    assert d["value"] > 0 and abs(d["ms_per_step"] * 1000 - d["value"]) < 1e-2
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] == 1
    assert d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": "us/call", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}


def test_reference_arm_other_ranks_exit_without_work():
    """Under torchrun only rank 0 runs and prints the reference arm."""
    r = _run_bench(["--impl", "reference", "--gpus", "2", "--steps", "3", "--warmup", "3"],
                   {"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"})
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip() == ""


def test_bench_rejects_too_few_warmup_steps():
    r = _run_bench(["--impl", "reference", "--steps", "3", "--warmup", "2"])
    assert r.returncode != 0 and "warmup" in r.stderr
