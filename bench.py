"""Benchmark of the vocab-parallel logits gather on one GB300 (or N replicas).

Default workload (one "step" = one hg_gather call over all TP virtual ranks):
the decode gather, TP=8 virtual ranks, shard 20480 bf16 columns (40 KB per
rank-row), V=163840, cap=8, M=1, back-to-back calls on one stream; logits
bf16(N(0, 3^2)) with 0.1 % sentinel words, seed 1. Inputs and outputs rotate
over enough sets that one pass touches more bytes than L2 holds, so every call
reads its shards and writes its outputs cold; the mailboxes are the method's
own persistent state. The timed calls are issued as a serving engine issues a
captured decode step: replays of CUDA graphs of captured calls (the handle
keeps its parity on the device). The same calls issued one by one from Python
are timed too (eager_us_per_call).

Prints one JSON line (rank 0). Besides the step metric it carries:
  eager_us_per_call  the step's calls issued one by one from Python
  per_m        us/call at M = 1..8 (TP8, V=163840, cap 8)
  large_m      us/call, algorithmic GB/s and fraction of the measured HBM peak
               at M = 64, 128, 256 (TP8, V=163840, cap = M)
  roofline     the gather kernel on the step workload
  e2e          the same metric with pinned host buffers, H2D + gather + D2H
  cpu_baseline the CPU oracle on a bounded sample of the step workload
  clocks       SM clocks sampled by nvidia-smi around the timed region

--impl reference times the CPU oracle on the same workload (the reference arm).
--sweep prints one line per point of the bandwidth sweep instead.
Multi-GPU: replicas only (one independent gather per GPU; no collective on
the data path); value = total calls / max-over-ranks time.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "gather µs/call at TP8 V=163840 M=1..8; HBM GB/s and % of peak at large M"
TP, W, CAP, M_STEP = 8, 20480, 8, 1
V = TP * W
SEED = 1
L2_BYTES = 129 * 1024 * 1024
KERNEL_SRC = os.path.join(ROOT, "tp_vocab_logits_gb300", "csrc", "hg_gather_kernel.cu")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "gather_traffic.json")


def algorithmic_bytes(tp: int, W: int, M: int) -> int:
    """Bytes the method must move per call: shard read (M*V*2), push into tp
    mailboxes, poll read, output write and re-arm write (tp*M*V*2 each)."""
    Vv = tp * W
    return M * Vv * 2 * (1 + 4 * tp)


def peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "source": "fallback"}


# --------------------------------------------------------------- distributed --

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def dist_init(world: int, backend: str):
    if world <= 1:
        return None
    import torch.distributed as dist
    if not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return dist


def reduce_max(dist, value: float, device) -> float:
    """Largest value over the ranks (a control-plane reduction of one float)."""
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_us_per_call(dist, ms_local: float, steps: int, world: int, device) -> tuple:
    """Whole-job figure of N independent replicas: (max-over-ranks milliseconds,
    µs per call = that time over all ranks' calls)."""
    ms_max = reduce_max(dist, ms_local, device)
    return ms_max, ms_max * 1000.0 / (steps * world)


def barrier(dist, device=None):
    if dist is not None:
        if device is not None and getattr(device, "type", "cpu") == "cuda":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


# -------------------------------------------------------------------- clocks --

class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 20 ms."""

    FIELDS = ("index,timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, cuda_index: int):
        self.gpu = self._smi_id(cuda_index)
        self.proc = None
        self.path = None
        self.t_start = self.t_stop = None

    @staticmethod
    def _smi_id(cuda_index: int) -> str:
        """nvidia-smi's id of a CUDA device: its UUID (nvidia-smi ignores
        CUDA_VISIBLE_DEVICES, so the CUDA index is not its index)."""
        try:
            import torch
            u = str(torch.cuda.get_device_properties(cuda_index).uuid)
            return u if u.startswith("GPU-") else "GPU-" + u
        except Exception:
            vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
            parts = [p for p in vis.split(",") if p.strip()]
            return parts[cuda_index] if cuda_index < len(parts) else str(cuda_index)

    def start(self):
        fd, self.path = tempfile.mkstemp(prefix="clocks", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, ValueError):
            self.proc = None
        time.sleep(0.3)

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 10:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[2]) for r in rows if num(r[2]) is not None]
        mx = [num(r[3]) for r in rows if num(r[3]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[6 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "samples": len(rows), "reasons": reasons}


# -------------------------------------------------------------------- timing --

def time_calls(torch, fns, steps: int, warmup: int, stream, label: str = "timed") -> float:
    """Milliseconds for `steps` calls (fns rotate), CUDA events on `stream`,
    synchronised on both sides; `warmup` untimed calls first. The timed calls
    sit in an NVTX range named `label` (ncu --nvtx-include "<label>/")."""
    for i in range(warmup):
        fns[i % len(fns)]()
    torch.cuda.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    torch.cuda.nvtx.range_push(label)
    start.record(stream)
    for i in range(steps):
        fns[i % len(fns)]()
    end.record(stream)
    torch.cuda.synchronize()
    torch.cuda.nvtx.range_pop()
    return start.elapsed_time(end)


def make_workload(torch, hg, synth, tp, W, cap, M, sets, device, rows=None, seed=SEED,
                  dist_kind="normal", scale=3.0, sent=0.001, **create_kw):
    h = hg.hg_create(tp, W, cap, rows, **create_kw)
    shards = torch.empty((sets, tp, M, W), dtype=torch.int16, device=device)
    for s in range(sets):
        shards[s] = synth.shards(seed, tp, M, W, dist=dist_kind, scale=scale, sent_frac=sent,
                                 set_index=s % 2000, device=device)
    outs = torch.empty((sets, tp, M, tp * W), dtype=torch.int16, device=device)
    calls = [hg.GatherCall(h, [shards[s, r] for r in range(tp)],
                           [outs[s, d] for d in range(tp)], M) for s in range(sets)]
    return h, shards, outs, calls


def check_concat(torch, shards, outs, tp, what):
    """outs[d] equals the rank-order concat of the shards with the sentinel
    word rewritten to (+0, +0), for every rank d (checked on the device)."""
    want = torch.cat([shards[r].view(torch.int32) for r in range(tp)], dim=1)
    want = torch.where(want == -(1 << 31), torch.zeros_like(want), want)
    for d in range(tp):
        if not torch.equal(outs[d].view(torch.int32), want):
            raise SystemExit(f"bench: {what}: output of rank {d} wrong")


def sets_for(tp, W, M, minimum=3) -> int:
    per = M * tp * W * 2 * (1 + tp)  # shard + output bytes of one set
    return max(minimum, -(-2 * L2_BYTES // per))


def traffic_from_profile(workload_key: str):
    """Per-launch DRAM bytes of the gather kernel from the committed ncu
    summary, if it was taken on the current kernel source (else None)."""
    if not os.path.exists(TRAFFIC_FILE):
        return None
    with open(TRAFFIC_FILE) as f:
        d = json.load(f)
    with open(KERNEL_SRC, "rb") as f:
        h = hashlib.sha256(f.read()).hexdigest()[:16]
    if d.get("kernel_sha256_16") != h:
        return None
    return d.get("per_launch_dram_bytes", {}).get(workload_key)


# ---------------------------------------------------------------- cpu oracle --

def oracle_calls_per_sample(seconds: float):
    """The CPU oracle on config-2 calls for about `seconds`: (us/call, calls)."""
    import numpy as np

    import oracle
    from tp_vocab_logits_gb300 import synth
    oracle.build()
    g = oracle.Gather(TP, W, CAP)
    sets = [synth.shards(SEED, TP, M_STEP, W, scale=3.0, sent_frac=0.001, set_index=i)
            .numpy().view(np.uint16) for i in range(3)]
    n = 0
    t0 = time.perf_counter()
    while True:
        g.call(sets[n % 3])
        n += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            break
    return el / n * 1e6, n


def _oracle_worker(seconds: float):
    """One process of the all-cores oracle timing: (calls, seconds)."""
    us, n = oracle_calls_per_sample(seconds)
    return n, us * n / 1e6


def oracle_all_cores(seconds: float):
    """The same single-threaded oracle in one independent process per host core
    (spawned: the parent holds a CUDA context), each running config-2 calls for
    about `seconds`: aggregate (us/call, calls, cores)."""
    import multiprocessing as mp
    cores = os.cpu_count() or 1
    with mp.get_context("spawn").Pool(cores) as pool:
        res = pool.map(_oracle_worker, [seconds] * cores)
    calls = sum(n for n, _ in res)
    wall = max(t for _, t in res)
    return wall / calls * 1e6, calls, cores


def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    import numpy as np

    import oracle
    from tp_vocab_logits_gb300 import synth
    oracle.build()
    g = oracle.Gather(TP, W, CAP)
    sets = [synth.shards(SEED, TP, M_STEP, W, scale=3.0, sent_frac=0.001, set_index=i)
            .numpy().view(np.uint16) for i in range(3)]
    for i in range(args.warmup):
        g.call(sets[i % 3])
    t0 = time.perf_counter()
    for i in range(args.steps):
        g.call(sets[i % 3])
    el = time.perf_counter() - t0
    us = el / args.steps * 1e6
    line = {
        "impl": "reference", "metric": METRIC, "value": round(us, 3), "unit": "us/call",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(us / 1000, 6), "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": "int32", "data": "synthetic",
        "config": workload_config(),
        "cpu_baseline": {"value": round(us, 3), "unit": "us/call", "cores": 1, "kind": "oracle",
                         "sample": f"{args.steps} full config-2 calls (TP8, V=163840, M=1) "
                                   f"through the single-threaded C++ oracle"},
        "e2e": {"value": round(us, 3), "unit": "us/call", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def workload_config(extra=None) -> dict:
    c = {"workload": "decode logits gather, TP=8 virtual ranks on one GPU, shard 20480 bf16 "
                     "(40 KB per rank-row), V=163840, cap=8, M=1, back-to-back calls on one "
                     "stream; bf16(N(0,9)) logits with 0.1% sentinel words, seed 1",
         "tp": TP, "shard_cols": W, "V": V, "M": M_STEP, "cap": CAP, "parallelism": "replicas"}
    if extra:
        c.update(extra)
    return c


def graph_replay_us(torch, hg, synth, tp, W, cap, M, device, stream, calls, rows=None,
                    seed=SEED, autotune=False, with_shape=False):
    """us per call of `calls` gathers issued by replaying one CUDA graph of 200
    captured calls (device-resident parity; no host work per call)."""
    n = sets_for(tp, W, M)
    h, sg, og_, cg = make_workload(torch, hg, synth, tp, W, cap, M, n, device, rows=rows,
                                   seed=seed, device_parity=True, autotune=autotune)
    cg[0]()
    torch.cuda.synchronize()
    gs = torch.cuda.Stream()
    gs.wait_stream(torch.cuda.current_stream())
    n_graph = 200
    with torch.cuda.stream(gs):
        calls_g = [hg.GatherCall(h, [sg[i % n, r] for r in range(tp)],
                                 [og_[i % n, d] for d in range(tp)], M, stream=gs)
                   for i in range(n_graph)]
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=gs):
        for c in calls_g:
            c()
    torch.cuda.synchronize()
    reps = max(1, calls // n_graph)
    gms = time_calls(torch, [graph.replay], reps, 3, stream, "timed_graph")
    hg.hg_sync(h)
    us = round(gms * 1000.0 / (reps * n_graph), 3)
    shape = hg.hg_launch_shape(h, M)
    del graph
    h.close()
    del sg, og_, cg, calls_g
    return (us, shape) if with_shape else us


def graph_us_per_launch(torch, issue, stream, n_graph=200, reps=5, label="timed_graph"):
    """us per launch of `issue()` (which enqueues one launch on the current
    stream), captured n_graph times into one CUDA graph and replayed reps
    times back to back after 3 untimed replays."""
    gs = torch.cuda.Stream()
    gs.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=gs):
        for _ in range(n_graph):
            issue()
    torch.cuda.synchronize()
    ms = time_calls(torch, [graph.replay], reps, 3, stream, label)
    del graph
    return round(ms * 1000.0 / (reps * n_graph), 3)


def l2_copy_gbs(torch, device, stream, mib: int = 24, reps: int = 200) -> float:
    """Bandwidth of a device copy whose source and destination (2 x `mib` MiB)
    stay resident in L2, read + write bytes over CUDA-event time: the rate the
    decode-size gather's L2-resident traffic could reach at best."""
    n = mib * 2**20 // 2
    a = torch.ones(n, dtype=torch.int16, device=device)
    b = torch.empty_like(a)
    ms = time_calls(torch, [lambda: b.copy_(a)], reps, 20, stream, "timed_l2_copy")
    del a, b
    return round(2 * n * 2 * reps / (ms * 1e-3) / 1e9, 1)


def latency_floors(torch, hg, shapes, stream, device) -> dict:
    """The two floor kernels of hg_probe at each launch shape {key: (ctas,
    threads)}: an empty dependent launch, and the one-vector push -> poll ->
    copy -> re-arm handoff; us per launch, replayed from CUDA graphs."""
    res = {}
    for key, (ctas, threads) in shapes.items():
        scratch = torch.zeros(hg.hg_probe_scratch_bytes(ctas, threads) // 4 + 4,
                              dtype=torch.int32, device=device)
        hg.hg_probe(2, ctas, threads, scratch)
        hg.hg_probe(1, ctas, threads, scratch)
        hg.hg_probe(0, ctas, threads)
        torch.cuda.synchronize()
        empty = graph_us_per_launch(torch, lambda: hg.hg_probe(0, ctas, threads), stream,
                                    label="timed_floor_empty")
        hand = graph_us_per_launch(torch, lambda: hg.hg_probe(1, ctas, threads, scratch),
                                   stream, label="timed_floor_handoff")
        torch.cuda.synchronize()
        n = ctas * threads
        if int(scratch[8 * n].item()) != 0:
            raise SystemExit(f"bench: handoff floor kernel timed out ({key})")
        res[key] = {"ctas": ctas, "threads": threads, "empty_launch_us": empty,
                    "handoff_us": hand}
        del scratch
    return res


def graph_split(steps: int, per_graph: int = 200) -> tuple:
    """How `steps` calls are issued as CUDA graphs: (calls per full graph,
    replays of it, calls in one trailing graph (0: none))."""
    n = min(steps, per_graph)
    return n, steps // n, steps % n


class GraphSteps:
    """Exactly `steps` gather calls, captured into CUDA graphs (a graph of up to
    200 calls replayed back to back, plus one graph of the remainder). Call i
    of a graph uses input/output set i % nsets. The handle must keep its parity
    on the device, so that captured calls flip it as they run."""

    def __init__(self, torch, hg, h, shards, outs, M, nsets, steps):
        self.n, self.reps, rem = graph_split(steps)
        self.sets_used = min(nsets, self.n)
        gs = torch.cuda.Stream()
        gs.wait_stream(torch.cuda.current_stream())

        def capture(n):
            with torch.cuda.stream(gs):
                cs = [hg.GatherCall(h, [shards[i % nsets, r] for r in range(TP)],
                                    [outs[i % nsets, d] for d in range(TP)], M, stream=gs)
                      for i in range(n)]
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=gs):
                for c in cs:
                    c()
            return g

        self.full = capture(self.n)
        self.tail = capture(rem) if rem else None
        torch.cuda.synchronize()

    def replays(self) -> list:
        """One replay per list entry; together they issue exactly `steps` calls."""
        return [self.full.replay] * self.reps + ([self.tail.replay] if self.tail else [])


def stats_graph_us(torch, hg, synth, M, device, stream, calls=1000) -> dict:
    """hg_gather_stats at TP8, V=163840, M rows, replayed from CUDA graphs of
    200 captured calls (device parity), beside the plain gather timed the same
    way on the same buffers: us per call of each."""
    import ctypes
    n = sets_for(TP, W, M)
    h, sh, ou, cg = make_workload(torch, hg, synth, TP, W, CAP, M, n, device, rows=[M],
                                  seed=2, device_parity=True)
    st = hg.new_row_stats(M)
    lib = hg.load()
    arrs = [((ctypes.c_void_p * TP)(*[sh[s_, r].data_ptr() for r in range(TP)]),
             (ctypes.c_void_p * TP)(*[ou[s_, d].data_ptr() for d in range(TP)]))
            for s_ in range(n)]
    k = [0]

    def issue_stats():
        a_ = arrs[k[0] % n]
        k[0] += 1
        rc = lib.hg_gather_stats(h.ptr, a_[0], a_[1], M, st.data_ptr(),
                                 torch.cuda.current_stream().cuda_stream)
        if rc != 0:
            raise SystemExit(f"hg_gather_stats failed: {hg.strerror(rc)}")

    def issue_plain():
        a_ = arrs[k[0] % n]
        k[0] += 1
        rc = lib.hg_gather(h.ptr, a_[0], a_[1], M, torch.cuda.current_stream().cuda_stream)
        if rc != 0:
            raise SystemExit(f"hg_gather failed: {hg.strerror(rc)}")
    issue_stats()
    hg.hg_sync(h)
    reps = max(1, calls // 200)
    us_s = graph_us_per_launch(torch, issue_stats, stream, reps=reps, label="timed_stats_graph")
    us_p = graph_us_per_launch(torch, issue_plain, stream, reps=reps, label="timed_plain_graph")
    hg.hg_sync(h)
    check_concat(torch, sh[0], ou[0], TP, f"stats graph M={M}")
    h.close()
    return {"stats_us": us_s, "plain_us": us_p, "stats_minus_plain_us": round(us_s - us_p, 3)}


# The drafter's gather beside the target's (one stream, one decode step = the
# drafter's gather of its draft block, then the target's gather of the token
# before it plus the drafted ones): the pages give the drafter no shape; this
# reads it as the target's tokenizer and TP group with a block of 4 drafted
# positions.
DRAFT_M, TARGET_M = 4, 5


def drafter_pair(torch, hg, synth, device, stream, warmup, steps=1000) -> dict:
    """us per decode step of the drafter's gather (TP8, V=163840, M=4) and the
    target's (M=5) issued back to back on one stream, replayed from CUDA
    graphs of 100 steps and issued one by one from Python, beside each
    handle's calls alone (graph-replayed)."""
    nd = sets_for(TP, W, DRAFT_M)
    nt = sets_for(TP, W, TARGET_M)
    hd, sd, od, cd = make_workload(torch, hg, synth, TP, W, 4, DRAFT_M, nd, device,
                                   rows=[1, 2, 3, 4], seed=31, device_parity=True)
    ht, st_, ot, ct = make_workload(torch, hg, synth, TP, W, 8, TARGET_M, nt, device,
                                    rows=[1, 2, 3, 4, 5, 8], seed=32, device_parity=True)
    cd[0]()
    ct[0]()
    hg.hg_sync(hd)
    hg.hg_sync(ht)
    gs = torch.cuda.Stream()
    gs.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(gs):
        pair_calls = []
        for i in range(100):
            pair_calls.append(hg.GatherCall(hd, [sd[i % nd, r] for r in range(TP)],
                                            [od[i % nd, d] for d in range(TP)], DRAFT_M, stream=gs))
            pair_calls.append(hg.GatherCall(ht, [st_[i % nt, r] for r in range(TP)],
                                            [ot[i % nt, d] for d in range(TP)], TARGET_M,
                                            stream=gs))
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=gs):
        for c in pair_calls:
            c()
    torch.cuda.synchronize()
    reps = steps // 100
    ms = time_calls(torch, [graph.replay], reps, 3, stream, "timed_drafter_pair")
    hg.hg_sync(hd)
    hg.hg_sync(ht)
    for s_ in range(min(nd, 100)):
        check_concat(torch, sd[s_], od[s_], TP, f"drafter set {s_}")
    for s_ in range(min(nt, 100)):
        check_concat(torch, st_[s_], ot[s_], TP, f"target set {s_}")
    pair_graph = round(ms * 1000.0 / (reps * 100), 3)
    del graph, pair_calls
    # the same steps issued one by one from Python (direct-call objects)
    fns = []
    for i in range(max(nd, nt)):
        fns.append(cd[i % nd])
        fns.append(ct[i % nt])
    ms_e = time_calls(torch, fns, 2 * steps, 2 * warmup, stream, "timed_drafter_pair_eager")
    hg.hg_sync(hd)
    hg.hg_sync(ht)
    pair_eager = round(ms_e * 1000.0 / steps, 3)
    # each handle alone, replayed from graphs
    alone = {}
    for name, h, sh_, ou_, n_, M in (("drafter", hd, sd, od, nd, DRAFT_M),
                                     ("target", ht, st_, ot, nt, TARGET_M)):
        k = [0]

        def issue(h=h, sh_=sh_, ou_=ou_, n_=n_, M=M, k=k):
            # on the current stream: the capture stream while the graph is taken
            i = k[0] % n_
            k[0] += 1
            hg.hg_gather(h, [sh_[i, r] for r in range(TP)], [ou_[i, d] for d in range(TP)], M)
        alone[name] = graph_us_per_launch(torch, issue, stream, label=f"timed_{name}_alone")
        hg.hg_sync(h)
    hd.close()
    ht.close()
    return {"drafter": {"tp": TP, "shard_cols": W, "rows": [1, 2, 3, 4], "M": DRAFT_M},
            "target": {"tp": TP, "shard_cols": W, "rows": [1, 2, 3, 4, 5, 8], "M": TARGET_M},
            "pair_us_per_step_graph_replay": pair_graph,
            "pair_us_per_step_eager": pair_eager,
            "drafter_alone_us": alone["drafter"], "target_alone_us": alone["target"],
            "sum_alone_us": round(alone["drafter"] + alone["target"], 3)}


# --------------------------------------------------------------------- ours --

def run_ours(args):
    import torch

    from tp_vocab_logits_gb300 import _build, hg, synth

    world, rank, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    dist = dist_init(world, "nccl")
    if rank == 0:
        _build.build()
    barrier(dist, device)
    hg.load()
    stream = torch.cuda.current_stream()
    pk = peaks()

    # ---- step workload: config 2 ----
    tune = args.autotune  # launch shapes timed on the device at hg_create
    nsets = sets_for(TP, W, M_STEP)
    h, shards, outs, calls = make_workload(torch, hg, synth, TP, W, CAP, M_STEP, nsets, device,
                                           autotune=tune)
    shape = hg.hg_launch_shape(h, M_STEP)
    # correctness of the timed configuration, untimed: every set once
    for c in calls:
        c()
    hg.hg_sync(h)
    for s in range(nsets):
        want = torch.cat([shards[s, r].view(torch.int32) for r in range(TP)], dim=1)
        want = torch.where(want == -(1 << 31), torch.zeros_like(want), want)
        for d in range(TP):
            if not torch.equal(outs[s, d].view(torch.int32), want):
                raise SystemExit(f"bench: gather output wrong (set {s}, rank {d})")

    # The timed step, issued as a serving engine issues its captured decode
    # step: the same calls on the same buffers, captured into CUDA graphs on a
    # handle whose parity lives on the device, replayed back to back.
    hgr = hg.hg_create(TP, W, CAP, None, device_parity=True, autotune=tune)
    hg.GatherCall(hgr, [shards[0, r] for r in range(TP)], [outs[0, d] for d in range(TP)],
                  M_STEP)()
    hg.hg_sync(hgr)
    steps_g = GraphSteps(torch, hg, hgr, shards, outs, M_STEP, nsets, args.steps)
    replays = steps_g.replays()

    sampler = ClockSampler(local) if rank == 0 else None
    if sampler:
        sampler.start()
    barrier(dist, device)
    for _ in range(-(-args.warmup // steps_g.n)):
        steps_g.full.replay()
    torch.cuda.synchronize()
    barrier(dist, device)
    torch.cuda.synchronize()
    ms = time_calls(torch, replays, len(replays), 0, stream, "timed_step")
    hg.hg_sync(hgr)
    # keep the same load for a moment so that the clock samples cover it
    t_end = time.perf_counter() + 0.3
    while time.perf_counter() < t_end:
        steps_g.full.replay()
        torch.cuda.synchronize()
    clocks = sampler.stop() if sampler else None
    hg.hg_sync(hgr)
    # every set the graphs wrote holds its last call's gather (untimed check)
    for s in range(steps_g.sets_used):
        check_concat(torch, shards[s], outs[s], TP, f"graph-replayed step, set {s}")
    ms_max, us_call = replica_us_per_call(dist, ms, args.steps, world, device)
    us_launch = ms * 1000.0 / args.steps  # this rank's average launch duration
    del steps_g, replays
    hgr.close()

    # the same calls issued one by one from Python through the binding's
    # direct-call object (host parity)
    for i in range(args.warmup):
        calls[i % nsets]()
    torch.cuda.synchronize()
    ms_e = time_calls(torch, calls, args.steps, 0, stream, "timed_eager")
    hg.hg_sync(h)
    _, eager_us = replica_us_per_call(dist, ms_e, args.steps, world, device)

    # ---- the same workload with row statistics, and with device parity ----
    stats_us = devpar_us = torch_stats_us = None
    if not args.quick:
        import ctypes
        st_buf = hg.new_row_stats(M_STEP)
        lib = hg.load()
        sp_ = stream.cuda_stream
        arrs = [((ctypes.c_void_p * TP)(*[shards[s_, r].data_ptr() for r in range(TP)]),
                 (ctypes.c_void_p * TP)(*[outs[s_, d].data_ptr() for d in range(TP)]))
                for s_ in range(nsets)]
        stp = st_buf.data_ptr()
        fns = [lambda a_=a_: lib.hg_gather_stats(h.ptr, a_[0], a_[1], M_STEP, stp, sp_)
               for a_ in arrs]
        t = time_calls(torch, fns, args.steps, args.warmup, stream, "timed_stats")
        hg.hg_sync(h)
        stats_us = round(t * 1000.0 / args.steps, 3)

        def gather_then_torch(i=[0]):  # the unfused alternative
            calls[i[0] % nsets]()
            row = outs[i[0] % nsets, 0].view(torch.bfloat16).float()
            torch.max(row, dim=1)
            torch.logsumexp(row, dim=1)
            i[0] += 1
        t = time_calls(torch, [gather_then_torch], 200, args.warmup, stream, "timed_torch_stats")
        hg.hg_sync(h)
        torch_stats_us = round(t * 1000.0 / 200, 3)
        hdp, sdp, odp, cdp = make_workload(torch, hg, synth, TP, W, CAP, M_STEP, nsets, device,
                                           device_parity=True, autotune=tune)
        t = time_calls(torch, cdp, args.steps, args.warmup, stream, "timed_devparity")
        hg.hg_sync(hdp)
        devpar_us = round(t * 1000.0 / args.steps, 3)
        hdp.close()
        del sdp, odp, cdp

    # ---- the same calls captured in a CUDA graph (device-resident parity) ----
    graph_us = None
    if not args.quick:
        graph_us = graph_replay_us(torch, hg, synth, TP, W, CAP, M_STEP, device, stream,
                                   args.steps, autotune=tune)

    # ---- row statistics replayed from CUDA graphs, as the plain gather ----
    stats_graph = {}
    if not args.quick:
        for M in (1, 4, 8):
            stats_graph[str(M)] = stats_graph_us(torch, hg, synth, M, device, stream)

    # ---- the drafter's gather beside the target's, on one stream ----
    drafter = None
    if not args.quick:
        drafter = drafter_pair(torch, hg, synth, device, stream, args.warmup)

    # ---- e2e: pinned host buffers through hg_gather_host (the kernel reads the
    # shards from host memory and writes the outputs into host memory over the
    # host-device link), rotating over as many sets as the device workload ----
    host_in = torch.empty((nsets, TP, M_STEP, W), dtype=torch.int16).pin_memory()
    host_in.copy_(shards.cpu())
    host_out = torch.empty((nsets, TP, M_STEP, V), dtype=torch.int16).pin_memory()
    e2e_calls = [hg.GatherCall(h, [host_in[s_, r] for r in range(TP)],
                               [host_out[s_, d] for d in range(TP)], M_STEP)
                 for s_ in range(nsets)]
    e2e_ms = time_calls(torch, e2e_calls, args.steps, args.warmup, stream, "timed_e2e")
    hg.hg_sync(h)
    used = min(nsets, max(args.steps, args.warmup))  # sets the calls above wrote
    for s_ in range(used):
        want = torch.cat([host_in[s_, r].view(torch.int32) for r in range(TP)], dim=1)
        want = torch.where(want == -(1 << 31), torch.zeros_like(want), want)
        for d in range(TP):
            if not torch.equal(host_out[s_, d].view(torch.int32), want):
                raise SystemExit(f"bench: e2e output wrong (set {s_}, rank {d})")
    del e2e_calls, host_out

    # the same with one copy of the result read back: rank 0's output in pinned
    # host memory, ranks 1..TP-1 on the device (every rank's output is the same)
    host_out0 = torch.empty((nsets, M_STEP, V), dtype=torch.int16).pin_memory()
    dev_rest = torch.empty((TP - 1, M_STEP, V), dtype=torch.int16, device=device)
    one_calls = [hg.GatherCall(h, [host_in[s_, r] for r in range(TP)],
                               [host_out0[s_]] + [dev_rest[d] for d in range(TP - 1)], M_STEP)
                 for s_ in range(nsets)]
    one_ms = time_calls(torch, one_calls, args.steps, args.warmup, stream, "timed_e2e_one")
    hg.hg_sync(h)
    for s_ in range(used):
        want = torch.cat([host_in[s_, r].view(torch.int32) for r in range(TP)], dim=1)
        want = torch.where(want == -(1 << 31), torch.zeros_like(want), want)
        if not torch.equal(host_out0[s_].view(torch.int32), want):
            raise SystemExit(f"bench: e2e (one copy) output wrong (set {s_})")
    one_us = round(one_ms * 1000.0 / args.steps, 3)
    del one_calls, host_out0, dev_rest

    # the same with staging copies: H2D of the shards, gather, D2H of the outputs
    dev_in = torch.empty((TP, M_STEP, W), dtype=torch.int16, device=device)
    dev_out = torch.empty((TP, M_STEP, V), dtype=torch.int16, device=device)
    host_out1 = torch.empty((TP, M_STEP, V), dtype=torch.int16).pin_memory()
    staged_call = hg.GatherCall(h, [dev_in[r] for r in range(TP)],
                                [dev_out[d] for d in range(TP)], M_STEP)

    def staged_step(i=[0]):
        dev_in.copy_(host_in[i[0] % nsets], non_blocking=True)
        staged_call()
        host_out1.copy_(dev_out, non_blocking=True)
        i[0] += 1

    staged_ms = time_calls(torch, [staged_step], args.steps, args.warmup, stream, "timed_staged")
    hg.hg_sync(h)
    staged_us = round(staged_ms * 1000.0 / args.steps, 3)
    # the host link's write rate for the same bytes: the copy engine moving all
    # ranks' outputs (TP * M * V bf16) to pinned host memory, nothing else
    d2h_ms = time_calls(torch, [lambda: host_out1.copy_(dev_out, non_blocking=True)],
                        args.steps, args.warmup, stream, "timed_d2h")
    d2h_us = round(d2h_ms * 1000.0 / args.steps, 3)
    del host_in, host_out1, dev_in, dev_out
    e2e_ms_max, e2e_us = replica_us_per_call(dist, e2e_ms, args.steps, world, device)
    h.close()
    del shards, outs, calls

    # ---- per-M (config 3 row counts) and large M ----
    per_m, per_m_tuned, per_m_shape, per_m_tuned_shape = {}, {}, {}, {}
    per_m_graph, per_m_graph_tuned = {}, {}
    if not args.quick:
        for M in range(1, 9):
            n = sets_for(TP, W, M)
            # calls issued one by one from Python: fixed rule, then shapes timed
            # at hg_create
            for tuned, res, shp in ((False, per_m, per_m_shape),
                                    (True, per_m_tuned, per_m_tuned_shape)):
                hm, sm_, om_, cm_ = make_workload(torch, hg, synth, TP, W, CAP, M, n, device,
                                                  rows=[M], seed=2, autotune=tuned)
                t = time_calls(torch, cm_, 200, 20, stream)
                hg.hg_sync(hm)
                res[str(M)] = round(t * 1000.0 / 200, 3)
                shp[str(M)] = hg.hg_launch_shape(hm, M)
                hm.close()
                del sm_, om_, cm_
            # host-free issue: 200 calls captured once, replayed (fixed rule, then
            # shapes timed at hg_create)
            per_m_graph[str(M)] = graph_replay_us(torch, hg, synth, TP, W, CAP, M, device,
                                                  stream, 1000, rows=[M], seed=2)
            per_m_graph_tuned[str(M)] = graph_replay_us(
                torch, hg, synth, TP, W, CAP, M, device, stream, 1000, rows=[M], seed=2,
                autotune=True)
    # ---- latency floors at the launch shapes of M = 1..8 (fixed rule) ----
    floors = {}
    hfl = hg.hg_create(TP, W, CAP)
    shapes = {str(M): (hg.hg_launch_shape(hfl, M)["ctas"], 32 * TP)
              for M in (range(1, 9) if not args.quick else [M_STEP])}
    hfl.close()
    floors = latency_floors(torch, hg, shapes, stream, device)
    l2_gbs = l2_copy_gbs(torch, device, stream)
    for M, f in floors.items():
        g = per_m_graph.get(M) if M != str(M_STEP) else round(us_call, 3)
        if g:
            f["gather_us"] = g
            f["gather_over_handoff"] = round(g / f["handoff_us"], 3)
            # algorithmic bytes at the L2-resident copy rate: a bandwidth bound
            bound = algorithmic_bytes(TP, W, int(M)) / (l2_gbs * 1e9) * 1e6
            f["l2_copy_bound_us"] = round(bound, 3)
            f["frac_of_l2_copy"] = round(bound / g, 3)

    large = {}
    for M in ([] if args.quick else [64, 128, 256]):
        hm, sm_, om_, cm_ = make_workload(torch, hg, synth, TP, W, M, M, 3, device, rows=[M],
                                          seed=3, dist_kind="uniform", scale=20.0, sent=0.0,
                                          autotune=tune)
        reps = 30
        t = time_calls(torch, cm_, reps, 5, stream)
        hg.hg_sync(hm)
        us = t * 1000.0 / reps
        gbs = algorithmic_bytes(TP, W, M) / (us * 1e-6) / 1e9
        large[str(M)] = {"us_per_call": round(us, 2), "algorithmic_GBps": round(gbs, 1),
                         "frac_of_measured_hbm": round(gbs / pk["hbm_gbs"], 3),
                         "launch": hg.hg_launch_shape(hm, M),
                         "useful_out_GBps": round(TP * M * V * 2 / (us * 1e-6) / 1e9, 1)}
        hm.close()
        del sm_, om_, cm_

    # ---- fused LM-head producer (config 5) ----
    fused = None
    if not args.quick:
        fused = run_fused_points(torch, hg, synth, device, [1, 4, 8], 20, 3, stream)

    # ---- stock cudaMemcpy2D concat baseline on the step workload ----
    stock_us = None
    if not args.quick:
        sb = torch.empty((3, TP, M_STEP, W), dtype=torch.int16, device=device)
        ob = torch.empty((3, TP, M_STEP, V), dtype=torch.int16, device=device)
        lib = hg.load()
        import ctypes
        arrs = [((ctypes.c_void_p * TP)(*[sb[s, r].data_ptr() for r in range(TP)]),
                 (ctypes.c_void_p * TP)(*[ob[s, d].data_ptr() for d in range(TP)]))
                for s in range(3)]
        sp = stream.cuda_stream
        fns = [lambda a=a: lib.hg_stock_gather(TP, W, a[0], a[1], M_STEP, sp) for a in arrs]
        t = time_calls(torch, fns, 200, 20, stream)
        stock_us = round(t * 1000.0 / 200, 3)

    # ---- CPU oracle on a bounded sample ----
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        us_cpu, n_cpu = oracle_calls_per_sample(args.cpu_seconds)
        cpu = {"value": round(us_cpu, 1), "unit": "us/call", "cores": 1, "kind": "oracle",
               "sample": f"{n_cpu} config-2 calls (TP8, V=163840, M=1) through the "
                         f"single-threaded C++ oracle, {args.cpu_seconds:.0f} s budget"}
        us_all, n_all, cores = oracle_all_cores(2.0)
        cpu["all_cores"] = {"value": round(us_all, 1), "unit": "us/call", "cores": cores,
                            "sample": f"{n_all} config-2 calls: the same single-threaded oracle "
                                      f"in {cores} independent processes for about 2 s each, "
                                      "aggregate throughput"}

    if rank != 0:
        return 0
    B = algorithmic_bytes(TP, W, M_STEP)
    achieved = B / (us_launch * 1e-6) / 1e9
    traffic = traffic_from_profile("tp8_w20480_m1")
    line = {
        "metric": METRIC, "value": round(us_call, 3), "unit": "us/call", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_max / args.steps, 6),
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "int32",
        "data": "synthetic",
        "config": workload_config(),
        "measurement": {
            "l2": f"inputs+outputs rotate over {nsets} sets "
                  f"({nsets * TP * M_STEP * W * 2 * (1 + TP) / 2**20:.0f} MiB > 129 MB L2); "
                  "mailboxes (42 MB) are the method's persistent state",
            "launch": dict(shape, launch="programmatic dependent launch",
                           shapes="autotuned at hg_create" if tune else "fixed rule"),
            "issue": "the timed calls replay CUDA graphs of up to 200 captured calls on a "
                     "handle with device-resident parity, as a captured decode step issues "
                     "them; eager_us_per_call: the same calls issued one by one from Python"},
        "gpu_launches": args.steps,
        "e2e": {"value": round(e2e_us, 3), "unit": "us/call",
                "h2d_bytes_per_step": TP * M_STEP * W * 2,
                "d2h_bytes_per_step": TP * M_STEP * V * 2,
                "path": "hg_gather_host: pinned host shards read and pinned host outputs "
                        "written by the gather kernel itself over the host-device link",
                "staged_copies_us_per_call": staged_us,
                "one_result_copy_to_host_us_per_call": one_us,
                "one_result_copy_d2h_bytes_per_step": M_STEP * V * 2,
                "d2h_copy_of_outputs_alone_us": d2h_us,
                "host_link_note": "d2h_copy_of_outputs_alone_us: the copy engine writing the "
                                  "same d2h bytes to pinned host memory and nothing else; the "
                                  "gather's e2e is bound by that write rate"},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": pk["hbm_gbs"],
                     "unit": "GB/s", "frac": round(achieved / pk["hbm_gbs"], 4),
                     "traffic": traffic,
                     "note": f"algorithmic bytes M*V*2*(1+4*TP) = {B} per launch; peak is the "
                             f"{pk['source']} HBM copy bandwidth; at M=1 the working set is "
                             "L2-resident and the launch is latency-bound: latency_floor_us is "
                             "the one-vector push->poll->copy->re-arm handoff kernel launched "
                             "like the gather (same grid, graph-replayed)",
                     "latency_floor_us": floors[str(M_STEP)]["handoff_us"],
                     "empty_launch_us": floors[str(M_STEP)]["empty_launch_us"],
                     "floor_multiple": round(us_launch / floors[str(M_STEP)]["handoff_us"], 3)},
        "latency_floors_per_m": floors,
        "l2_copy_GBps": l2_gbs,
        "eager_us_per_call": round(eager_us, 3),
        "per_m": per_m,
        "per_m_launch": per_m_shape,
        "per_m_autotuned": per_m_tuned,
        "per_m_autotuned_launch": per_m_tuned_shape,
        "per_m_graph_replay": per_m_graph,
        "per_m_graph_replay_autotuned": per_m_graph_tuned,
        "large_m": large,
        "with_row_stats_us_per_call": stats_us,
        "with_row_stats_graph_replay": stats_graph,
        "drafter_pair": drafter,
        "gather_then_torch_row_stats_us_per_call": torch_stats_us,
        "device_parity_us_per_call": devpar_us,
        "graph_replay_us_per_call": graph_us,
        "stock_memcpy2d_us_per_call": stock_us,
        "fused_lm_head": fused,
        "cpu_baseline": cpu,
        "clocks": clocks,
    }
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


# -------------------------------------------------------------------- fused --

def fused_bytes(tp: int, W: int, K: int, M: int) -> int:
    """Algorithmic bytes of one fused call: every weight byte once, the hidden
    rows, and the gather's push, poll, output write and re-arm."""
    V = tp * W
    return tp * W * K * 2 + tp * M * K * 2 + 4 * tp * M * V * 2


def run_fused_points(torch, hg, synth, device, Ms, reps, warmup, stream, with_unfused=True,
                     Wd=20480):
    """Config 5: TP8, V=163840 (W=20480), K=7168; weights resident (2.35 GB,
    larger than L2). Returns {M: {...}}."""
    import ctypes
    tp, K = 8, 7168
    pk = peaks()
    weight = [synth.weight(4, r, Wd, K, device=device) for r in range(tp)]
    res = {}
    lib = hg.load()
    for M in Ms:
        h = hg.hg_create(tp, Wd, max(Ms), rows=sorted(set(Ms)))
        hid = synth.hidden(4, tp, M, K, device=device)
        outs = torch.empty((tp, M, tp * Wd), dtype=torch.int16, device=device)
        hp = (ctypes.c_void_p * tp)(*[hid[r].data_ptr() for r in range(tp)])
        wp = (ctypes.c_void_p * tp)(*[w.data_ptr() for w in weight])
        op = (ctypes.c_void_p * tp)(*[outs[d].data_ptr() for d in range(tp)])
        sp = stream.cuda_stream

        def call():
            st = lib.hg_gather_fused(h.ptr, hp, wp, None, op, M, K, sp)
            if st != 0:
                raise SystemExit(f"hg_gather_fused failed: {hg.strerror(st)}")
        ms = time_calls(torch, [call], reps, warmup, stream, f"timed_fused_m{M}")
        hg.hg_sync(h)
        us = ms * 1000.0 / reps
        wgbs = tp * Wd * K * 2 / (us * 1e-6) / 1e9
        entry = {"us_per_call": round(us, 2), "weight_GBps": round(wgbs, 1),
                 "weight_frac_of_measured_hbm": round(wgbs / pk["hbm_gbs"], 3),
                 "algorithmic_GBps": round(fused_bytes(tp, Wd, K, M) / (us * 1e-6) / 1e9, 1)}
        if with_unfused:
            # Baseline: cuBLAS GEMM per rank (torch.matmul) then the gather.
            logits = torch.empty((tp, M, Wd), dtype=torch.bfloat16, device=device)
            hb = hid.view(torch.bfloat16)
            wb = [w.view(torch.bfloat16) for w in weight]
            g = hg.GatherCall(h, [logits[r].view(torch.int16) for r in range(tp)],
                              [outs[d] for d in range(tp)], M)

            def unfused():
                for r in range(tp):
                    torch.matmul(hb[r], wb[r].t(), out=logits[r])
                g()
            ms2 = time_calls(torch, [unfused], reps, warmup, stream, f"timed_unfused_m{M}")
            hg.hg_sync(h)
            entry["unfused_cublas_then_gather_us"] = round(ms2 * 1000.0 / reps, 2)
        res[str(M)] = entry
        h.close()
    return res


# -------------------------------------------------------------------- sweep --

def run_sweep(args):
    import torch

    from tp_vocab_logits_gb300 import _build, hg, synth
    _build.build()
    torch.cuda.set_device(0)
    device = torch.device("cuda", 0)
    stream = torch.cuda.current_stream()
    pk = peaks()
    tps = [int(x) for x in args.tps.split(",")]
    widths = [int(x) for x in args.widths.split(",")]
    ms = [int(x) for x in args.ms.split(",")]
    for tp in tps:
        for Wd in widths:
            for M in ms:
                n = sets_for(tp, Wd, M, minimum=2)
                foot = n * M * tp * Wd * 2 * (1 + tp) + 2 * M * tp * tp * Wd * 2
                if foot > args.max_gb * 2**30:
                    n = 2
                h, s_, o_, c_ = make_workload(torch, hg, synth, tp, Wd, M, M, n, device,
                                              rows=[M], seed=3, dist_kind="uniform", scale=20.0,
                                              sent=0.0, elems_per_lane=args.vpt, ctas=args.ctas,
                                              prefetch=args.prefetch,
                                              cooperative=args.cooperative,
                                              autotune=args.autotune)
                c_[0]()  # first call of the point, checked before timing
                hg.hg_sync(h)
                check_concat(torch, s_[0], o_[0], tp, f"sweep tp={tp} W={Wd} M={M} first call")
                t = time_calls(torch, c_, args.calls, 10, stream)
                hg.hg_sync(h)
                last = (args.calls - 1) % n  # set of the last timed call
                check_concat(torch, s_[last], o_[last], tp,
                             f"sweep tp={tp} W={Wd} M={M} last call")
                us = t * 1000.0 / args.calls
                gbs = algorithmic_bytes(tp, Wd, M) / (us * 1e-6) / 1e9
                print(json.dumps({"sweep": "bandwidth", "tp": tp, "shard_cols": Wd, "M": M,
                                  "cooperative": args.cooperative,
                                  "autotune": args.autotune,
                                  "cap": M, "calls": args.calls, "us_per_call": round(us, 3),
                                  "algorithmic_GBps": round(gbs, 1),
                                  "frac_of_measured_hbm": round(gbs / pk["hbm_gbs"], 3),
                                  "launch": hg.hg_launch_shape(h, M), "sets": n}), flush=True)
                h.close()
                del s_, o_, c_
                torch.cuda.empty_cache()
    return 0


def timeline_summary(rec, tp: int, grid: int) -> dict:
    """Launch-by-launch figures of a timeline [calls, ctas, slots] (int64 ns,
    calls in call order): when each launch's first and last CTA started, when
    its wait for the previous kernel returned (first and last CTA), and when
    its last warp finished."""
    import numpy as np
    r = rec[:, :grid, :]
    entry = r[:, :, 0]
    waited = r[:, :, 1]
    cta_end = r[:, :, 2:2 + tp].max(axis=2)
    e_min, e_max = entry.min(axis=1), entry.max(axis=1)
    w_min, w_max = waited.min(axis=1), waited.max(axis=1)
    end = cta_end.max(axis=1)
    n = r.shape[0]
    period = np.diff(w_min)                   # wait release to wait release
    gap = w_min[1:] - end[:-1]                # previous kernel's last warp -> next wait release
    span = end - w_min                        # first wait release -> last warp
    early = (entry[1:] < end[:-1, None]).mean(axis=1)  # CTAs resident before the previous ended
    ser = end - e_min                         # first CTA start -> last warp (what a serialised
                                              # launch would take from its first CTA)

    def st(x):
        return {"mean": round(float(x.mean()) / 1000, 3), "median": round(float(np.median(x)) / 1000, 3),
                "p10": round(float(np.percentile(x, 10)) / 1000, 3),
                "p90": round(float(np.percentile(x, 90)) / 1000, 3)}
    return {"launches": n, "ctas": grid,
            "period_us": st(period), "exposed_gap_us": st(gap), "span_after_wait_us": st(span),
            "first_to_last_cta_wait_us": st(w_max - w_min),
            "first_cta_start_to_last_warp_us": st(ser),
            "first_cta_start_before_wait_release_us": st(w_min - e_min),
            "cta_end_median_after_wait_us": st(np.median(cta_end, axis=1) - w_min),
            "share_of_ctas_resident_before_previous_ended": round(float(early.mean()), 3),
            "total_us_first_wait_to_last_end": round(float(end[-1] - w_min[0]) / 1000, 3)}


def run_timeline(args):
    """Timeline of back-to-back graph-replayed gathers (TP8, V=163840, cap 8)
    from the measurement build (hg_options.timeline_calls): one JSON line per
    M with the launch-by-launch figures, beside the per-call time of the same
    graph replayed without the timeline build."""
    import torch

    from tp_vocab_logits_gb300 import _build, hg, synth
    _build.build()
    torch.cuda.set_device(0)
    device = torch.device("cuda", 0)
    stream = torch.cuda.current_stream()
    for M in [int(x) for x in args.timeline_ms.split(",")]:
        n = sets_for(TP, W, M)
        res = {}
        for tl in (200, 0):
            h, sh, ou, calls = make_workload(torch, hg, synth, TP, W, CAP, M, n, device,
                                             rows=[M], seed=2, device_parity=True,
                                             timeline_calls=tl)
            stats = hg.new_row_stats(M) if args.timeline_stats else None
            k = [0]

            def issue():
                i = k[0] % n
                k[0] += 1
                if stats is not None:
                    hg.hg_gather_stats(h, [sh[i, r] for r in range(TP)],
                                       [ou[i, d] for d in range(TP)], stats, M)
                else:
                    hg.hg_gather(h, [sh[i, r] for r in range(TP)], [ou[i, d] for d in range(TP)],
                                 M)
            issue()
            hg.hg_sync(h)
            us = graph_us_per_launch(torch, issue, stream, reps=5,
                                     label=f"timed_timeline_m{M}_{tl}")
            hg.hg_sync(h)
            check_concat(torch, sh[0], ou[0], TP, f"timeline M={M}")
            if tl:
                rec, nxt = hg.hg_timeline(h)
                rec = rec.cpu().numpy()
                import numpy as np
                rec = np.concatenate([rec[nxt:], rec[:nxt]])  # call order
                if args.timeline_dump:  # the first 50 launches
                    np.save(f"{args.timeline_dump}_m{M}.npy", rec[:50])
                grid = hg.hg_launch_shape(h, M)["ctas"] if stats is None else \
                    int((rec[0, :, 0] > 0).sum())
                res = timeline_summary(rec, TP, grid)
                res["graph_replay_us_per_call_timeline_build"] = us
            else:
                res["graph_replay_us_per_call"] = us
            h.close()
            del sh, ou, calls
        print(json.dumps(dict(res, timeline="gather" if not args.timeline_stats else
                              "gather_stats", tp=TP, shard_cols=W, M=M)), flush=True)
    return 0


def run_fused_timeline(args):
    """Timeline of back-to-back fused calls (TP8, V=163840, K=7168) at each M:
    per launch, when the CTAs started, finished set-up, pushed each item,
    consumed the neighbour's items and finished (hg_gather_fused records in the
    handle's timeline). One JSON line per M; raw records with --timeline-dump."""
    import ctypes

    import numpy as np
    import torch

    from tp_vocab_logits_gb300 import _build, hg, synth
    _build.build()
    torch.cuda.set_device(0)
    device = torch.device("cuda", 0)
    stream = torch.cuda.current_stream()
    tp, K, Wd, n = 8, 7168, 20480, 12
    weight = [synth.weight(4, r, Wd, K, device=device) for r in range(tp)]
    lib = hg.load()
    wp = (ctypes.c_void_p * tp)(*[w.data_ptr() for w in weight])
    for M in [int(x) for x in args.timeline_ms.split(",")]:
        h = hg.hg_create(tp, Wd, max(8, M), rows=sorted({1, 4, 8, M}), timeline_calls=n)
        hid = synth.hidden(4, tp, M, K, device=device)
        outs = torch.empty((tp, M, tp * Wd), dtype=torch.int16, device=device)
        hp = (ctypes.c_void_p * tp)(*[hid[r].data_ptr() for r in range(tp)])
        op = (ctypes.c_void_p * tp)(*[outs[d].data_ptr() for d in range(tp)])
        for _ in range(n):
            st = lib.hg_gather_fused(h.ptr, hp, wp, None, op, M, K, stream.cuda_stream)
            if st != 0:
                raise SystemExit(f"hg_gather_fused failed: {hg.strerror(st)}")
        hg.hg_sync(h)
        rec, nxt = hg.hg_timeline(h)
        rec = rec.cpu().numpy()
        rec = np.concatenate([rec[nxt:], rec[:nxt]])  # call order
        G = int((rec[0, :, 0] > 0).sum())
        r = rec[:, :G, :]
        if args.timeline_dump:
            np.save(f"{args.timeline_dump}_fused_m{M}.npy", r)
        e0 = r[:, :, 0].min(axis=1)

        def rel(x):
            return (x - e0[:, None]) / 1000.0
        done = rel(r[:, :, 17])
        out = {"fused_timeline": True, "M": M, "ctas": G, "calls": n,
               "period_us": round(float(np.median(np.diff(e0))) / 1000, 3),
               "setup_done_us": round(float(np.median(rel(r[:, :, 1]))), 3),
               "push_item_us_median": [round(float(np.median(rel(r[:, :, 2 + i]))), 2)
                                       for i in range(8)],
               "consume_item_us_median": [round(float(np.median(rel(r[:, :, 10 + j]))), 2)
                                          for j in range(6)],
               "loop_done_us": [round(float(np.percentile(rel(r[:, :, 16]), q)), 2)
                                for q in (0, 50, 100)],
               "cta_done_us": [round(float(np.percentile(done, q)), 2) for q in (0, 50, 100)]}
        print(json.dumps(out), flush=True)
        h.close()
    return 0


def run_stats_only(args):
    """hg_gather_stats on the step workload (TP8, V=163840, cap 8, M rows),
    one JSON line per M: us/call, checked against the plain gather's outputs."""
    import ctypes

    import torch

    from tp_vocab_logits_gb300 import _build, hg, synth
    _build.build()
    torch.cuda.set_device(0)
    device = torch.device("cuda", 0)
    stream = torch.cuda.current_stream()
    lib = hg.load()
    for M in [int(x) for x in args.stats_ms.split(",")]:
        n = sets_for(TP, W, M)
        kw = {"elems_per_lane": args.vpt} if args.vpt else {}
        h, sh, ou, calls = make_workload(torch, hg, synth, TP, W, CAP, M, n, device, rows=[M], **kw)
        st = hg.new_row_stats(M)
        arrs = [((ctypes.c_void_p * TP)(*[sh[s_, r].data_ptr() for r in range(TP)]),
                 (ctypes.c_void_p * TP)(*[ou[s_, d].data_ptr() for d in range(TP)]))
                for s_ in range(n)]
        sp = stream.cuda_stream
        fns = [lambda a_=a_: lib.hg_gather_stats(h.ptr, a_[0], a_[1], M, st.data_ptr(), sp)
               for a_ in arrs]
        fns[0]()
        hg.hg_sync(h)
        check_concat(torch, sh[0], ou[0], TP, f"stats M={M}")
        t = time_calls(torch, fns, args.calls, 5, stream, "timed_stats")
        hg.hg_sync(h)
        print(json.dumps({"stats": "hg_gather_stats", "tp": TP, "shard_cols": W, "M": M,
                          "calls": args.calls, "us_per_call": round(t * 1000.0 / args.calls, 3),
                          "elems_per_lane": args.vpt or None}),
              flush=True)
        h.close()
        del sh, ou, calls, fns
    return 0


def run_fused_only(args):
    import torch

    from tp_vocab_logits_gb300 import _build, hg, synth
    _build.build()
    torch.cuda.set_device(0)
    device = torch.device("cuda", 0)
    Ms = [int(x) for x in args.fused_ms.split(",")]
    res = run_fused_points(torch, hg, synth, device, Ms, args.calls, 3,
                           torch.cuda.current_stream(), with_unfused=not args.quick,
                           Wd=args.fused_w)
    for M, e in res.items():
        print(json.dumps(dict(e, fused="lm_head+gather", tp=8, shard_cols=args.fused_w, K=7168,
                              M=int(M))), flush=True)
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawTextHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--quick", action="store_true", help="step workload only")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--sweep", action="store_true", help="bandwidth sweep, one line per point")
    ap.add_argument("--fused", action="store_true",
                    help="fused LM-head producer only (TP8, K=7168, V=163840), one line per M")
    ap.add_argument("--fused-ms", default="1,4,8")
    ap.add_argument("--stats", action="store_true",
                    help="hg_gather_stats only (TP8, V=163840), one line per M")
    ap.add_argument("--stats-ms", default="1,4,8")
    ap.add_argument("--timeline", action="store_true",
                    help="launch timeline of graph-replayed gathers (TP8, V=163840), one line "
                         "per M")
    ap.add_argument("--timeline-ms", default="1,8")
    ap.add_argument("--fused-timeline", action="store_true",
                    help="launch timeline of back-to-back fused calls (TP8, K=7168), one line "
                         "per M of --timeline-ms")
    ap.add_argument("--timeline-dump", default="",
                    help="--timeline: also save the raw records to <prefix>_m<M>.npy")
    ap.add_argument("--timeline-stats", action="store_true",
                    help="--timeline: time hg_gather_stats instead of hg_gather")
    ap.add_argument("--fused-w", type=int, default=20480, help="fused: shard columns per rank")
    ap.add_argument("--tps", default="2,4,8,16")
    ap.add_argument("--widths", default="4096,8192,20480,65536")
    ap.add_argument("--ms", default="1,8,32,64,128,256")
    ap.add_argument("--calls", type=int, default=200)
    ap.add_argument("--max-gb", type=float, default=120.0)
    ap.add_argument("--vpt", type=int, default=0, help="sweep and --stats: force elements per lane")
    ap.add_argument("--ctas", type=int, default=0, help="sweep: force the CTA count")
    ap.add_argument("--prefetch", type=int, default=0,
                    help="sweep: 1 shard prefetch on, 2 off (0: chosen per row count)")
    ap.add_argument("--autotune", action="store_true",
                    help="launch shapes timed at hg_create (hg_options.autotune) instead of "
                         "the library's fixed rule")
    ap.add_argument("--cooperative", action="store_true", help="sweep: cooperative launch")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        return run_reference(args)
    if args.sweep:
        return run_sweep(args)
    if args.fused:
        return run_fused_only(args)
    if args.stats:
        return run_stats_only(args)
    if args.timeline:
        return run_timeline(args)
    if args.fused_timeline:
        return run_fused_timeline(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
