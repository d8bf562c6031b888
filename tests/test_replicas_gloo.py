"""Host logic of bench.py's multi-GPU path (replicas only), run as two gloo
ranks on the CPU: the whole-job time is the maximum over the ranks, and the
per-call figure divides it by every rank's calls."""

import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, times, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import torch
        ms_max, us = bench.replica_us_per_call(dist, times[rank], 100, world, torch.device("cpu"))
        w, r, lr = bench.dist_env()
        q.put((rank, ms_max, us, w, r, lr))
        bench.barrier(dist)
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("times", [(2.0, 3.5), (7.25, 1.0)])
def test_replica_aggregation_two_ranks(times):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, times, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, ms_max, us, w, r, lr in got:
        assert ms_max == max(times)
        assert us == pytest.approx(max(times) * 1000.0 / (100 * 2))
        assert (w, r, lr) == (2, rank, rank)
