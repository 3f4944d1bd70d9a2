"""The multi-rank bench logic on CPU (gloo, world size 2): each rank runs its
own replica batch (the path shards over (b, h) with no exchange), the job's
time is the slowest rank's, and throughput counts every rank's tokens."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        step_ms = 1.0 + rank          # rank 1 is the slow one
        t = bench.max_over_ranks(step_ms, dist, "cpu")
        v = bench.job_tokens_per_s(16384, world, t)
        q.put((rank, t, v))
    finally:
        dist.destroy_process_group()


def test_two_ranks_max_time_and_job_throughput():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for rank, t, v in res:
        assert t == 2.0                      # slowest rank's time on every rank
        assert v == pytest.approx(16384 * 2 / 2e-3)


def test_single_rank_helpers():
    import bench
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.job_tokens_per_s(1000, 1, 1.0) == pytest.approx(1e6)
