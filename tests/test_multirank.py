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


# ---------------------------------------------------------------- the sequence exchange

_SEQ_CUTS = (0, 70, 150, 201)   # rank r holds tokens [cuts[r], cuts[r+1]) of every (b, h)


def _seq_case():
    import torch
    from chunkwise_gated_linear_gla_gb300 import inputs as gi
    w = gi.Workload("seqpar", B=2, H=2, T=_SEQ_CUTS[-1], dk=8, dv=6, dtype=torch.float32,
                    gate=gi.GATE_PER_KEY, s0_std=0.5)
    return gi.make_inputs(w, seed=51)


def _seq_worker(rank, world, port, q):
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import numpy as np
    import torch
    import oracle
    from chunkwise_gated_linear_gla_gb300 import seqpar
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        x = _seq_case()
        a, b = _SEQ_CUTS[rank], _SEQ_CUTS[rank + 1]
        sl = lambda t: t[:, :, a:b]
        # this rank's pair, computed by the oracle; rank 0 folds in the sequence's S0
        lg, Sst = oracle.segment_pair(sl(x["k"]), sl(x["v"]), sl(x["log_g"]), x["gate"])
        if rank == 0:
            Sst = np.exp(lg)[..., None] * x["S0"].double().numpy() + Sst
        lgs, sss = seqpar.exchange_pairs(torch.from_numpy(lg), torch.from_numpy(Sst))
        # the state entering this rank's segment, chained from the ranks before it
        if rank == 0:
            S_in = x["S0"].double().numpy()
        else:
            _, S_in = oracle.pair_scan(list(lgs[:rank].numpy()), list(sss[:rank].numpy()), None)
        q.put((rank, lgs.shape[0], lgs.numpy(), sss.numpy(), S_in))
    finally:
        dist.destroy_process_group()


def test_sequence_exchange_two_ranks():
    """gloo, world size 2 (plus a 3-rank run): every rank gets all pairs in segment
    order, and the state it chains from them is the recurrence's state at its
    segment's first token, from the fp64 oracle over the whole sequence."""
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import numpy as np
    import oracle
    x = _seq_case()
    for world in (2, 3):
        ctx = mp.get_context("spawn")
        q = ctx.Queue()
        port = _free_port()
        procs = [ctx.Process(target=_seq_worker, args=(r, world, port, q)) for r in range(world)]
        for p in procs:
            p.start()
        res = sorted((q.get(timeout=120) for _ in range(world)), key=lambda r: r[0])
        for p in procs:
            p.join(timeout=120)
            assert p.exitcode == 0
        for rank, P, lgs, sss, S_in in res:
            assert P == world
            # rank order is segment order: entry d is rank d's own pair
            for d in range(world):
                a, b = _SEQ_CUTS[d], _SEQ_CUTS[d + 1]
                lg, Sst = oracle.segment_pair(x["k"][:, :, a:b], x["v"][:, :, a:b], x["log_g"][:, :, a:b],
                                              x["gate"])
                np.testing.assert_array_equal(lgs[d], lg)
                if d > 0:
                    np.testing.assert_array_equal(sss[d], Sst)
            a = _SEQ_CUTS[rank]
            _, S_a = oracle.gla_forward(x["q"][:, :, :a], x["k"][:, :, :a], x["v"][:, :, :a],
                                        x["log_g"][:, :, :a], x["gate"], x["S0"])
            np.testing.assert_allclose(S_in, S_a, rtol=0, atol=1e-10)
