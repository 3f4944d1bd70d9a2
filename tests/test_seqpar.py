"""GPU parity of the sequence exchange (gla_segment_pair, gla_pair_scan,
gla_pair_combine, and the output pass from the exchanged state) against the
fp64 oracle: a sequence cut into P segments, each handled as one rank would,
must give the whole sequence's O and final state."""
import threading

import numpy as np
import pytest
import torch

import oracle
import chunkwise_gated_linear_gla_gb300 as gla
from chunkwise_gated_linear_gla_gb300 import binding as bnd
from chunkwise_gated_linear_gla_gb300 import build as gbuild
from chunkwise_gated_linear_gla_gb300 import inputs as gi
from chunkwise_gated_linear_gla_gb300 import seqpar

from _util import assert_close, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    gbuild.build()
    oracle.build()


def _dev(x):
    return {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}


def _sl(x, a, b):
    """Tokens [a, b) of every input (a per-head gate is shared by all segments)."""
    g = x["log_g"]
    if g is not None and x["gate"] != gi.GATE_HEAD_SCALAR:
        g = g[:, :, a:b].contiguous()
    return {"q": x["q"][:, :, a:b].contiguous(), "k": x["k"][:, :, a:b].contiguous(),
            "v": x["v"][:, :, a:b].contiguous(), "log_g": g, "gate": x["gate"]}


CASES = [
    # (name, dk, dv, dtype, gate): the tensor route (bf16, dk <= 256) and the CUDA-core one
    ("per_key_dk256", 256, 512, torch.bfloat16, gi.GATE_PER_KEY),
    ("per_key_dk128", 128, 256, torch.bfloat16, gi.GATE_PER_KEY),
    ("head_scalar", 128, 128, torch.bfloat16, gi.GATE_HEAD_SCALAR),
    ("token_scalar", 64, 128, torch.bfloat16, gi.GATE_TOKEN_SCALAR),
    ("no_gate", 128, 128, torch.bfloat16, gi.GATE_NONE),
    ("fp32_simt", 64, 48, torch.float32, gi.GATE_PER_KEY),
    ("dk512_simt", 512, 128, torch.bfloat16, gi.GATE_PER_KEY),
]


@pytest.mark.parametrize("name,dk,dv,dtype,gate", CASES, ids=[c[0] for c in CASES])
def test_segment_pair_matches_oracle(name, dk, dv, dtype, gate):
    w = gi.Workload("t", B=2, H=2, T=203, dk=dk, dv=dv, dtype=dtype, gate=gate)
    x = gi.make_inputs(w, seed=61)
    c = _dev(x)
    lg, Sst = gla.segment_pair(c["k"], c["v"], c["log_g"], gate=x["gate"], q=c["q"])
    torch.cuda.synchronize()
    assert gla.gla_device_status() == 0
    lg_ref, S_ref = oracle.segment_pair(x["k"], x["v"], x["log_g"], x["gate"])
    # log Gamma: an fp64 sum rounded once to fp32
    np.testing.assert_allclose(to_np(lg), lg_ref, rtol=1e-6, atol=1e-6)
    assert_close(to_np(Sst), S_ref, dtype, "S*")
    # q does not enter the pair
    lg2, S2 = gla.segment_pair(c["k"], c["v"], c["log_g"], gate=x["gate"], q=None)
    torch.cuda.synchronize()
    assert torch.equal(lg, lg2)
    assert_close(to_np(S2), S_ref, dtype, "S* (no q)")


@pytest.mark.parametrize("name,dk,dv,dtype,gate", CASES[:2] + CASES[4:6], ids=[c[0] for c in CASES[:2] + CASES[4:6]])
@pytest.mark.parametrize("cuts", [[], [64], [1, 130], [37, 38, 100, 192]], ids=["P1", "P2", "P3", "P5"])
def test_split_sequence_matches_oracle(name, dk, dv, dtype, gate, cuts):
    """P segments (ragged, one of a single token, one ending on a chunk edge): the pairs,
    the scan with the sequence's S0, then each segment's pass from its S_in; the pieces of
    O and the last state are the whole sequence's."""
    T = 230
    w = gi.Workload("t", B=2, H=2, T=T, dk=dk, dv=dv, dtype=dtype, gate=gate, s0_std=0.1)
    x = gi.make_inputs(w, seed=62 + len(cuts))
    c = _dev(x)
    edges = [0] + cuts + [T]
    pairs = [gla.segment_pair(s["k"], s["v"], s["log_g"], gate=s["gate"])
             for s in (_sl(c, a, b) for a, b in zip(edges, edges[1:]))]
    LG = torch.stack([p[0] for p in pairs])
    SS = torch.stack([p[1] for p in pairs])
    S_in, S_T = gla.pair_scan(LG, SS, c["S0"])
    Os, ST_last = [], None
    for d, (a, b) in enumerate(zip(edges, edges[1:])):
        s = _sl(c, a, b)
        O, ST_last = gla.forward(s["q"], s["k"], s["v"], s["log_g"], S_in[d], gate=s["gate"])
        Os.append(O)
    torch.cuda.synchronize()
    assert gla.gla_device_status() == 0
    Oref, STref = oracle.gla_forward(x["q"], x["k"], x["v"], x["log_g"], x["gate"], x["S0"])
    assert_close(to_np(torch.cat(Os, dim=2)), Oref, dtype, "O")
    assert_close(to_np(ST_last), STref, dtype, "S_T (last segment's pass)")
    assert_close(to_np(S_T), STref, dtype, "S_T (scan)")
    for d, a in enumerate(edges[:-1]):
        _, S_a = oracle.gla_forward(x["q"][:, :, :a], x["k"][:, :, :a], x["v"][:, :, :a],
                                    None if x["log_g"] is None else x["log_g"][:, :, :a], x["gate"], x["S0"])
        assert_close(to_np(S_in[d]), S_a, dtype, f"S_in[{d}]")


def test_scan_in_place_and_single_pair_forms():
    """S_in may overwrite S_star; the scan over the first d pairs gives segment d's S_in."""
    w = gi.Workload("t", B=1, H=3, T=150, dk=128, dv=256, dtype=torch.bfloat16, gate=gi.GATE_PER_KEY,
                    s0_std=0.2)
    x = gi.make_inputs(w, seed=63)
    c = _dev(x)
    edges = [0, 50, 100, 150]
    pairs = [gla.segment_pair(s["k"], s["v"], s["log_g"]) for s in (_sl(c, a, b) for a, b in zip(edges, edges[1:]))]
    LG = torch.stack([p[0] for p in pairs])
    SS = torch.stack([p[1] for p in pairs])
    S_in, S_T = gla.pair_scan(LG, SS, c["S0"])
    B, H, dk, dv = c["S0"].shape
    SS2 = SS.clone()
    T2 = c["S0"].clone()
    bnd.gla_pair_scan(3, LG, SS2, T2, SS2, T2, B, H, dk, dv)   # both outputs in place
    for d in range(3):
        _, Sd = gla.pair_scan(LG[:d], SS[:d], c["S0"], want_S_in=False)
        torch.cuda.synchronize()
        assert torch.equal(Sd, S_in[d])
    torch.cuda.synchronize()
    assert torch.equal(SS2, S_in) and torch.equal(T2, S_T)


def test_pair_combine_tree_equals_scan():
    """The composition is associative: ((p3 o p2) o (p1 o p0)) and the serial scan agree."""
    w = gi.Workload("t", B=2, H=2, T=256, dk=64, dv=128, dtype=torch.bfloat16, gate=gi.GATE_PER_KEY, s0_std=0.3)
    x = gi.make_inputs(w, seed=64)
    c = _dev(x)
    edges = [0, 40, 128, 129, 256]
    pairs = [gla.segment_pair(s["k"], s["v"], s["log_g"]) for s in (_sl(c, a, b) for a, b in zip(edges, edges[1:]))]
    _, S_T = gla.pair_scan(torch.stack([p[0] for p in pairs]), torch.stack([p[1] for p in pairs]), c["S0"],
                           want_S_in=False)
    lo = [pairs[0][0].clone(), pairs[0][1].clone()]
    gla.pair_combine(pairs[1][0], pairs[1][1], lo[0], lo[1])           # p1 o p0
    hi = [pairs[2][0].clone(), pairs[2][1].clone()]
    gla.pair_combine(pairs[3][0], pairs[3][1], hi[0], hi[1])           # p3 o p2
    gla.pair_combine(hi[0], hi[1], lo[0], lo[1])                       # (p3 o p2) o (p1 o p0)
    S0_in = c["S0"].clone()
    zero = torch.zeros_like(lo[0])
    gla.pair_combine(lo[0], lo[1], zero, S0_in)                        # the whole map applied to S0
    torch.cuda.synchronize()
    scale = float(S_T.abs().max())
    assert (S0_in - S_T).abs().max().item() <= 1e-5 * max(1.0, scale)
    torch.testing.assert_close(zero, sum(p[0] for p in pairs), rtol=1e-6, atol=1e-4)


def test_empty_segment_is_the_identity():
    w = gi.Workload("t", B=1, H=2, T=0, dk=128, dv=128, dtype=torch.bfloat16, gate=gi.GATE_PER_KEY)
    x = gi.make_inputs(w, seed=65)
    c = _dev(x)
    lg, Sst = gla.segment_pair(c["k"], c["v"], c["log_g"])
    torch.cuda.synchronize()
    assert torch.count_nonzero(lg) == 0 and torch.count_nonzero(Sst) == 0


def test_segment_pair_argument_errors():
    w = gi.Workload("t", B=1, H=2, T=64, dk=128, dv=128, dtype=torch.bfloat16, gate=gi.GATE_PER_KEY)
    x = gi.make_inputs(w, seed=66)
    c = _dev(x)
    lg = torch.empty(1, 2, 128, device="cuda")
    Sst = torch.empty(1, 2, 128, 128, device="cuda")
    p = bnd.make_params(c["k"], c["k"], c["v"], c["log_g"], None, None, None)
    assert bnd.gla_segment_pair_workspace_size(p) > 0
    assert bnd.gla_segment_pair(p, lg, Sst, check=False) == bnd.GLA_ERR_WORKSPACE
    assert bnd.gla_segment_pair(p, lg, None, check=False) == bnd.GLA_ERR_INVALID_ARG
    # the log decay may not alias the state
    assert bnd.gla_segment_pair(p, Sst, Sst, check=False) == bnd.GLA_ERR_INVALID_ARG
    pb = bnd.make_params(c["k"], c["k"], c["v"], c["log_g"], None, None, None, gate=bnd.GLA_GATE_BILINEAR,
                         log_b=c["v"].float())
    assert bnd.gla_segment_pair(pb, lg, Sst, check=False) == bnd.GLA_ERR_UNSUPPORTED


@pytest.mark.parametrize("P", [2, 3])
def test_forward_sequence_parallel_ranks_as_threads(P):
    """forward_sequence_parallel as P ranks would run it, here host threads on one GPU
    whose exchange is an in-memory all-gather (no kernel waits on another)."""
    T = 300
    w = gi.Workload("t", B=2, H=2, T=T, dk=256, dv=512, dtype=torch.bfloat16, gate=gi.GATE_PER_KEY, s0_std=0.05)
    x = gi.make_inputs(w, seed=67 + P)
    c = _dev(x)
    edges = [round(T * r / P) for r in range(P + 1)]
    slots = [None] * P
    barrier = threading.Barrier(P, timeout=120)
    results, errors = [None] * P, []

    def rank_main(r):
        try:
            def exchange(lg, ss):
                torch.cuda.synchronize()
                slots[r] = (lg, ss)
                barrier.wait()
                return torch.stack([s[0] for s in slots]), torch.stack([s[1] for s in slots])
            s = _sl(c, edges[r], edges[r + 1])
            results[r] = seqpar.forward_sequence_parallel(s["q"], s["k"], s["v"], s["log_g"],
                                                          c["S0"] if r == 0 else None, rank=r, exchange=exchange)
            torch.cuda.synchronize()
        except Exception as e:  # pragma: no cover - reported below
            errors.append(e)
            barrier.abort()

    threads = [threading.Thread(target=rank_main, args=(r,)) for r in range(P)]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=300)
    assert not errors, errors
    assert gla.gla_device_status() == 0
    Oref, STref = oracle.gla_forward(x["q"], x["k"], x["v"], x["log_g"], x["gate"], x["S0"])
    assert_close(to_np(torch.cat([r[0] for r in results], dim=2)), Oref, torch.bfloat16, "O")
    assert_close(to_np(results[-1][1]), STref, torch.bfloat16, "S_T")
