"""gla_fwd_noalloc: the entry point for callers that cannot allocate device
memory (a framework that pools all HBM itself, a loop where cudaMalloc is
banned because it can synchronise the device, a plugin with no allocator).
It runs the same pass with a fixed library-owned scratch array as workspace.

This file is collected last on purpose: it checks the no-allocation entry
point against the ordinary one and against the fp64 oracle, and must pass
both on its own in a fresh process and after every other test."""
import pytest
import torch

import oracle
import chunkwise_gated_linear_gla_gb300 as gla
from chunkwise_gated_linear_gla_gb300 import binding as bnd
from chunkwise_gated_linear_gla_gb300 import build as gbuild
from chunkwise_gated_linear_gla_gb300 import inputs as gi

from _util import assert_close, to_np

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 32 * 1024 * 1024   # GLA_NOALLOC_SCRATCH_BYTES in include/gla.h


@pytest.fixture(scope="module", autouse=True)
def _built():
    gbuild.build()
    oracle.build()
    bnd.load()


def _inputs(seed, T, gate):
    # dk = 128 plans the two-kernel tensor path, whose workspace (Q (.) Lambda, K (.) Gamma,
    # the scores, the chunk decays) lives in the scratch array
    w = gi.Workload("noalloc", B=2, H=2, T=T, dk=128, dv=256, dtype=torch.bfloat16, gate=gate, s0_std=0.02)
    x = gi.make_inputs(w, seed=seed)
    return w, x, {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}


def test_noalloc_matches_gla_fwd_and_oracle_on_calls_in_a_row():
    # Consecutive calls share the scratch array. The first is the largest, so the later,
    # smaller ones run over whatever it left there; every T is ragged, and the last call has
    # no gate. Each result must equal gla_fwd's (workspace from the allocator) and the oracle's.
    for seed, T, gate in ((1, 517, gi.GATE_PER_KEY), (2, 300, gi.GATE_PER_KEY), (3, 129, gi.GATE_NONE)):
        w, x, c = _inputs(seed, T, gate)
        args = (w.B, w.H, w.T, w.dk, w.dv, 64)
        O_ref = torch.empty(w.B, w.H, w.T, w.dv, dtype=torch.bfloat16, device="cuda")
        ST_ref = torch.empty(w.B, w.H, w.dk, w.dv, device="cuda")
        bnd.gla_fwd(c["q"], c["k"], c["v"], c["log_g"], c["S0"], O_ref, ST_ref, *args)
        O = torch.full_like(O_ref, float("nan"))
        ST = torch.full_like(ST_ref, float("nan"))
        bnd.gla_fwd_noalloc(c["q"], c["k"], c["v"], c["log_g"], c["S0"], O, ST, *args)
        torch.cuda.synchronize()
        assert gla.gla_device_status() == 0
        assert_close(to_np(O), to_np(O_ref), torch.bfloat16, f"O vs gla_fwd (T={T})")
        assert_close(to_np(ST), to_np(ST_ref), torch.bfloat16, f"ST vs gla_fwd (T={T})")
        Oo, STo = oracle.gla_forward(x["q"], x["k"], x["v"], x["log_g"], x["gate"], x["S0"])
        assert_close(to_np(O), Oo, torch.bfloat16, f"O vs oracle (T={T})")
        assert_close(to_np(ST), STo, torch.bfloat16, f"ST vs oracle (T={T})")


def test_noalloc_rejects_calls_beyond_the_scratch_size():
    # B*H*T far beyond what the scratch array holds: refused before any launch. The pointers
    # are placeholders, so first make sure (host-side planning only) that this shape's plan
    # does need more workspace than the array has; otherwise the call would launch on them.
    B, H, T, dk, dv = 1, 4, 1 << 20, 128, 512
    base = 1 << 40   # placeholder addresses, far apart so no argument check trips first
    p = bnd.gla_fwd_params()
    p.q, p.k, p.v, p.log_g, p.O = base, 2 * base, 3 * base, 4 * base, 5 * base
    p.B, p.H, p.T, p.dk, p.dv, p.chunk = B, H, T, dk, dv, 64
    p.dtype, p.gate, p.path, p.force_segments = bnd.GLA_BF16, bnd.GLA_GATE_PER_KEY, bnd.GLA_PATH_AUTO, 1
    assert bnd.gla_fwd_workspace_size(p) > SCRATCH_BYTES
    s = bnd.gla_fwd_noalloc(base, 2 * base, 3 * base, 4 * base, None, 5 * base, None,
                            B, H, T, dk, dv, 64, check=False)
    assert s == bnd.GLA_ERR_WORKSPACE
