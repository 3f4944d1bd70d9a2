"""gla_fwd_noalloc: the entry point for callers that cannot allocate device
memory (a framework that pools all HBM itself, a loop where cudaMalloc is
banned because it can synchronise the device, a plugin with no allocator).
It runs the same pass with a fixed library-owned scratch array as workspace.

This file is collected last on purpose: it checks the no-allocation entry
point against the ordinary one, and must pass both on its own in a fresh
process and after every other test."""
import pytest
import torch

import chunkwise_gated_linear_gla_gb300 as gla
from chunkwise_gated_linear_gla_gb300 import binding as bnd
from chunkwise_gated_linear_gla_gb300 import build as gbuild
from chunkwise_gated_linear_gla_gb300 import inputs as gi

from _util import assert_close, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    gbuild.build()
    bnd.load()


def _inputs(seed, T):
    w = gi.Workload("noalloc", B=2, H=2, T=T, dk=128, dv=256, dtype=torch.bfloat16,
                    gate=gi.GATE_PER_KEY, s0_std=0.02)
    x = gi.make_inputs(w, seed=seed)
    return w, {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}


def test_noalloc_matches_gla_fwd_on_two_calls_in_a_row():
    # two consecutive calls with different inputs share the scratch array;
    # each must agree with gla_fwd (which takes its workspace from the allocator)
    for seed, T in ((1, 300), (2, 517)):
        w, c = _inputs(seed, T)
        args = (w.B, w.H, w.T, w.dk, w.dv, 64)
        O_ref = torch.empty(w.B, w.H, w.T, w.dv, dtype=torch.bfloat16, device="cuda")
        ST_ref = torch.empty(w.B, w.H, w.dk, w.dv, device="cuda")
        bnd.gla_fwd(c["q"], c["k"], c["v"], c["log_g"], c["S0"], O_ref, ST_ref, *args)
        O = torch.full_like(O_ref, float("nan"))
        ST = torch.full_like(ST_ref, float("nan"))
        bnd.gla_fwd_noalloc(c["q"], c["k"], c["v"], c["log_g"], c["S0"], O, ST, *args)
        torch.cuda.synchronize()
        assert gla.gla_device_status() == 0
        assert_close(to_np(O), to_np(O_ref), torch.bfloat16, f"O (call T={T})")
        assert_close(to_np(ST), to_np(ST_ref), torch.bfloat16, f"ST (call T={T})")


def test_noalloc_rejects_calls_beyond_the_scratch_size():
    # B*H*T far beyond what 32 MiB of workspace holds: refused before any launch
    T = 1 << 20
    base = 1 << 40   # placeholder addresses, far apart so no argument check trips first
    s = bnd.gla_fwd_noalloc(base, 2 * base, 3 * base, 4 * base, None, 5 * base, None,
                            1, 4, T, 256, 512, 64, check=False)
    assert s == bnd.GLA_ERR_WORKSPACE
