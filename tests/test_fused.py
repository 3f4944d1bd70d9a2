"""GPU parity of the fused per-key pass (gla_chunk_fused: the gate prep inside the chunk
pass, one thread-block cluster per head sharing it through distributed shared memory)
against the fp64 oracle, through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
import chunkwise_gated_linear_gla_gb300 as gla
from chunkwise_gated_linear_gla_gb300 import binding as bnd
from chunkwise_gated_linear_gla_gb300 import build as gbuild
from chunkwise_gated_linear_gla_gb300 import inputs as gi

from _util import assert_close, errors, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    gbuild.build()
    oracle.build()


def _dev(x):
    return {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}


def _stages(c, x, path=gla.GLA_PATH_FUSED):
    O = torch.empty(x["v"].shape, dtype=x["v"].dtype, device="cuda")
    p = bnd.make_params(c["q"], c["k"], c["v"], c["log_g"], c["S0"], O, None, gate=x["gate"], path=path)
    return [bnd.gla_fwd_stage_name(p, i) for i in range(bnd.gla_fwd_num_stages(p))]


def _check(w, seed, x=None):
    x = gi.make_inputs(w, seed=seed) if x is None else x
    c = _dev(x)
    assert _stages(c, x) == ["gla_chunk_fused"]
    O, ST = gla.forward(c["q"], c["k"], c["v"], c["log_g"], c["S0"], gate=x["gate"], path=gla.GLA_PATH_FUSED)
    torch.cuda.synchronize()
    assert gla.gla_device_status() == 0
    Oref, STref = oracle.gla_forward(x["q"], x["k"], x["v"], x["log_g"], x["gate"], x["S0"])
    assert_close(to_np(O), Oref, torch.bfloat16, "O")
    assert_close(to_np(ST), STref, torch.bfloat16, "ST")
    return x, O, ST


@pytest.mark.parametrize("dv", [512, 256])
@pytest.mark.parametrize("T", [1, 63, 64, 65, 200, 333])
def test_fused_ragged_T(dv, T):
    """Clusters of 4 (dv = 512) and of 2 (dv = 256) CTAs, a ragged last chunk, S0 given."""
    w = gi.Workload("t", B=2, H=2, T=T, dk=256, dv=dv, dtype=torch.bfloat16, gate=gi.GATE_PER_KEY, s0_std=0.02)
    _check(w, seed=100 + T + dv)


def test_fused_no_initial_state():
    w = gi.Workload("t", B=1, H=3, T=256, dk=256, dv=512, dtype=torch.bfloat16, gate=gi.GATE_PER_KEY)
    _check(w, seed=111)


def test_fused_matches_staged_path():
    """The fused pass and the two-kernel (prep, chunk pass) form of the same tensor path."""
    w = gi.Workload("t", B=2, H=2, T=300, dk=256, dv=512, dtype=torch.bfloat16, gate=gi.GATE_PER_KEY, s0_std=0.02)
    x = gi.make_inputs(w, seed=112)
    c = _dev(x)
    assert _stages(c, x, gla.GLA_PATH_STAGED) == ["gla_chunk_prep", "gla_chunk_fwd"]
    O1, S1 = gla.forward(c["q"], c["k"], c["v"], c["log_g"], c["S0"], path=gla.GLA_PATH_FUSED)
    O2, S2 = gla.forward(c["q"], c["k"], c["v"], c["log_g"], c["S0"], path=gla.GLA_PATH_STAGED)
    torch.cuda.synchronize()
    assert gla.gla_device_status() == 0
    assert errors(to_np(O1), to_np(O2))[0] < 5e-3
    assert errors(to_np(S1), to_np(S2))[0] < 5e-3


@pytest.mark.parametrize("dist", ["steep", "const:-60", "zero"])
def test_fused_gate_extremes(dist):
    """log alpha = -U(0,4) (every key's chunk decay beyond e^-60: all scores from the exact
    pairwise terms), a constant -60, and 0 (no decay)."""
    w = gi.Workload("t", B=1, H=2, T=200, dk=256, dv=512, dtype=torch.bfloat16, gate=gi.GATE_PER_KEY,
                    gate_dist=dist, s0_std=0.3)
    _check(w, seed=113)


def test_fused_mixed_steep_keys():
    """A few keys fall off a cliff inside a chunk (exact terms for those keys only), the rest are
    mild (tensor-core product); the steep keys sit in different CTAs' key slices."""
    w = gi.Workload("t", B=1, H=2, T=192, dk=256, dv=512, dtype=torch.bfloat16, gate=gi.GATE_PER_KEY, s0_std=0.1)
    x = gi.make_inputs(w, seed=114)
    x["log_g"][:, :, 70, ::9] = -80.0
    x["log_g"][:, 1, 150, 200] = -200.0
    x["log_g"][:, 0, 10:14, 64:70] = -20.0
    _check(w, seed=114, x=x)


def test_fused_in_place_state():
    w = gi.Workload("t", B=1, H=2, T=250, dk=256, dv=512, dtype=torch.bfloat16, gate=gi.GATE_PER_KEY, s0_std=0.3)
    x = gi.make_inputs(w, seed=115)
    c = _dev(x)
    S = c["S0"].clone()
    O, _ = gla.forward(c["q"], c["k"], c["v"], c["log_g"], S, ST=S, path=gla.GLA_PATH_FUSED)
    torch.cuda.synchronize()
    assert gla.gla_device_status() == 0
    Oref, STref = oracle.gla_forward(x["q"], x["k"], x["v"], x["log_g"], x["gate"], x["S0"])
    assert_close(to_np(O), Oref, torch.bfloat16, "O")
    assert_close(to_np(S), STref, torch.bfloat16, "ST (in place)")


def test_fused_deterministic_and_every_output_written():
    w = gi.Workload("t", B=2, H=2, T=190, dk=256, dv=512, dtype=torch.bfloat16, gate=gi.GATE_PER_KEY, s0_std=0.02)
    x = gi.make_inputs(w, seed=116)
    c = _dev(x)
    outs = []
    for _ in range(2):
        O = torch.full((2, 2, 190, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
        ST = torch.full((2, 2, 256, 512), float("nan"), device="cuda")
        gla.forward(c["q"], c["k"], c["v"], c["log_g"], c["S0"], O=O, ST=ST, path=gla.GLA_PATH_FUSED)
        torch.cuda.synchronize()
        assert torch.isfinite(O.float()).all() and torch.isfinite(ST).all()
        outs.append((O.clone(), ST.clone()))
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])


def test_fused_many_heads_several_waves():
    """More clusters than fit on the GPU at once (the grid runs in waves)."""
    w = gi.Workload("t", B=50, H=4, T=70, dk=256, dv=512, dtype=torch.bfloat16, gate=gi.GATE_PER_KEY, s0_std=0.02)
    x = gi.make_inputs(w, seed=117)
    c = _dev(x)
    O, ST = gla.forward(c["q"], c["k"], c["v"], c["log_g"], c["S0"], path=gla.GLA_PATH_FUSED)
    torch.cuda.synchronize()
    assert gla.gla_device_status() == 0
    heads = [(0, 0), (24, 3), (49, 2)]
    ref = oracle.gla_forward_rows(x["q"], x["k"], x["v"], x["log_g"], x["gate"], x["S0"], heads)
    for (b, h), (Oref, STref) in ref.items():
        assert_close(to_np(O[b, h]), Oref, torch.bfloat16, f"O[{b},{h}]")
        assert_close(to_np(ST[b, h]), STref, torch.bfloat16, f"ST[{b},{h}]")


def test_fused_plans_no_workspace():
    """The fused pass plans no workspace (nothing round-trips HBM); the 1.3B layer's head shape."""
    w = gi.Workload("t", B=1, H=1, T=130, dk=256, dv=512, dtype=torch.bfloat16, gate=gi.GATE_PER_KEY, s0_std=0.02)
    x = gi.make_inputs(w, seed=118)
    c = _dev(x)
    O = torch.empty(1, 1, 130, 512, dtype=torch.bfloat16, device="cuda")
    ST = torch.empty(1, 1, 256, 512, device="cuda")
    p = bnd.make_params(c["q"], c["k"], c["v"], c["log_g"], c["S0"], O, ST, path=gla.GLA_PATH_FUSED)
    assert bnd.gla_fwd_workspace_size(p) == 0
    bnd.gla_fwd_ex(p)
    torch.cuda.synchronize()
    Oref, STref = oracle.gla_forward(x["q"], x["k"], x["v"], x["log_g"], x["gate"], x["S0"])
    assert_close(to_np(O), Oref, torch.bfloat16, "O")
    assert_close(to_np(ST), STref, torch.bfloat16, "ST")


def test_fused_full_gla_1p3b_sampled():
    """The 1.3B-shaped layer at full size through the fused pass, sampled heads."""
    w = gi.WORKLOADS["gla_1p3b"]
    x = gi.make_inputs(w, seed=0)
    c = _dev(x)
    O, ST = gla.forward(c["q"], c["k"], c["v"], c["log_g"], c["S0"], path=gla.GLA_PATH_FUSED)
    torch.cuda.synchronize()
    assert gla.gla_device_status() == 0
    ref = oracle.gla_forward_rows(x["q"], x["k"], x["v"], x["log_g"], x["gate"], x["S0"], [(0, 0), (7, 3)])
    for (b, h), (Oref, STref) in ref.items():
        assert_close(to_np(O[b, h]), Oref, torch.bfloat16, f"O[{b},{h}]")
        assert_close(to_np(ST[b, h]), STref, torch.bfloat16, f"ST[{b},{h}]")
