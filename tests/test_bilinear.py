"""The bilinear gate G_t = alpha_t^T beta_t ("Gated Linear Attention
Transformers with Hardware-Efficient Training", §4.1 Table 1, DFW row) against
the fp64 oracle (pinned in test_oracle_pins.py), on both paths:

* the CUDA-core path (fp32 inputs, and bf16 shapes outside the tensor path):
  fp32 arithmetic throughout, so fp32 inputs hold 1e-5;
* the tensor path (bf16, dk in {64, 128, 256}, dv a multiple of 128): the
  chunkwise form of the paper's appendix on the general formulation, one
  reference per chunk at its end, held to the bf16 contract (5e-3 / 1e-2).
  Heads whose in-chunk value decay leaves e^60 are flagged by the value prep
  and computed by the CUDA-core pass in the same call."""
import numpy as np
import pytest
import torch

import oracle
import chunkwise_gated_linear_gla_gb300 as gla
from chunkwise_gated_linear_gla_gb300 import binding as bnd
from chunkwise_gated_linear_gla_gb300 import build as gbuild
from chunkwise_gated_linear_gla_gb300 import inputs as gi

from _util import assert_close, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    gbuild.build()
    oracle.build()


def _dev(t):
    return None if t is None else t.cuda()


def _run(x, path=gla.GLA_PATH_AUTO):
    O, ST = gla.forward(_dev(x["q"]), _dev(x["k"]), _dev(x["v"]), _dev(x["log_g"]), _dev(x["S0"]),
                        gate=gi.GATE_BILINEAR, path=path, log_b=_dev(x["log_b"]))
    torch.cuda.synchronize()
    assert gla.gla_device_status() == 0
    return O, ST


def _check(w, seed):
    x = gi.make_inputs(w, seed=seed)
    O, ST = _run(x)
    Oref, STref = oracle.gla_forward(x["q"], x["k"], x["v"], x["log_g"], gi.GATE_BILINEAR, x["S0"], log_b=x["log_b"])
    assert_close(to_np(O), Oref, w.dtype, "O")
    assert_close(to_np(ST), STref, w.dtype, "ST")


@pytest.mark.parametrize("T", [1, 16, 17, 100])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_bilinear_ragged(T, dtype):
    w = gi.Workload("t", B=2, H=2, T=T, dk=64, dv=80, dtype=dtype, gate=gi.GATE_BILINEAR, s0_std=0.3,
                    qkv_scale="q" if dtype == torch.float32 else "all")
    _check(w, seed=70 + T)


@pytest.mark.parametrize("dk,dv", [(128, 128), (256, 512), (32, 48)])
def test_bilinear_head_shapes(dk, dv):
    w = gi.Workload("t", B=1, H=2, T=150, dk=dk, dv=dv, dtype=torch.bfloat16, gate=gi.GATE_BILINEAR, s0_std=0.02)
    _check(w, seed=71)


@pytest.mark.parametrize("dist", ["steep", "const:-60"])
def test_bilinear_extreme_gates(dist):
    w = gi.Workload("t", B=1, H=2, T=90, dk=64, dv=64, dtype=torch.float32, gate=gi.GATE_BILINEAR,
                    gate_dist=dist, s0_std=0.2, qkv_scale="q")
    _check(w, seed=72)


def test_bilinear_with_unit_beta_is_the_per_key_gate():
    w = gi.Workload("t", B=2, H=2, T=120, dk=64, dv=64, dtype=torch.float32, gate=gi.GATE_BILINEAR, s0_std=0.2,
                    qkv_scale="q")
    x = gi.make_inputs(w, seed=73)
    x["log_b"] = torch.zeros_like(x["log_b"])
    O1, S1 = _run(x)
    O2, S2 = gla.forward(_dev(x["q"]), _dev(x["k"]), _dev(x["v"]), _dev(x["log_g"]), _dev(x["S0"]),
                         gate=gi.GATE_PER_KEY, path=gla.GLA_PATH_SIMT)
    torch.cuda.synchronize()
    assert torch.equal(O1, O2) and torch.equal(S1, S2)


def test_bilinear_host_entry_in_slices():
    w = gi.Workload("t", B=3, H=2, T=70, dk=64, dv=128, dtype=torch.bfloat16, gate=gi.GATE_BILINEAR, s0_std=0.1)
    x = gi.make_inputs(w, seed=74)
    Od, Sd = _run(x)
    h = {n: (None if x[n] is None else x[n].pin_memory()) for n in ("q", "k", "v", "log_g", "log_b", "S0")}
    O = torch.empty(Od.shape, dtype=Od.dtype).pin_memory()
    ST = torch.empty(Sd.shape, dtype=Sd.dtype).pin_memory()
    p = bnd.make_params(h["q"], h["k"], h["v"], h["log_g"], h["S0"], O, ST, log_b=h["log_b"])
    per_unit = 70 * (2 * 64 * 2 + 2 * 128 * 2 + 64 * 4 + 128 * 4) + 2 * 64 * 128 * 4
    bnd.gla_fwd_host(p, per_unit * 2)
    assert torch.equal(O, Od.cpu()) and torch.equal(ST, Sd.cpu())


def test_bilinear_full_layer_sampled():
    w = gi.WORKLOADS["bilinear"]
    x = gi.make_inputs(w, seed=0)
    O, ST = _run(x)
    ref = oracle.gla_forward_rows(x["q"], x["k"], x["v"], x["log_g"], gi.GATE_BILINEAR, x["S0"], [(0, 0), (7, 3)],
                                  log_b=x["log_b"])
    for (b, h), (Oref, STref) in ref.items():
        assert_close(to_np(O[b, h]), Oref, torch.bfloat16, f"O[{b},{h}]")
        assert_close(to_np(ST[b, h]), STref, torch.bfloat16, f"ST[{b},{h}]")


# ---------------------------------------------------------------- tensor path

def _stage_names(x):
    dev = {n: _dev(x[n]) for n in ("q", "k", "v", "log_g", "log_b", "S0")}
    O = torch.empty(x["v"].shape, dtype=x["v"].dtype, device="cuda")
    ST = torch.empty(x["q"].shape[:2] + (x["q"].shape[-1], x["v"].shape[-1]), device="cuda")
    p = bnd.make_params(dev["q"], dev["k"], dev["v"], dev["log_g"], dev["S0"], O, ST, log_b=dev["log_b"])
    return [bnd.gla_fwd_stage_name(p, i) for i in range(bnd.gla_fwd_num_stages(p))]


def _check_tensor(w, seed, x=None):
    x = x if x is not None else gi.make_inputs(w, seed=seed)
    O, ST = _run(x, path=gla.GLA_PATH_TENSOR)
    Oref, STref = oracle.gla_forward(x["q"], x["k"], x["v"], x["log_g"], gi.GATE_BILINEAR, x["S0"], log_b=x["log_b"])
    assert_close(to_np(O), Oref, torch.bfloat16, "O")
    assert_close(to_np(ST), STref, torch.bfloat16, "ST")
    return O, ST


def test_bilinear_tensor_plan():
    w = gi.Workload("t", B=1, H=2, T=100, dk=64, dv=128, dtype=torch.bfloat16, gate=gi.GATE_BILINEAR)
    assert _stage_names(gi.make_inputs(w, seed=0)) == ["gla_chunk_prep", "gla_value_prep", "gla_chunk_fwd",
                                                       "gla_fwd_simt_flagged"]


@pytest.mark.parametrize("T", [1, 63, 64, 65, 200, 1000])
def test_bilinear_tensor_ragged(T):
    """Several chunks and a ragged tail; three dv tiles; S0 given."""
    w = gi.Workload("t", B=2, H=2, T=T, dk=64, dv=384, dtype=torch.bfloat16, gate=gi.GATE_BILINEAR, s0_std=0.3)
    _check_tensor(w, seed=80 + T)


@pytest.mark.parametrize("dk", [64, 128, 256])
@pytest.mark.parametrize("s0", [0.0, 0.02])
def test_bilinear_tensor_head_shapes(dk, s0):
    w = gi.Workload("t", B=1, H=3, T=333, dk=dk, dv=256, dtype=torch.bfloat16, gate=gi.GATE_BILINEAR, s0_std=s0)
    _check_tensor(w, seed=81 + dk)


def test_bilinear_tensor_unit_beta_is_the_per_key_pass():
    """beta = 1: V^ = V, gamma' = 1 and every output factor is exactly 1, so the bilinear
    instantiation must give the per-key tensor pass's bits."""
    w = gi.Workload("t", B=2, H=2, T=500, dk=128, dv=256, dtype=torch.bfloat16, gate=gi.GATE_BILINEAR, s0_std=0.1)
    x = gi.make_inputs(w, seed=82)
    x["log_b"] = torch.zeros_like(x["log_b"])
    O1, S1 = _run(x, path=gla.GLA_PATH_TENSOR)
    O2, S2 = gla.forward(_dev(x["q"]), _dev(x["k"]), _dev(x["v"]), _dev(x["log_g"]), _dev(x["S0"]),
                         gate=gi.GATE_PER_KEY, path=gla.GLA_PATH_TENSOR)
    torch.cuda.synchronize()
    assert torch.equal(O1, O2) and torch.equal(S1, S2)


@pytest.mark.parametrize("lb", [-0.9, -0.95])
def test_bilinear_tensor_near_the_guard(lb):
    """A constant log beta whose 64-row chunk sum (57.6, 60.8) sits just inside or just past
    e^60: the first runs on the tensor pass with output factors up to e^57, the second is
    flagged and computed by the CUDA-core pass."""
    w = gi.Workload("t", B=1, H=2, T=300, dk=64, dv=128, dtype=torch.bfloat16, gate=gi.GATE_BILINEAR, s0_std=0.2)
    x = gi.make_inputs(w, seed=83)
    x["log_b"] = torch.full_like(x["log_b"], lb)
    _check_tensor(w, 0, x)


def test_bilinear_tensor_mixed_heads_in_place_state():
    """One call where heads 0 and 3 have steep value gates (flagged, CUDA-core pass) and the
    others mild ones (tensor pass), with S_T written over S0 in place."""
    w = gi.Workload("t", B=2, H=2, T=260, dk=128, dv=256, dtype=torch.bfloat16, gate=gi.GATE_BILINEAR, s0_std=0.3)
    x = gi.make_inputs(w, seed=84)
    g = torch.Generator().manual_seed(85)
    x["log_b"][0, 0] = -4 * torch.rand(x["log_b"][0, 0].shape, generator=g)
    x["log_b"][1, 1] = -4 * torch.rand(x["log_b"][1, 1].shape, generator=g)
    Oref, STref = oracle.gla_forward(x["q"], x["k"], x["v"], x["log_g"], gi.GATE_BILINEAR, x["S0"], log_b=x["log_b"])
    S = _dev(x["S0"]).clone()
    O, ST = gla.forward(_dev(x["q"]), _dev(x["k"]), _dev(x["v"]), _dev(x["log_g"]), S, gate=gi.GATE_BILINEAR,
                        path=gla.GLA_PATH_TENSOR, log_b=_dev(x["log_b"]), ST=S)
    torch.cuda.synchronize()
    assert gla.gla_device_status() == 0
    assert ST.data_ptr() == S.data_ptr()
    assert_close(to_np(O), Oref, torch.bfloat16, "O")
    assert_close(to_np(ST), STref, torch.bfloat16, "ST")
