"""The bilinear gate G_t = alpha_t^T beta_t ("Gated Linear Attention
Transformers with Hardware-Efficient Training", §4.1 Table 1, DFW row) on the
CUDA-core path, against the fp64 oracle (pinned in test_oracle_pins.py).
Tolerances are those of the path: fp32 arithmetic throughout, so fp32 inputs
hold 1e-5 and bf16 inputs the bf16 output rounding (5e-3 / 1e-2)."""
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
