"""The backward pass with the bilinear gate G_t = alpha_t^T beta_t ("Gated Linear
Attention Transformers with Hardware-Efficient Training", §4.1 Table 1, DFW row)
against the fp64 adjoint of the oracle (pinned in test_oracle_bwd_pins.py), on
the CUDA-core path (fp32 arithmetic): every gradient, dL/dlog beta included."""
import numpy as np
import pytest
import torch

import oracle
import chunkwise_gated_linear_gla_gb300 as gla
from chunkwise_gated_linear_gla_gb300 import build as gbuild
from chunkwise_gated_linear_gla_gb300 import inputs as gi

from _util import errors, to_np

pytestmark = pytest.mark.gpu

REL_FRO, MAX_ABS = 2e-5, 2e-4


@pytest.fixture(scope="module", autouse=True)
def _built():
    gbuild.build()
    oracle.build()


def _rev(x):
    return np.flip(np.cumsum(np.flip(x, axis=2), axis=2), axis=2)


def _check(w, seed):
    x = gi.make_inputs(w, seed=seed)
    g = torch.Generator().manual_seed(seed + 1000)
    dO = torch.randn((w.B, w.H, w.T, w.dv), generator=g).to(w.dtype)
    dST = torch.randn((w.B, w.H, w.dk, w.dv), generator=g) * 0.1
    c = lambda t: None if t is None else t.cuda()
    got = gla.backward(c(x["q"]), c(x["k"]), c(x["v"]), c(x["log_g"]), c(x["S0"]), c(dO), c(dST),
                       log_b=c(x["log_b"]))
    torch.cuda.synchronize()
    assert gla.gla_device_status() == 0
    got = [to_np(t) for t in got]
    ref = oracle.gla_backward(x["q"], x["k"], x["v"], x["log_g"], gi.GATE_BILINEAR, x["S0"], dO, dST,
                              log_b=x["log_b"])
    for n, a, r in zip(["dq", "dk", "dv", "dS0"], [got[i] for i in (0, 1, 2, 4)], [ref[i] for i in (0, 1, 2, 4)]):
        assert np.all(np.isfinite(a)), n
        if np.abs(r).max() < 1e-30:
            # below fp32's range (dS0 under alpha = beta = e^-60 is about e^-120 |D|): zero in fp32
            assert np.abs(a).max() < 1e-30, n
            continue
        rf, ma = errors(a, r)
        assert rf <= REL_FRO and ma <= MAX_ABS, (n, rf, ma)
    # the gate gradients are reverse sums over tokens that can nearly cancel: each element
    # is held to 1e-5 times the same sums over the terms' absolute values
    q, k, v, do = to_np(x["q"]), to_np(x["k"]), to_np(x["v"]), to_np(dO)
    O, ST = oracle.gla_forward(x["q"], x["k"], x["v"], x["log_g"], gi.GATE_BILINEAR, x["S0"], log_b=x["log_b"])
    ta = np.abs(q * ref[0]) + np.abs(k * ref[1])
    tb = np.abs(O * do) + np.abs(v * ref[2])
    if w.T > 0:
        ta[:, :, -1] += np.sum(np.abs(to_np(dST) * ST), axis=-1)
        tb[:, :, -1] += np.sum(np.abs(to_np(dST) * ST), axis=-2)
    for n, a, r, t in (("dlog_g", got[3], ref[3], ta), ("dlog_b", got[5], ref[5], tb)):
        bound = 1e-5 * _rev(t) + 1e-30
        assert np.all(np.abs(a - r) <= bound), (n, np.abs(a - r).max(), bound.max())


@pytest.mark.parametrize("T", [1, 16, 17, 100])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_bwd_bilinear_ragged(T, dtype):
    w = gi.Workload("t", B=2, H=2, T=T, dk=64, dv=80, dtype=dtype, gate=gi.GATE_BILINEAR, s0_std=0.3)
    _check(w, seed=90 + T)


@pytest.mark.parametrize("dist", ["steep", "const:-60"])
def test_bwd_bilinear_extreme_gates(dist):
    """log alpha = log beta = -U(0,4), or a constant -60: every factor the sweep forms is
    exp of a non-positive number, so nothing overflows."""
    w = gi.Workload("t", B=1, H=2, T=70, dk=32, dv=48, dtype=torch.float32, gate=gi.GATE_BILINEAR,
                    gate_dist=dist, s0_std=0.3)
    _check(w, seed=95)


def test_bwd_bilinear_wide_head_bf16():
    """bf16 with dk = 256 and dv = 128 (the bilinear gate takes the CUDA-core path there too),
    several chunks."""
    w = gi.Workload("t", B=1, H=1, T=200, dk=256, dv=128, dtype=torch.bfloat16, gate=gi.GATE_BILINEAR,
                    s0_std=0.02)
    _check(w, seed=96)
