"""The torch.autograd wrapper (gla_attention): a scalar loss through O and S_T gives, by
loss.backward(), exactly the gradients of the gla_bwd call with dL/dO and dL/dS_T (cast to
the inputs' dtypes), and those agree with the fp64 oracle's adjoint."""
import numpy as np
import pytest
import torch

import oracle
import chunkwise_gated_linear_gla_gb300 as gla
from chunkwise_gated_linear_gla_gb300 import build as gbuild
from chunkwise_gated_linear_gla_gb300 import inputs as gi

from _util import errors, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    gbuild.build()
    oracle.build()


@pytest.mark.parametrize("gate", [gi.GATE_PER_KEY, gi.GATE_HEAD_SCALAR, gi.GATE_TOKEN_SCALAR, gi.GATE_NONE])
def test_autograd_gives_the_backward_calls_gradients(gate):
    w = gi.Workload("t", B=2, H=2, T=200, dk=128, dv=128, dtype=torch.bfloat16, gate=gate, s0_std=0.2)
    x = gi.make_inputs(w, seed=21)
    leaf = lambda t: None if t is None else t.cuda().clone().requires_grad_()
    q, k, v, lg, S0 = leaf(x["q"]), leaf(x["k"]), leaf(x["v"]), leaf(x["log_g"]), leaf(x["S0"])
    O, ST = gla.gla_attention(q, k, v, lg, S0, gate=x["gate"])
    g = torch.Generator().manual_seed(22)
    W = torch.randn(O.shape, generator=g).to(torch.bfloat16).cuda()
    U = (torch.randn(ST.shape, generator=g) * 0.1).cuda()
    loss = (O.float() * W.float()).sum() + (ST * U).sum()
    loss.backward()
    torch.cuda.synchronize()
    assert gla.gla_device_status() == 0
    d = lambda t: None if t is None else t.detach()
    ref = gla.backward(d(q), d(k), d(v), d(lg), d(S0), W, U, gate=x["gate"])
    torch.cuda.synchronize()
    assert q.grad.dtype == torch.bfloat16 and torch.equal(q.grad, ref[0].to(torch.bfloat16))
    assert torch.equal(k.grad, ref[1].to(torch.bfloat16)) and torch.equal(v.grad, ref[2].to(torch.bfloat16))
    if lg is not None:
        assert lg.grad.dtype == torch.float32 and torch.equal(lg.grad, ref[3])
    assert torch.equal(S0.grad, ref[4])
    # and against the oracle (the bf16 cast of dq, dk, dv adds one rounding to the chunk form's bar)
    oref = oracle.gla_backward(x["q"], x["k"], x["v"], x["log_g"], x["gate"], x["S0"], W.cpu(), U.cpu())
    for name, a, r in (("dq", q.grad, oref[0]), ("dk", k.grad, oref[1]), ("dv", v.grad, oref[2]),
                       ("dS0", S0.grad, oref[4])):
        rf, ma = errors(to_np(a), r)
        assert rf <= 6e-3 and ma <= 1.2e-2, (name, rf, ma)


def test_autograd_loss_through_the_state_only():
    """O unused: its gradient is zero, and the wrapper still runs the backward."""
    w = gi.Workload("t", B=1, H=2, T=130, dk=128, dv=128, dtype=torch.bfloat16, gate=gi.GATE_PER_KEY, s0_std=0.2)
    x = gi.make_inputs(w, seed=23)
    leaf = lambda t: t.cuda().clone().requires_grad_()
    q, k, v, lg, S0 = leaf(x["q"]), leaf(x["k"]), leaf(x["v"]), leaf(x["log_g"]), leaf(x["S0"])
    _, ST = gla.gla_attention(q, k, v, lg, S0)
    ST.sum().backward()
    torch.cuda.synchronize()
    oref = oracle.gla_backward(x["q"], x["k"], x["v"], x["log_g"], x["gate"], x["S0"],
                               torch.zeros((1, 2, 130, 128), dtype=torch.bfloat16), torch.ones((1, 2, 128, 128)))
    rf, _ = errors(to_np(v.grad), oref[2])
    assert rf <= 6e-3, rf
    assert np.all(to_np(q.grad) == 0)   # q only reaches O
