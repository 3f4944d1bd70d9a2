"""The failure path of the kernels' bounded waits, exercised without a fault:
a one-warp kernel waits on an mbarrier nothing arrives on, gives up after a
short limit, records the timeout in the device status word and returns. The
host then reads GLA_ERR_TIMEOUT, and the next ordinary call works."""
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


def _ordinary_call_matches_oracle(seed):
    w = gi.Workload("t", B=1, H=2, T=130, dk=128, dv=128, dtype=torch.bfloat16, gate=gi.GATE_PER_KEY, s0_std=0.1)
    x = gi.make_inputs(w, seed=seed)
    c = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    O, ST = gla.forward(c["q"], c["k"], c["v"], c["log_g"], c["S0"])
    torch.cuda.synchronize()
    assert gla.gla_device_status() == bnd.GLA_OK
    Oref, STref = oracle.gla_forward(x["q"], x["k"], x["v"], x["log_g"], x["gate"], x["S0"])
    assert_close(to_np(O), Oref, torch.bfloat16, "O")
    assert_close(to_np(ST), STref, torch.bfloat16, "ST")


def test_wait_that_runs_out_reports_timeout_and_context_stays_usable():
    torch.cuda.synchronize()
    assert gla.gla_device_status() == bnd.GLA_OK
    s = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s)
    bnd.gla_selftest_bounded_wait(1000)            # 1 ms, nothing arrives
    e1.record(s)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1)
    assert 0.9 <= ms < 1000.0, ms                  # it waited its limit, then returned
    assert gla.gla_device_status() == bnd.GLA_ERR_TIMEOUT
    assert gla.gla_device_status() == bnd.GLA_OK   # reading the word clears it
    _ordinary_call_matches_oracle(seed=71)


def test_wait_that_is_satisfied_reports_nothing():
    bnd.gla_selftest_bounded_wait(1000, arrive=True)
    torch.cuda.synchronize()
    assert gla.gla_device_status() == bnd.GLA_OK


def test_timeout_then_ordinary_calls_in_a_row():
    for i in range(3):
        bnd.gla_selftest_bounded_wait(200)
        assert gla.gla_device_status() == bnd.GLA_ERR_TIMEOUT
        _ordinary_call_matches_oracle(seed=72 + i)
