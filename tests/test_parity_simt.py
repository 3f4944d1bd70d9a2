"""GPU parity of the CUDA-core path (fp32 and bf16) against the fp64 oracle,
element by element, through the C ABI."""
import pytest
import torch

import oracle
import chunkwise_gated_linear_gla_gb300 as gla
from chunkwise_gated_linear_gla_gb300 import inputs as gi
from chunkwise_gated_linear_gla_gb300 import build as gbuild

from _util import assert_close, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    gbuild.build()
    oracle.build()


def _run(w, seed=0, path=gla.GLA_PATH_SIMT, **kw):
    x = gi.make_inputs(w, seed=seed)
    d = lambda t: None if t is None else t.cuda()
    O, ST = gla.forward(d(x["q"]), d(x["k"]), d(x["v"]), d(x["log_g"]), d(x["S0"]),
                        gate=x["gate"], path=path, **kw)
    torch.cuda.synchronize()
    assert gla.gla_device_status() == 0
    Oref, STref = oracle.gla_forward(x["q"], x["k"], x["v"], x["log_g"], x["gate"], x["S0"])
    return x, to_np(O), to_np(ST), Oref, STref


def _run_any(w, seed=0, path=gla.GLA_PATH_SIMT):
    """_run for every gate mode, the bilinear gate's log beta included."""
    x = gi.make_inputs(w, seed=seed)
    d = lambda t: None if t is None else t.cuda()
    O, ST = gla.forward(d(x["q"]), d(x["k"]), d(x["v"]), d(x["log_g"]), d(x["S0"]),
                        gate=x["gate"], path=path, log_b=d(x.get("log_b")))
    torch.cuda.synchronize()
    assert gla.gla_device_status() == 0
    Oref, STref = oracle.gla_forward(x["q"], x["k"], x["v"], x["log_g"], x["gate"], x["S0"], log_b=x.get("log_b"))
    return x, to_np(O), to_np(ST), Oref, STref


def test_fp32_workload_full_size():
    """The fp32 workload (B=1, H=2, T=256, dk=dv=64, per-key gate) at its full size."""
    w = gi.WORKLOADS["fp32_small"]
    x, O, ST, Oref, STref = _run(w, path=gla.GLA_PATH_AUTO)
    assert_close(O, Oref, torch.float32, "O")
    assert_close(ST, STref, torch.float32, "ST")


@pytest.mark.parametrize("gate", [gi.GATE_NONE, gi.GATE_HEAD_SCALAR, gi.GATE_PER_KEY, gi.GATE_TOKEN_SCALAR])
@pytest.mark.parametrize("T", [1, 15, 16, 63, 65, 200])
def test_fp32_gates_ragged(gate, T):
    w = gi.Workload("t", B=2, H=3, T=T, dk=32, dv=80, dtype=torch.float32, gate=gate, s0_std=0.1)
    x, O, ST, Oref, STref = _run(w, seed=T)
    assert_close(O, Oref, torch.float32, "O")
    assert_close(ST, STref, torch.float32, "ST")


@pytest.mark.parametrize("gate", [gi.GATE_NONE, gi.GATE_HEAD_SCALAR, gi.GATE_PER_KEY, gi.GATE_TOKEN_SCALAR])
def test_bf16_simt(gate):
    w = gi.Workload("t", B=1, H=2, T=130, dk=64, dv=96, dtype=torch.bfloat16, gate=gate, s0_std=0.02)
    x, O, ST, Oref, STref = _run(w, seed=3)
    assert_close(O, Oref, torch.bfloat16, "O")
    assert_close(ST, STref, torch.bfloat16, "ST")


def test_fp32_steep_gate_is_finite_and_exact():
    """log alpha ~ -U(0,4) per entry: cumulative products underflow fast; the
    pairwise log-space intra scores keep every factor <= 1."""
    w = gi.Workload("t", B=1, H=2, T=100, dk=64, dv=64, dtype=torch.float32,
                    gate=gi.GATE_PER_KEY, gate_dist="steep", s0_std=0.5)
    x, O, ST, Oref, STref = _run(w, seed=5)
    assert_close(O, Oref, torch.float32, "O")
    assert_close(ST, STref, torch.float32, "ST")


def test_fp32_dk256_dv_tail():
    w = gi.Workload("t", B=1, H=1, T=70, dk=256, dv=144, dtype=torch.float32, gate=gi.GATE_PER_KEY, s0_std=0.1)
    x, O, ST, Oref, STref = _run(w, seed=7)
    assert_close(O, Oref, torch.float32, "O")
    assert_close(ST, STref, torch.float32, "ST")


@pytest.mark.parametrize("gate", [gi.GATE_NONE, gi.GATE_HEAD_SCALAR, gi.GATE_PER_KEY, gi.GATE_TOKEN_SCALAR,
                                  gi.GATE_BILINEAR])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_wide_keys(gate, dtype):
    """Keys wider than 256 (8-row chunks, 32 state columns per CTA): dk = 320 with a
    ragged last chunk and a ragged last dv tile, every gate mode, both dtypes."""
    w = gi.Workload("t", B=1, H=2, T=45, dk=320, dv=80, dtype=dtype, gate=gate, s0_std=0.05)
    x, O, ST, Oref, STref = _run_any(w, seed=11, path=gla.GLA_PATH_AUTO)
    assert_close(O, Oref, dtype, "O")
    assert_close(ST, STref, dtype, "ST")


@pytest.mark.parametrize("dk,T", [(512, 70), (768, 17)])
def test_widest_keys(dk, T):
    """dk = 512 (one head of the 340M model's ablation with a single head: d_model 1024,
    dk = d/2, dv = d) and the widest supported, dk = 768, with a steep gate."""
    w = gi.Workload("t", B=1, H=1, T=T, dk=dk, dv=64, dtype=torch.float32, gate=gi.GATE_PER_KEY,
                    gate_dist="steep", s0_std=0.1)
    x, O, ST, Oref, STref = _run_any(w, seed=dk, path=gla.GLA_PATH_AUTO)
    assert_close(O, Oref, torch.float32, "O")
    assert_close(ST, STref, torch.float32, "ST")


def test_wide_heads_workload_sampled():
    """The wide-head workload (B=8, H=2, T=2048, dk=512, dv=1024, bf16, per-key gate) at
    its full size, in the launch configuration the bench times (the tensor path in two
    key halves), checked on two sampled heads the oracle computes alone."""
    w = gi.WORKLOADS["gla_wide_heads"]
    x = gi.make_inputs(w, seed=0)
    d = lambda t: None if t is None else t.cuda()
    O, ST = gla.forward(d(x["q"]), d(x["k"]), d(x["v"]), d(x["log_g"]), d(x["S0"]), gate=x["gate"])
    torch.cuda.synchronize()
    assert gla.gla_device_status() == 0
    ref = oracle.gla_forward_rows(x["q"], x["k"], x["v"], x["log_g"], x["gate"], x["S0"], [(0, 0), (7, 1)])
    for (b, h), (Oref, STref) in ref.items():
        assert_close(to_np(O[b, h]), Oref, torch.bfloat16, f"O[{b},{h}]")
        assert_close(to_np(ST[b, h]), STref, torch.bfloat16, f"ST[{b},{h}]")


def test_wide_keys_rejected_on_tensor_path_and_beyond_768():
    """dk = 384 has no tensor path (dk = 512 does, in key halves); dk = 784 none at all."""
    w = gi.Workload("t", B=1, H=1, T=8, dk=384, dv=128, dtype=torch.bfloat16, gate=gi.GATE_PER_KEY)
    x = gi.make_inputs(w, seed=0)
    d = lambda t: None if t is None else t.cuda()
    with pytest.raises(RuntimeError, match="UNSUPPORTED"):
        gla.forward(d(x["q"]), d(x["k"]), d(x["v"]), d(x["log_g"]), None, gate=x["gate"], path=gla.GLA_PATH_TENSOR)
    w = w.with_(dk=784)
    x = gi.make_inputs(w, seed=0)
    with pytest.raises(RuntimeError, match="UNSUPPORTED"):
        gla.forward(d(x["q"]), d(x["k"]), d(x["v"]), d(x["log_g"]), None, gate=x["gate"])


def test_empty_sequence_copies_state():
    S0 = torch.randn(1, 2, 32, 48, device="cuda")
    q = torch.empty(1, 2, 0, 32, device="cuda")
    v = torch.empty(1, 2, 0, 48, device="cuda")
    g = torch.empty(1, 2, 0, 32, device="cuda")
    O, ST = gla.forward(q, q, v, g, S0)
    torch.cuda.synchronize()
    assert O.shape == (1, 2, 0, 48)
    assert torch.equal(ST, S0)


def test_in_place_state_carry():
    """ST == S0 (the TBPTT carry): two half runs chained in place equal one run."""
    w = gi.Workload("t", B=1, H=2, T=96, dk=32, dv=64, dtype=torch.float32, gate=gi.GATE_PER_KEY, s0_std=0.3)
    x = gi.make_inputs(w, seed=11)
    c = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    S = c["S0"].clone()
    outs = []
    for sl in (slice(0, 40), slice(40, 96)):
        O = torch.empty((1, 2, sl.stop - sl.start, 64), device="cuda")
        gla.forward(c["q"][:, :, sl].contiguous(), c["k"][:, :, sl].contiguous(), c["v"][:, :, sl].contiguous(),
                    c["log_g"][:, :, sl].contiguous(), S, O=O, ST=S)
        outs.append(O)
    torch.cuda.synchronize()
    Oref, STref = oracle.gla_forward(x["q"], x["k"], x["v"], x["log_g"], x["gate"], x["S0"])
    assert_close(to_np(torch.cat(outs, dim=2)), Oref, torch.float32, "O")
    assert_close(to_np(S), STref, torch.float32, "ST")
