"""gla_fwd_host: the pass with host tensors, copied in slices that overlap
with the compute. Slicing changes only which (b, h) pairs share a launch, and
every (b, h) pair is an independent problem, so where the plan does not split
the sequence the result must equal the device-pointer path bit for bit; the
larger case is held to the oracle instead. The argument checks run on the CPU."""
import pytest
import torch

import oracle
import chunkwise_gated_linear_gla_gb300 as gla
from chunkwise_gated_linear_gla_gb300 import binding as bnd
from chunkwise_gated_linear_gla_gb300 import build as gbuild
from chunkwise_gated_linear_gla_gb300 import inputs as gi

from _util import assert_close, to_np


def _host_run(x, w, slice_bytes, pinned=True, want_state=True, in_place=False, path=bnd.GLA_PATH_AUTO):
    def h(t):
        return None if t is None else (t.pin_memory() if pinned else t.clone())
    q, k, v, g = h(x["q"]), h(x["k"]), h(x["v"]), h(x["log_g"])
    S0 = h(x["S0"])
    O = torch.full((w.B, w.H, w.T, w.dv), float("nan"), dtype=w.dtype)
    if pinned:
        O = O.pin_memory()
    ST = None
    if in_place:
        ST = S0
    elif want_state:
        ST = torch.full((w.B, w.H, w.dk, w.dv), float("nan"), dtype=torch.float32)
        if pinned:
            ST = ST.pin_memory()
    p = bnd.make_params(q, k, v, g, S0, O, ST, gate=x["gate"], path=path)
    bnd.gla_fwd_host(p, slice_bytes)
    assert gla.gla_device_status() == 0
    return O, ST


def _device_run(x, w, want_state=True, path=bnd.GLA_PATH_AUTO):
    c = {n: (t.cuda() if isinstance(t, torch.Tensor) else t) for n, t in x.items()}
    O, ST = gla.forward(c["q"], c["k"], c["v"], c["log_g"], c["S0"], gate=x["gate"], want_state=want_state,
                        path=path)
    torch.cuda.synchronize()
    return O.cpu(), None if ST is None else ST.cpu()


def _unit_bytes(w):
    e = 2 if w.dtype == torch.bfloat16 else 4
    g = w.T * w.dk * 4 if w.gate == gi.GATE_PER_KEY else w.T * 4 if w.gate == gi.GATE_TOKEN_SCALAR else 0
    return 2 * w.T * w.dk * e + 2 * w.T * w.dv * e + g + 2 * w.dk * w.dv * 4


CASES = [
    # name, workload, slices wanted (sets slice_bytes)
    ("batch slices, ragged tail", gi.Workload("t", B=3, H=2, T=200, dk=64, dv=128, dtype=torch.bfloat16,
                                               gate=gi.GATE_PER_KEY, s0_std=0.02), 2),
    ("one slice per batch row", gi.Workload("t", B=4, H=2, T=130, dk=128, dv=256, dtype=torch.bfloat16,
                                             gate=gi.GATE_PER_KEY, s0_std=0.02), 4),
    ("head slices, scalar gate", gi.Workload("t", B=1, H=5, T=300, dk=128, dv=128, dtype=torch.bfloat16,
                                              gate=gi.GATE_HEAD_SCALAR, s0_std=0.02), 3),
    ("head slices, per-token gate", gi.Workload("t", B=1, H=6, T=333, dk=128, dv=128, dtype=torch.bfloat16,
                                                 gate=gi.GATE_TOKEN_SCALAR, s0_std=0.02), 4),
    ("head slices of two rows, scalar gate", gi.Workload("t", B=2, H=4, T=100, dk=64, dv=128,
                                                          dtype=torch.bfloat16, gate=gi.GATE_HEAD_SCALAR,
                                                          s0_std=0.02), 8),
    ("ungated, zero S0", gi.Workload("t", B=2, H=3, T=257, dk=128, dv=128, dtype=torch.bfloat16,
                                     gate=gi.GATE_NONE), 3),
    ("fp32 CUDA-core path", gi.Workload("t", B=2, H=2, T=70, dk=64, dv=64, dtype=torch.float32,
                                        gate=gi.GATE_PER_KEY, qkv_scale="q", s0_std=0.02), 4),
    ("single slice", gi.Workload("t", B=2, H=2, T=64, dk=64, dv=128, dtype=torch.bfloat16,
                                 gate=gi.GATE_PER_KEY, s0_std=0.02), 1),
]


@pytest.mark.gpu
@pytest.mark.parametrize("name,w,nslices", CASES, ids=[c[0] for c in CASES])
def test_host_equals_device_path(name, w, nslices):
    gbuild.build()
    x = gi.make_inputs(w, seed=21)
    units = w.B * w.H
    sb = 0 if nslices == 1 else -(-units * _unit_bytes(w) // nslices)
    O, ST = _host_run(x, w, sb)
    Od, STd = _device_run(x, w)
    assert torch.equal(O, Od), name
    assert torch.equal(ST, STd), name


@pytest.mark.gpu
def test_host_pageable_no_state_and_in_place():
    gbuild.build()
    w = gi.Workload("t", B=3, H=2, T=150, dk=128, dv=128, dtype=torch.bfloat16, gate=gi.GATE_PER_KEY,
                    s0_std=0.02)
    x = gi.make_inputs(w, seed=22)
    sb = -(-w.B * w.H * _unit_bytes(w) // 3)
    Od, STd = _device_run(x, w)
    O, _ = _host_run(x, w, sb, pinned=False, want_state=False)
    assert torch.equal(O, Od)
    # ST == S0: the final state overwrites the initial one in host memory
    O2, ST2 = _host_run(x, w, sb, in_place=True)
    assert torch.equal(O2, Od)
    assert torch.equal(ST2, STd)


@pytest.mark.gpu
def test_host_zero_length():
    gbuild.build()
    w = gi.Workload("t", B=2, H=3, T=0, dk=64, dv=128, dtype=torch.bfloat16, gate=gi.GATE_PER_KEY, s0_std=0.5)
    x = gi.make_inputs(w, seed=23)
    _, ST = _host_run(x, w, 1)
    assert torch.equal(ST, x["S0"])
    w0 = w.with_(s0_std=0.0)
    x0 = gi.make_inputs(w0, seed=23)
    _, ST0 = _host_run(x0, w0, 1)
    assert torch.count_nonzero(ST0) == 0


@pytest.mark.gpu
def test_host_default_slicing_against_oracle():
    """Default slicing of a 50 MB batch: slices of two rows, one row and two heads,
    each planning its own sequence split."""
    gbuild.build()
    oracle.build()
    w = gi.Workload("t", B=4, H=4, T=2048, dk=128, dv=128, dtype=torch.bfloat16, gate=gi.GATE_PER_KEY,
                    s0_std=0.02)
    x = gi.make_inputs(w, seed=24)
    O, ST = _host_run(x, w, 0)
    Oref, STref = oracle.gla_forward(x["q"], x["k"], x["v"], x["log_g"], x["gate"], x["S0"])
    assert_close(to_np(O), Oref, torch.bfloat16, "O")
    assert_close(to_np(ST), STref, torch.bfloat16, "ST")


# ---------------------------------------------------------------- host-side checks (no GPU)

def _params(**kw):
    p = bnd.gla_fwd_params()
    base = dict(q=0x10000, k=0x20000, v=0x30000, log_g=0x40000, S0=None, O=0x50000, ST=None,
                B=1, H=1, T=64, dk=64, dv=64, chunk=64, dtype=bnd.GLA_BF16,
                gate=bnd.GLA_GATE_PER_KEY, workspace=None, workspace_bytes=0,
                force_segments=0, path=bnd.GLA_PATH_AUTO)
    base.update(kw)
    for k, v in base.items():
        setattr(p, k, v)
    return p


BAD_HOST = [
    ("null q", dict(q=None), bnd.GLA_ERR_INVALID_ARG),
    ("null O", dict(O=None), bnd.GLA_ERR_INVALID_ARG),
    ("B=0", dict(B=0), bnd.GLA_ERR_INVALID_ARG),
    ("dk not /16", dict(dk=40), bnd.GLA_ERR_INVALID_ARG),
    ("per-key gate without log_g", dict(log_g=None), bnd.GLA_ERR_INVALID_ARG),
    ("O overlaps v", dict(O=0x30000 + 64), bnd.GLA_ERR_INVALID_ARG),
    ("ST overlaps k", dict(ST=0x20000), bnd.GLA_ERR_INVALID_ARG),
    ("ST partially overlaps S0", dict(S0=0x100000, ST=0x100000 + 256), bnd.GLA_ERR_INVALID_ARG),
    ("bad gate", dict(gate=9), bnd.GLA_ERR_INVALID_ARG),
    ("chunk 32", dict(chunk=32), bnd.GLA_ERR_UNSUPPORTED),
    ("tensor path with fp32", dict(dtype=bnd.GLA_FP32, path=bnd.GLA_PATH_TENSOR), bnd.GLA_ERR_UNSUPPORTED),
]


@pytest.mark.parametrize("name,kw,want", BAD_HOST, ids=[b[0] for b in BAD_HOST])
def test_host_rejects_before_any_copy(name, kw, want):
    gbuild.build()
    assert bnd.gla_fwd_host(_params(**kw), 0, stream=0, check=False) == want


def test_host_release_without_use():
    gbuild.build()
    # nothing was staged on this device (or there is no device): nothing to give back
    s = bnd.gla_host_release(check=False)
    assert s in (bnd.GLA_OK, bnd.GLA_ERR_CUDA)
    if torch.cuda.is_available():
        assert s == bnd.GLA_OK
