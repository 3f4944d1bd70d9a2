"""The backward pass (gla_bwd, CUDA cores, fp32) against the fp64 backward
oracle (tests/test_oracle_bwd_pins.py pins it), through the C ABI.

Tolerance. Every gradient is accumulated in fp32 from inputs that the oracle
sees exactly (bf16 values widened), with factors exp(x), x <= 0, so the error
is fp32 rounding of sums of at most T * (dk + dv) terms. dq, dk, dv and dS0 are
held to a relative Frobenius error of 2e-5 and a max-abs error of
2e-4 * max|ref| per tensor. The gate gradient is a sum of the terms
q (.) dq - k (.) dk (and rowsum(dST (.) S_T)) over later tokens, and over keys
and batch rows for the scalar gates; it can nearly cancel, so each element is
held to 1e-5 times the same sum taken over the terms' absolute values.

The split path (GLA_PATH_SPLIT; what AUTO takes for bf16 with dk = 64 or dv
not a multiple of 128) splits every operand that is not a bf16 input (the
chunk states, D, q (.) Lambda, k (.) Gamma) into hi + lo bf16 parts, so its
products keep about 16 mantissa bits (2^-16 ~ 1.5e-5 relative) with fp32
accumulation. It is held to relative Frobenius 5e-5 and max-abs
5e-4 * max|ref|. Its gate gradient, a sum of q (.) dq - k (.) dk in which dq
and dk carry that error relative to their own (possibly cancelling) terms, is
held over the whole tensor to relative Frobenius 2e-4 and max-abs
2e-3 * max|ref|.

The chunk form (GLA_PATH_TENSOR; what AUTO takes for bf16 with dk in
{128, 256} and dv a multiple of 128) computes like the forward pass: bf16
operands (q (.) Lambda, k (.) Gamma, the scores, the chunk states H and D,
dO V^T), fp32 accumulation. It is held to the forward's bf16 contract
(relative Frobenius 5e-3, max-abs 1e-2 * max|ref|) and, per element, to a
bound on the rounding: each term of a gradient is a product of at most five
bf16 roundings of exact values (for dv: k (.) Gamma twice, then D, itself a
sum of rounded q (.) Lambda times dO, rounded once more), so its relative
error is below 5 * 2^-9 < 2^-6, and the error of the element is below 2^-6
times the sum of its terms' absolute values. That sum is the oracle's
gradient of the absolute values of the inputs (every term is a product of
inputs with a non-negative decay coefficient). The gate gradient, a reverse
sum of q (.) dq - k (.) dk, is held to 2^-6 times the same sum taken over
|q| (.) |dq|abs + |k| (.) |dk|abs (and |dST| (.) |S_T|abs at the last token).
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import chunkwise_gated_linear_gla_gb300 as gla
from chunkwise_gated_linear_gla_gb300 import binding as bnd
from chunkwise_gated_linear_gla_gb300 import build as gbuild
from chunkwise_gated_linear_gla_gb300 import inputs as gi

from _util import errors, to_np

REL_FRO, MAX_ABS = 2e-5, 2e-4
TC_REL_FRO, TC_MAX_ABS = 5e-5, 5e-4
TC_GATE_REL_FRO, TC_GATE_MAX_ABS = 2e-4, 2e-3
CH_REL_FRO, CH_MAX_ABS = 5e-3, 1e-2
CH_TERM = 2.0 ** -6
AUTO, SIMT, SPLIT, TENSOR = bnd.GLA_PATH_AUTO, bnd.GLA_PATH_SIMT, bnd.GLA_PATH_SPLIT, bnd.GLA_PATH_TENSOR


def _kind(w, path):
    """Which form runs: "simt", "split" or "chunk" (inputs 16-byte aligned)."""
    if w.dtype != torch.bfloat16 or path == SIMT:
        return "simt"
    if path == SPLIT:
        return "split"
    if w.dk in (128, 256) and w.dv % 128 == 0 and w.T > 0 and w.gate != gi.GATE_BILINEAR:
        return "chunk"
    return "split" if w.dk in (64, 128, 256) else "simt"


def _tensor(w, path):
    return _kind(w, path) == "split"
GATES = [gi.GATE_NONE, gi.GATE_HEAD_SCALAR, gi.GATE_PER_KEY, gi.GATE_TOKEN_SCALAR]


def _inputs(w, seed, dst=True):
    x = gi.make_inputs(w, seed=seed)
    g = torch.Generator().manual_seed(seed + 1000)
    dO = torch.randn((w.B, w.H, w.T, w.dv), generator=g).to(w.dtype)
    dST = torch.randn((w.B, w.H, w.dk, w.dv), generator=g) * 0.1 if dst else None
    return x, dO, dST


def _gpu(x, dO, dST, path=AUTO):
    c = lambda t: None if t is None else t.cuda()
    out = gla.backward(c(x["q"]), c(x["k"]), c(x["v"]), c(x["log_g"]), c(x["S0"]), c(dO), c(dST), gate=x["gate"],
                       path=path)
    torch.cuda.synchronize()
    assert gla.gla_device_status() == 0
    return [None if t is None else to_np(t) for t in out]


def _abs(t):
    return None if t is None else t.abs()


def _mags(x, dO, dST):
    """Per element, the sum of the absolute values of its terms: the oracle's gradients of
    the inputs' absolute values under the same gates."""
    return oracle.gla_backward(_abs(x["q"]), _abs(x["k"]), _abs(x["v"]), x["log_g"], x["gate"], _abs(x["S0"]),
                               _abs(dO), _abs(dST))


def _gate_abs_sum(x, dST, ref, mag=False):
    """The gate gradient's reductions applied to the absolute values of its terms; with
    `mag`, ref holds the magnitude gradients (_mags) and the final state is taken on the
    inputs' absolute values too."""
    q, k = to_np(x["q"]), to_np(x["k"])
    terms = np.abs(q * ref[0]) + np.abs(k * ref[1])
    if dST is not None and q.shape[2] > 0:
        if mag:
            _, ST = oracle.gla_forward(_abs(x["q"]), _abs(x["k"]), _abs(x["v"]), x["log_g"], x["gate"],
                                       _abs(x["S0"]))
        else:
            _, ST = oracle.gla_forward(x["q"], x["k"], x["v"], x["log_g"], x["gate"], x["S0"])
        terms[:, :, -1] += np.sum(np.abs(to_np(dST) * ST), axis=-1)
    rev = np.flip(np.cumsum(np.flip(terms, axis=2), axis=2), axis=2)
    if x["gate"] == gi.GATE_TOKEN_SCALAR:
        return rev.sum(axis=-1)
    if x["gate"] == gi.GATE_HEAD_SCALAR:
        return rev.sum(axis=(0, 2, 3))
    return rev


def _check_chunk(x, dO, dST, got, ref, report=None, where=""):
    """The chunk form's two bars: the bf16 contract per tensor and the rounding bound per element."""
    mags = _mags(x, dO, dST)
    for n, a, r, m in zip(["dq", "dk", "dv", "dlog_g", "dS0"], got, ref, mags):
        if r is None:
            assert a is None
            continue
        assert np.all(np.isfinite(a)), (n, where)
        rf, ma = errors(a, r)
        if report is not None:
            report.append((n, rf, ma))
        if n == "dlog_g":
            bound = CH_TERM * _gate_abs_sum(x, dST, mags, mag=True) + 1e-30
        else:
            assert rf <= CH_REL_FRO and ma <= CH_MAX_ABS, (n, where, rf, ma)
            bound = CH_TERM * np.asarray(m) + 1e-30
        worst = (np.abs(a - r) / bound).max() if r.size else 0.0
        assert worst <= 1.0, (n, where, "error / bound", worst)


def _check(w, seed=0, dst=True, report=None, path=AUTO):
    x, dO, dST = _inputs(w, seed, dst)
    got = _gpu(x, dO, dST, path)
    ref = oracle.gla_backward(x["q"], x["k"], x["v"], x["log_g"], x["gate"], x["S0"], dO, dST)
    if _kind(w, path) == "chunk":
        _check_chunk(x, dO, dST, got, ref, report)
        return got
    tc = _tensor(w, path)
    rel_fro, max_abs = (TC_REL_FRO, TC_MAX_ABS) if tc else (REL_FRO, MAX_ABS)
    names = ["dq", "dk", "dv", "dlog_g", "dS0"]
    for n, a, r in zip(names, got, ref):
        if r is None:
            assert a is None
            continue
        assert np.all(np.isfinite(a)), n
        rf, ma = errors(a, r)
        if report is not None:
            report.append((n, rf, ma))
        if n == "dlog_g" and tc:
            assert rf <= TC_GATE_REL_FRO and ma <= TC_GATE_MAX_ABS, (n, rf, ma)
        elif n == "dlog_g":
            bound = 1e-5 * _gate_abs_sum(x, dST, ref) + 1e-30
            assert np.all(np.abs(a - r) <= bound), (n, np.abs(a - r).max(), bound.max())
        else:
            assert rf <= rel_fro and ma <= max_abs, (n, rf, ma)
    return got


@pytest.mark.gpu
@pytest.mark.parametrize("gate", GATES)
@pytest.mark.parametrize("T", [1, 16, 17, 100])
@pytest.mark.parametrize("dtype,path", [(torch.bfloat16, AUTO), (torch.bfloat16, SIMT), (torch.float32, AUTO)])
def test_bwd_gates_ragged(gate, T, dtype, path):
    gbuild.build(); oracle.build()
    w = gi.Workload("t", B=2, H=2, T=T, dk=64, dv=80, dtype=dtype, gate=gate, s0_std=0.3)
    rep = []
    _check(w, seed=T + 7 * gate, report=rep, path=path)
    print(gate, T, dtype, path, [(n, f"{rf:.1e}", f"{ma:.1e}") for n, rf, ma in rep])


@pytest.mark.gpu
@pytest.mark.parametrize("gate", [gi.GATE_PER_KEY, gi.GATE_TOKEN_SCALAR])
def test_bwd_no_state_terms(gate):
    """S0 = 0 and dST = 0: dS0 is then sum_t (q_t (.) b_t)^T do_t."""
    gbuild.build(); oracle.build()
    w = gi.Workload("t", B=1, H=3, T=77, dk=128, dv=128, dtype=torch.bfloat16, gate=gate)
    _check(w, seed=5, dst=False)


@pytest.mark.gpu
@pytest.mark.parametrize("dist", ["steep", "const:-60", "zero"])
def test_bwd_extreme_gates(dist):
    gbuild.build(); oracle.build()
    w = gi.Workload("t", B=1, H=2, T=90, dk=64, dv=64, dtype=torch.float32, gate=gi.GATE_PER_KEY,
                    gate_dist=dist, s0_std=0.2, qkv_scale="q")
    _check(w, seed=6)


@pytest.mark.gpu
@pytest.mark.parametrize("path", [AUTO, SPLIT, SIMT])
def test_bwd_long_wide(path):
    gbuild.build(); oracle.build()
    w = gi.Workload("t", B=2, H=2, T=1000, dk=128, dv=256, dtype=torch.bfloat16, gate=gi.GATE_PER_KEY,
                    s0_std=0.02)
    rep = []
    _check(w, seed=8, path=path, report=rep)
    print("long_wide", path, [(n, f"{rf:.1e}", f"{ma:.1e}") for n, rf, ma in rep])


@pytest.mark.gpu
@pytest.mark.parametrize("path", [AUTO, SPLIT, SIMT])
@pytest.mark.parametrize("gate", [gi.GATE_PER_KEY, gi.GATE_TOKEN_SCALAR, gi.GATE_NONE])
def test_bwd_dk256_many_tiles(path, gate):
    gbuild.build(); oracle.build()
    w = gi.Workload("t", B=1, H=2, T=130, dk=256, dv=512, dtype=torch.bfloat16, gate=gate,
                    s0_std=0.02)
    rep = []
    _check(w, seed=9, path=path, report=rep)
    print("dk256", path, gate, [(n, f"{rf:.1e}", f"{ma:.1e}") for n, rf, ma in rep])


@pytest.mark.gpu
@pytest.mark.parametrize("gate", GATES)
@pytest.mark.parametrize("T", [1, 64, 65, 200])
@pytest.mark.parametrize("dk,dv", [(128, 128), (256, 256)])
def test_bwd_chunk_form_gates_ragged(gate, T, dk, dv):
    """The chunk form on every gate: one partial chunk, one whole chunk, a ragged tail,
    several chunks; one and two key halves, odd and even numbers of dv blocks."""
    gbuild.build(); oracle.build()
    w = gi.Workload("t", B=2, H=2, T=T, dk=dk, dv=dv, dtype=torch.bfloat16, gate=gate, s0_std=0.3)
    assert _kind(w, AUTO) == "chunk"
    rep = []
    _check(w, seed=T + 7 * gate + dk, report=rep, path=TENSOR)
    print(gate, T, dk, dv, [(n, f"{rf:.1e}", f"{ma:.1e}") for n, rf, ma in rep])


@pytest.mark.gpu
@pytest.mark.parametrize("dist", ["steep", "const:-60", "const:-1.2", "zero"])
def test_bwd_chunk_form_extreme_gates(dist):
    """Gates whose chunk decay falls below exp(-60) on some keys (const:-1.2 over 64 rows, and
    steeper) take the pairwise intra rule for those keys; the result holds the same bars."""
    gbuild.build(); oracle.build()
    w = gi.Workload("t", B=1, H=2, T=150, dk=128, dv=128, dtype=torch.bfloat16, gate=gi.GATE_PER_KEY,
                    gate_dist=dist, s0_std=0.2, qkv_scale="q")
    rep = []
    _check(w, seed=16, report=rep)
    print(dist, [(n, f"{rf:.1e}", f"{ma:.1e}") for n, rf, ma in rep])


def _stage_names(w, dst=True):
    """The backward's stages for workload w's shapes (host-side planning only)."""
    x, dO, dST = _inputs(w, 0, dst)
    c = lambda t: None if t is None else t.cuda()
    dev = torch.device("cuda")
    f32 = lambda *sh: torch.empty(sh, dtype=torch.float32, device=dev)
    p = bnd.make_bwd_params(c(x["q"]), c(x["k"]), c(x["v"]), c(x["log_g"]), c(x["S0"]), c(dO), c(dST),
                            f32(w.B, w.H, w.T, w.dk), f32(w.B, w.H, w.T, w.dk), f32(w.B, w.H, w.T, w.dv),
                            None if x["log_g"] is None else f32(*x["log_g"].shape), f32(w.B, w.H, w.dk, w.dv),
                            gate=x["gate"])
    return [bnd.gla_bwd_stage_name(p, i) for i in range(bnd.gla_bwd_num_stages(p))]


@pytest.mark.gpu
@pytest.mark.parametrize("gate", GATES)
@pytest.mark.parametrize("T,dk,dv", [(1100, 128, 128), (2000, 128, 128), (2100, 256, 256)])
def test_bwd_chunk_form_sequence_split(gate, T, dk, dv):
    """Few heads and a long sequence: both sweeps run split into segments (each segment's
    zero-start state, the scan over segments, forward for the states and backward for
    dL/dS), with S0 and dST given."""
    gbuild.build(); oracle.build()
    w = gi.Workload("t", B=1, H=2, T=T, dk=dk, dv=dv, dtype=torch.bfloat16, gate=gate, s0_std=0.3)
    names = _stage_names(w)
    assert "gla_chunk_dstate" in names and "gla_dstate_scan" in names, names
    rep = []
    _check(w, seed=T + gate, report=rep)
    print("split", gate, T, dk, [(n, f"{rf:.1e}", f"{ma:.1e}") for n, rf, ma in rep])


@pytest.mark.gpu
@pytest.mark.parametrize("gate", [gi.GATE_PER_KEY, gi.GATE_HEAD_SCALAR])
def test_bwd_chunk_form_optional_outputs(gate):
    """The chunk form without dL/dS0 and without the gate gradient (no boundary term, no
    gate tail): dq, dk and dv are unchanged, and nothing is written where no output was
    asked for."""
    gbuild.build(); oracle.build()
    w = gi.Workload("t", B=2, H=2, T=150, dk=128, dv=128, dtype=torch.bfloat16, gate=gate, s0_std=0.2)
    x, dO, dST = _inputs(w, 19)
    ref = oracle.gla_backward(x["q"], x["k"], x["v"], x["log_g"], x["gate"], x["S0"], dO, dST)
    c = lambda t: None if t is None else t.cuda()
    dev = torch.device("cuda")
    f32 = lambda *sh: torch.empty(sh, dtype=torch.float32, device=dev)
    dq, dk, dv = f32(2, 2, 150, 128), f32(2, 2, 150, 128), f32(2, 2, 150, 128)
    p = bnd.make_bwd_params(c(x["q"]), c(x["k"]), c(x["v"]), c(x["log_g"]), c(x["S0"]), c(dO), c(dST), dq, dk, dv,
                            None, None, gate=x["gate"])
    assert [bnd.gla_bwd_stage_name(p, i) for i in range(bnd.gla_bwd_num_stages(p))] == [
        "gla_chunk_prep", "gla_bwd_state_sweep", "gla_bwd_dstate_sweep", "gla_bwd_grads"]
    n = bnd.gla_bwd_workspace_size(p)
    ws = torch.empty(n, dtype=torch.uint8, device=dev)
    p.workspace, p.workspace_bytes = ws.data_ptr(), n
    bnd.gla_bwd(p)
    torch.cuda.synchronize()
    assert gla.gla_device_status() == 0
    for name, a, r in zip(["dq", "dk", "dv"], [dq, dk, dv], ref[:3]):
        rf, ma = errors(to_np(a), r)
        assert rf <= CH_REL_FRO and ma <= CH_MAX_ABS, (name, rf, ma)


@pytest.mark.gpu
def test_bwd_misaligned_inputs_take_the_split_form():
    """q two bytes past a 16-byte boundary: AUTO takes the 16-row split form (the chunk form's
    tensor-memory-access copies need 16-byte bases), GLA_PATH_TENSOR is refused, and the
    split form's bar holds."""
    gbuild.build(); oracle.build()
    w = gi.Workload("t", B=1, H=2, T=130, dk=128, dv=128, dtype=torch.bfloat16, gate=gi.GATE_PER_KEY, s0_std=0.1)
    x, dO, dST = _inputs(w, 20)
    buf = torch.empty(x["q"].numel() + 8, dtype=torch.bfloat16, device="cuda")
    qs = buf[1:1 + x["q"].numel()].view(x["q"].shape)
    qs.copy_(x["q"].cuda())
    assert qs.data_ptr() % 16 == 2
    c = lambda t: None if t is None else t.cuda()
    dev = torch.device("cuda")
    f32 = lambda *sh: torch.empty(sh, dtype=torch.float32, device=dev)
    outs = [f32(1, 2, 130, 128), f32(1, 2, 130, 128), f32(1, 2, 130, 128), f32(1, 2, 130, 128), f32(1, 2, 128, 128)]
    p = bnd.make_bwd_params(qs, c(x["k"]), c(x["v"]), c(x["log_g"]), c(x["S0"]), c(dO), c(dST), *outs,
                            gate=x["gate"])
    assert bnd.gla_bwd_num_stages(p) == 1 and bnd.gla_bwd_stage_name(p, 0) == "gla_bwd_split"
    pt = bnd.make_bwd_params(qs, c(x["k"]), c(x["v"]), c(x["log_g"]), c(x["S0"]), c(dO), c(dST), *outs,
                             gate=x["gate"], path=TENSOR)
    assert bnd.gla_bwd(pt, check=False) == bnd.GLA_ERR_UNSUPPORTED
    n = bnd.gla_bwd_workspace_size(p)
    ws = torch.empty(n, dtype=torch.uint8, device=dev)
    p.workspace, p.workspace_bytes = ws.data_ptr(), n
    bnd.gla_bwd(p)
    torch.cuda.synchronize()
    assert gla.gla_device_status() == 0
    ref = oracle.gla_backward(x["q"], x["k"], x["v"], x["log_g"], x["gate"], x["S0"], dO, dST)
    for name, a, r in zip(["dq", "dk", "dv", "dlog_g", "dS0"], outs, ref):
        rf, ma = errors(to_np(a), r)
        if name == "dlog_g":
            assert rf <= TC_GATE_REL_FRO and ma <= TC_GATE_MAX_ABS, (name, rf, ma)
        else:
            assert rf <= TC_REL_FRO and ma <= TC_MAX_ABS, (name, rf, ma)


FUZZ = [(int(b), int(h), int(t), int(dk), int(dv), int(g), int(seed))
        for b, h, t, dk, dv, g, seed in zip(
            np.random.default_rng(7).integers(1, 4, 10), np.random.default_rng(8).integers(1, 4, 10),
            np.random.default_rng(9).integers(1, 700, 10), np.random.default_rng(10).choice([128, 256], 10),
            np.random.default_rng(11).choice([128, 256, 384], 10), np.random.default_rng(12).choice(GATES, 10),
            range(10))]


@pytest.mark.gpu
@pytest.mark.parametrize("B,H,T,dk,dv,gate,seed", FUZZ, ids=[f"{f[0]}x{f[1]}x{f[2]}-{f[3]}-{f[4]}-g{f[5]}" for f in FUZZ])
def test_bwd_chunk_form_seeded_shapes(B, H, T, dk, dv, gate, seed):
    """Seeded shapes across the chunk form's range (one to three batch rows and heads, T up to
    700 with ragged tails, dk in {128, 256}, dv in {128, 256, 384}, every gate), with S0 and
    dST present or absent by seed."""
    gbuild.build(); oracle.build()
    w = gi.Workload("t", B=B, H=H, T=T, dk=dk, dv=dv, dtype=torch.bfloat16, gate=gate,
                    s0_std=0.2 if seed % 2 else 0.0)
    assert _kind(w, AUTO) == "chunk"
    _check(w, seed=100 + seed, dst=seed % 3 != 0)


@pytest.mark.gpu
def test_bwd_chunk_form_many_items_per_cta():
    """More (b, h, chunk) items than multiprocessors, so each CTA of the persistent gradient
    kernel takes several chunks, with no S0 and no dST."""
    gbuild.build(); oracle.build()
    w = gi.Workload("t", B=3, H=4, T=1000, dk=128, dv=256, dtype=torch.bfloat16, gate=gi.GATE_PER_KEY)
    rep = []
    _check(w, seed=17, dst=False, report=rep)
    print("many items", [(n, f"{rf:.1e}", f"{ma:.1e}") for n, rf, ma in rep])


@pytest.mark.gpu
def test_bwd_stages_in_sequence_equal_the_call():
    """gla_bwd_stage(p, 0) ... gla_bwd_stage(p, n-1) gives bitwise the same gradients as gla_bwd."""
    gbuild.build()
    w = gi.Workload("t", B=2, H=2, T=300, dk=128, dv=256, dtype=torch.bfloat16, gate=gi.GATE_PER_KEY, s0_std=0.2)
    x, dO, dST = _inputs(w, 18)
    ref = _gpu(x, dO, dST)
    c = lambda t: None if t is None else t.cuda()
    dev = torch.device("cuda")
    f32 = lambda *sh: torch.empty(sh, dtype=torch.float32, device=dev)
    dq, dk, dv = f32(2, 2, 300, 128), f32(2, 2, 300, 128), f32(2, 2, 300, 256)
    dg, dS0 = f32(2, 2, 300, 128), f32(2, 2, 128, 256)
    p = bnd.make_bwd_params(c(x["q"]), c(x["k"]), c(x["v"]), c(x["log_g"]), c(x["S0"]), c(dO), c(dST), dq, dk, dv,
                            dg, dS0, gate=x["gate"])
    n = bnd.gla_bwd_workspace_size(p)
    ws = torch.empty(n, dtype=torch.uint8, device=dev)
    p.workspace, p.workspace_bytes = ws.data_ptr(), n
    assert bnd.gla_bwd_num_stages(p) == 6
    for i in range(6):
        bnd.gla_bwd_stage(p, i)
    torch.cuda.synchronize()
    assert gla.gla_device_status() == 0
    for a, b in zip(ref, [dq, dk, dv, dg, dS0]):
        np.testing.assert_array_equal(a, to_np(b))


@pytest.mark.gpu
def test_bwd_empty_sequence():
    gbuild.build(); oracle.build()
    for gate in GATES:
        w = gi.Workload("t", B=2, H=2, T=0, dk=64, dv=64, dtype=torch.bfloat16, gate=gate, s0_std=0.3)
        x, dO, dST = _inputs(w, 10)
        dq, dk, dv, dg, dS0 = _gpu(x, dO, dST)
        np.testing.assert_array_equal(dS0, dST.numpy())
        if gate == gi.GATE_HEAD_SCALAR:
            np.testing.assert_array_equal(dg, np.zeros(2))


@pytest.mark.gpu
def test_bwd_bitwise_reproducible():
    gbuild.build()
    w = gi.Workload("t", B=2, H=2, T=200, dk=128, dv=128, dtype=torch.bfloat16, gate=gi.GATE_TOKEN_SCALAR,
                    s0_std=0.1)
    x, dO, dST = _inputs(w, 11)
    for path in (AUTO, SIMT):
        a, b = _gpu(x, dO, dST, path), _gpu(x, dO, dST, path)
        for u, v in zip(a, b):
            np.testing.assert_array_equal(u, v)


@pytest.mark.gpu
def test_bwd_unaligned_inputs_match_aligned():
    """v and dO at bases 2 bytes past a 16-byte boundary (the backward asks only for element
    alignment): the intra kernel stages them element by element instead of in 16-byte
    pieces, and every gradient is bitwise the same as from aligned copies."""
    gbuild.build()
    w = gi.Workload("t", B=1, H=2, T=100, dk=128, dv=320, dtype=torch.bfloat16, gate=gi.GATE_PER_KEY,
                    s0_std=0.1)
    x, dO, dST = _inputs(w, 12)
    ref = _gpu(x, dO, dST)

    def shifted(t):
        buf = torch.empty(t.numel() + 8, dtype=t.dtype, device="cuda")
        u = buf[1:1 + t.numel()].view(t.shape)
        u.copy_(t.cuda())
        assert u.data_ptr() % 16 == 2
        return u
    c = lambda t: None if t is None else t.cuda()
    out = gla.backward(c(x["q"]), c(x["k"]), shifted(x["v"]), c(x["log_g"]), c(x["S0"]), shifted(dO), c(dST),
                       gate=x["gate"])
    torch.cuda.synchronize()
    assert gla.gla_device_status() == 0
    for u, v in zip(ref, out):
        if u is not None:
            np.testing.assert_array_equal(u, to_np(v))


@pytest.mark.gpu
def test_bwd_full_gla_layer_sampled_heads():
    """The 1.3B-shaped layer (B=8 H=4 T=2048 dk=256 dv=512) in one launch; two heads held to the oracle."""
    gbuild.build(); oracle.build()
    w = gi.WORKLOADS["gla_1p3b"]
    x, dO, dST = _inputs(w, 12)
    got = _gpu(x, dO, dST)
    for (b, h) in [(0, 0), (7, 3)]:
        sl = lambda t: None if t is None else t[b:b + 1, h:h + 1]
        ref = oracle.gla_backward(sl(x["q"]), sl(x["k"]), sl(x["v"]), sl(x["log_g"]), x["gate"], sl(x["S0"]),
                                  sl(dO), sl(dST))
        xs = {n: (sl(t) if isinstance(t, torch.Tensor) else t) for n, t in x.items()}
        _check_chunk(xs, sl(dO), sl(dST), [a[b:b + 1, h:h + 1] for a in got], ref, where=(b, h))


# ---------------------------------------------------------------- host-side checks (no GPU)

def test_bwd_struct_layout():
    # 12 pointers, 7 ints (padded to 8 bytes), pointer, size_t, int (padded), 2 pointers
    assert ctypes.sizeof(bnd.gla_bwd_params) == 12 * 8 + 8 * 4 + 8 + 8 + 8 + 2 * 8
    assert bnd.gla_bwd_params.workspace.offset == 128
    assert bnd.gla_bwd_params.path.offset == 144
    assert bnd.gla_bwd_params.log_b.offset == 152
    assert bnd.gla_bwd_params.grad_log_b.offset == 160


def _bp(**kw):
    p = bnd.gla_bwd_params()
    base = dict(q=0x10000, k=0x20000, v=0x30000, log_g=0x40000, S0=None, grad_O=0x50000, grad_ST=None,
                grad_q=0x60000, grad_k=0x70000, grad_v=0x80000, grad_log_g=0x90000, grad_S0=None,
                B=1, H=1, T=64, dk=64, dv=64, dtype=bnd.GLA_BF16, gate=bnd.GLA_GATE_PER_KEY,
                workspace=None, workspace_bytes=0)
    base.update(kw)
    for k, v in base.items():
        setattr(p, k, v)
    return p


BAD = [
    ("null grad_O", dict(grad_O=None), bnd.GLA_ERR_INVALID_ARG),
    ("null grad_q", dict(grad_q=None), bnd.GLA_ERR_INVALID_ARG),
    ("dk not /16", dict(dk=40), bnd.GLA_ERR_INVALID_ARG),
    ("gate none with log_g", dict(gate=bnd.GLA_GATE_NONE), bnd.GLA_ERR_INVALID_ARG),
    ("gate none with grad_log_g", dict(gate=bnd.GLA_GATE_NONE, log_g=None), bnd.GLA_ERR_INVALID_ARG),
    ("per-key gate without log_g", dict(log_g=None), bnd.GLA_ERR_INVALID_ARG),
    ("grad_q overlaps q", dict(grad_q=0x10000 + 64), bnd.GLA_ERR_INVALID_ARG),
    ("grad_k overlaps grad_q", dict(grad_k=0x60000 + 4), bnd.GLA_ERR_INVALID_ARG),
    ("misaligned grad_v", dict(grad_v=0x80002), bnd.GLA_ERR_INVALID_ARG),
    ("misaligned workspace", dict(workspace=0x7000010, workspace_bytes=1 << 20), bnd.GLA_ERR_INVALID_ARG),
    ("bad dtype", dict(dtype=5), bnd.GLA_ERR_INVALID_ARG),
    ("dk 512", dict(dk=512), bnd.GLA_ERR_UNSUPPORTED),
    ("bilinear gate without log_b", dict(gate=4), bnd.GLA_ERR_INVALID_ARG),
    ("log_b with the per-key gate", dict(log_b=0x900000), bnd.GLA_ERR_INVALID_ARG),
    ("bilinear gate on the tensor path", dict(gate=4, log_b=0x900000, path=bnd.GLA_PATH_TENSOR),
     bnd.GLA_ERR_UNSUPPORTED),
    ("tensor path with fp32", dict(dtype=bnd.GLA_FP32, path=bnd.GLA_PATH_TENSOR), bnd.GLA_ERR_UNSUPPORTED),
    ("tensor path with dk 48", dict(dk=48, path=bnd.GLA_PATH_TENSOR), bnd.GLA_ERR_UNSUPPORTED),
    ("tensor path with dk 64", dict(path=bnd.GLA_PATH_TENSOR), bnd.GLA_ERR_UNSUPPORTED),
    ("tensor path with dv 192", dict(dk=128, dv=192, path=bnd.GLA_PATH_TENSOR), bnd.GLA_ERR_UNSUPPORTED),
    ("tensor path with q off 16 bytes", dict(dk=128, dv=128, q=0x10008, path=bnd.GLA_PATH_TENSOR),
     bnd.GLA_ERR_UNSUPPORTED),
    ("split path with dk 48", dict(dk=48, path=bnd.GLA_PATH_SPLIT), bnd.GLA_ERR_UNSUPPORTED),
    ("split path with fp32", dict(dtype=bnd.GLA_FP32, path=bnd.GLA_PATH_SPLIT), bnd.GLA_ERR_UNSUPPORTED),
    ("bad path", dict(path=7), bnd.GLA_ERR_INVALID_ARG),
    ("no workspace", dict(), bnd.GLA_ERR_WORKSPACE),
]


@pytest.mark.parametrize("name,kw,want", BAD, ids=[b[0] for b in BAD])
def test_bwd_rejects_before_launch(name, kw, want):
    gbuild.build()
    assert bnd.gla_bwd(_bp(**kw), stream=0, check=False) == want


def test_bwd_workspace_size():
    gbuild.build()
    far = {n: (i + 1) << 28 for i, n in enumerate(["q", "k", "v", "log_g", "grad_O", "grad_q", "grad_k", "grad_v",
                                                   "grad_log_g"])}
    p = _bp(B=2, H=3, T=100, dk=64, dv=128, **far)
    n = bnd.gla_bwd_workspace_size(p)
    nch, ndvt, BH = 7, 2, 6
    assert n >= 4 * (BH * nch * 64 * 128 + 2 * ndvt * BH * 100 * 64 + BH * 100 * 64)
    assert bnd.gla_bwd_workspace_size(_bp(dk=40)) == 0


def test_bwd_stages():
    """The staged backward: the chunk form's six stages (four without a gate gradient, five
    without grad_ST), the 16-row forms' one; out-of-range names."""
    gbuild.build()
    far = {n: (i + 1) << 28 for i, n in enumerate(["q", "k", "v", "log_g", "grad_O", "grad_q", "grad_k", "grad_v",
                                                   "grad_log_g", "grad_ST"])}
    p = _bp(B=2, H=3, T=100, dk=128, dv=256, **far)
    names = [bnd.gla_bwd_stage_name(p, i) for i in range(bnd.gla_bwd_num_stages(p))]
    assert names == ["gla_chunk_prep", "gla_bwd_state_sweep", "gla_bwd_dstate_sweep", "gla_bwd_boundary",
                     "gla_bwd_grads", "gla_bwd_gate_tail"]
    assert bnd.gla_bwd_num_stages(_bp(B=2, H=3, T=100, dk=128, dv=256, **dict(far, grad_ST=None))) == 5
    assert bnd.gla_bwd_num_stages(_bp(B=2, H=3, T=100, dk=128, dv=256, **dict(far, grad_log_g=None))) == 4
    split = _bp(B=2, H=3, T=100, dk=64, dv=128, **far)
    assert bnd.gla_bwd_num_stages(split) == 1 and bnd.gla_bwd_stage_name(split, 0) == "gla_bwd_split"
    assert bnd.gla_bwd_stage_name(split, 1) == "invalid"
    assert bnd.gla_bwd_num_stages(_bp(dk=40)) == -1
    assert bnd.gla_bwd_stage(p, 7, stream=0, check=False) == bnd.GLA_ERR_INVALID_ARG


def test_bwd_chunk_form_workspace_size():
    """The chunk form's workspace: Q (.) Lambda and K (.) Gamma, scores, chunk decays, the two
    sweeps' bf16 chunk states, S_T and the boundary term (with grad_ST), the per-chunk gate
    totals (the per-key gate's per-token terms go straight to grad_log_g); less than the
    16-row form's fp32 chunk states."""
    gbuild.build()
    far = {n: (i + 1) << 28 for i, n in enumerate(["q", "k", "v", "log_g", "grad_O", "grad_q", "grad_k", "grad_v",
                                                   "grad_log_g", "grad_ST"])}
    B, H, T, dk, dv = 2, 3, 100, 128, 256
    p = _bp(B=B, H=H, T=T, dk=dk, dv=dv, **far)
    n = bnd.gla_bwd_workspace_size(p)
    BH, nch, Tpad = B * H, 2, 128
    up = lambda x: (x + 255) // 256 * 256
    want = (2 * up(BH * Tpad * dk * 2) + up(BH * nch * 64 * 64 * 2) + up(BH * nch * dk * 4)
            + 2 * up(BH * nch * dv * dk * 2) + up(BH * dk * dv * 4) + up(BH * dk * 4) + up(BH * nch * dk * 4))
    assert n == want
    split = bnd.gla_bwd_workspace_size(_bp(B=B, H=H, T=T, dk=dk, dv=dv, path=bnd.GLA_PATH_SPLIT, **far))
    assert split > n
