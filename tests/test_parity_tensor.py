"""GPU parity of the tensor-core path (gla_chunk_prep + gla_chunk_fwd, and the
sequence split with gla_state_scan) against the fp64 oracle, through the C ABI."""
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


def _run(w, seed=0, path=gla.GLA_PATH_TENSOR, force_segments=0):
    x = gi.make_inputs(w, seed=seed)
    c = _dev(x)
    O, ST = gla.forward(c["q"], c["k"], c["v"], c["log_g"], c["S0"], gate=x["gate"], path=path,
                        force_segments=force_segments)
    torch.cuda.synchronize()
    assert gla.gla_device_status() == 0
    return x, O, ST


def _check_full(w, seed=0, force_segments=0):
    x, O, ST = _run(w, seed=seed, force_segments=force_segments)
    Oref, STref = oracle.gla_forward(x["q"], x["k"], x["v"], x["log_g"], x["gate"], x["S0"])
    assert_close(to_np(O), Oref, torch.bfloat16, "O")
    assert_close(to_np(ST), STref, torch.bfloat16, "ST")


# ---------------------------------------------------------------- prep stage unit check

def test_prep_stage_outputs():
    """Stage 0 alone: Q (.) Lambda, K (.) Gamma, gamma and the masked intra scores
    against fp64 numpy formulas of the same quantities (§4.2 of the GLA paper)."""
    w = gi.Workload("t", B=1, H=2, T=100, dk=64, dv=128, dtype=torch.bfloat16, gate=gi.GATE_PER_KEY)
    x = gi.make_inputs(w, seed=1)
    c = _dev(x)
    O = torch.empty(1, 2, 100, 128, dtype=torch.bfloat16, device="cuda")
    p = bnd.make_params(c["q"], c["k"], c["v"], c["log_g"], None, O, None, path=bnd.GLA_PATH_TENSOR)
    n = bnd.gla_fwd_workspace_size(p)
    ws = torch.zeros(n, dtype=torch.uint8, device="cuda")
    p.workspace, p.workspace_bytes = ws.data_ptr(), n
    bnd.gla_fwd_stage(p, 0)
    torch.cuda.synchronize()
    BH, Tpad, dk, nch = 2, 128, 64, 2
    qt = ws[: BH * Tpad * dk * 2].view(torch.bfloat16).view(BH, Tpad, dk).float().cpu().numpy()
    off = BH * Tpad * dk * 2
    kt = ws[off: 2 * off].view(torch.bfloat16).view(BH, Tpad, dk).float().cpu().numpy()
    A = ws[2 * off: 2 * off + BH * nch * 64 * 64 * 2].view(torch.bfloat16).view(BH, nch, 64, 64).float().cpu().numpy()
    o3 = 2 * off + BH * nch * 64 * 64 * 2
    gam = ws[o3: o3 + BH * nch * dk * 4].view(torch.float32).view(BH, nch, dk).cpu().numpy()
    q = x["q"].double().numpy().reshape(BH, 100, dk)
    k = x["k"].double().numpy().reshape(BH, 100, dk)
    g = x["log_g"].double().numpy().reshape(BH, 100, dk)
    for bh in range(BH):
        for ch in range(nch):
            t0, t1 = ch * 64, min(100, ch * 64 + 64)
            L = np.cumsum(g[bh, t0:t1], axis=0)
            Lq = q[bh, t0:t1] * np.exp(L)
            Lk = k[bh, t0:t1] * np.exp(L[-1] - L)
            np.testing.assert_allclose(qt[bh, t0:t1], Lq, rtol=1e-2, atol=1e-3)
            np.testing.assert_allclose(kt[bh, t0:t1], Lk, rtol=1e-2, atol=1e-3)
            np.testing.assert_allclose(gam[bh, ch], np.exp(L[-1]), rtol=1e-5)
            D = L[:, None, :] - L[None, :, :]
            P = np.einsum("rk,sk,rsk->rs", q[bh, t0:t1], k[bh, t0:t1], np.exp(np.minimum(D, 0.0)))
            P = np.tril(P)
            n_ = t1 - t0
            Ag = A[bh, ch, :n_, :n_]
            assert errors(Ag, P)[0] < 5e-3
            assert np.all(A[bh, ch][np.triu_indices(64, 1)] == 0)
            assert np.all(A[bh, ch, n_:, :] == 0)
    assert np.all(qt[:, 100:] == 0) and np.all(kt[:, 100:] == 0)


def test_prep_stage_factored_scalar_gate():
    """Stage 0 under a per-head scalar gate: a chunk whose decay (rows x log lambda) stays
    above -60 leaves the query factor lambda^(r+1) and its scores to the chunk pass, so only
    its K (.) Gamma rows are written (no Q (.) Lambda rows, no score tile); a steeper head
    keeps the scores (q_r . k_s) lambda^(r-s) and its Q (.) Lambda rows."""
    w = gi.Workload("t", B=1, H=2, T=100, dk=64, dv=128, dtype=torch.bfloat16, gate=gi.GATE_HEAD_SCALAR)
    x = gi.make_inputs(w, seed=2)
    x["log_g"] = torch.tensor([-0.04, -2.0], dtype=torch.float32)   # 64 x 2.0 > 60: head 1 is not factored
    c = _dev(x)
    O = torch.empty(1, 2, 100, 128, dtype=torch.bfloat16, device="cuda")
    p = bnd.make_params(c["q"], c["k"], c["v"], c["log_g"], None, O, None, path=bnd.GLA_PATH_TENSOR)
    n = bnd.gla_fwd_workspace_size(p)
    ws = torch.zeros(n, dtype=torch.uint8, device="cuda")
    p.workspace, p.workspace_bytes = ws.data_ptr(), n
    bnd.gla_fwd_stage(p, 0)
    torch.cuda.synchronize()
    BH, Tpad, dk, nch = 2, 128, 64, 2
    off = BH * Tpad * dk * 2
    qt = ws[:off].view(torch.bfloat16).view(BH, Tpad, dk).float().cpu().numpy()
    kt = ws[off:2 * off].view(torch.bfloat16).view(BH, Tpad, dk).float().cpu().numpy()
    A = ws[2 * off: 2 * off + BH * nch * 64 * 64 * 2].view(torch.bfloat16).view(BH, nch, 64, 64).float().cpu().numpy()
    q = x["q"].double().numpy().reshape(BH, 100, dk)
    k = x["k"].double().numpy().reshape(BH, 100, dk)
    lam = x["log_g"].double().numpy()
    for bh in range(BH):
        for ch in range(nch):
            t0, t1 = ch * 64, min(100, ch * 64 + 64)
            n_ = t1 - t0
            r = np.arange(n_)
            factored = n_ * lam[bh] >= -60.0
            S = q[bh, t0:t1] @ k[bh, t0:t1].T
            np.testing.assert_allclose(kt[bh, t0:t1], k[bh, t0:t1] * np.exp((n_ - 1 - r) * lam[bh])[:, None],
                                       rtol=1e-2, atol=1e-3)
            if factored:
                # the chunk pass forms these scores from raw q and K (.) Gamma
                assert np.all(qt[bh, t0:t1] == 0) and np.all(A[bh, ch] == 0)
                continue
            else:
                P = np.tril(S * np.exp((r[:, None] - r[None, :]) * lam[bh] * (r[:, None] >= r[None, :])))
                np.testing.assert_allclose(qt[bh, t0:t1], q[bh, t0:t1] * np.exp((r + 1) * lam[bh])[:, None],
                                           rtol=1e-2, atol=1e-3)
            assert errors(A[bh, ch, :n_, :n_], P)[0] < 5e-3, (bh, ch, factored)
            assert np.all(A[bh, ch][np.triu_indices(64, 1)] == 0)


@pytest.mark.parametrize("dk", [64, 128, 256])
def test_scalar_gate_factored_and_plain_heads(dk):
    """Per-head decays on both sides of the query-factor guard (rows x log lambda >= -60)
    in one call, a ragged last chunk, with and without the sequence split; at dk = 256
    every chunk takes the plain form."""
    w = gi.Workload("t", B=2, H=3, T=333, dk=dk, dv=128, dtype=torch.bfloat16, gate=gi.GATE_HEAD_SCALAR,
                    s0_std=0.1)
    x = gi.make_inputs(w, seed=37 + dk)
    # 64 rows x 0.9 = 57.6 (factored), x 1.2 = 76.8 (plain; the 13-row tail, 15.6, factored)
    x["log_g"] = torch.tensor([-0.02, -0.9, -1.2], dtype=torch.float32)
    for nseg in (0, 3):
        c = _dev(x)
        O, ST = gla.forward(c["q"], c["k"], c["v"], c["log_g"], c["S0"], path=gla.GLA_PATH_TENSOR,
                            force_segments=nseg)
        torch.cuda.synchronize()
        assert gla.gla_device_status() == 0
        Oref, STref = oracle.gla_forward(x["q"], x["k"], x["v"], x["log_g"], x["gate"], x["S0"])
        assert_close(to_np(O), Oref, torch.bfloat16, f"O (segments {nseg})")
        assert_close(to_np(ST), STref, torch.bfloat16, f"ST (segments {nseg})")


# ---------------------------------------------------------------- small shapes

@pytest.mark.parametrize("gate", [gi.GATE_NONE, gi.GATE_HEAD_SCALAR, gi.GATE_PER_KEY, gi.GATE_TOKEN_SCALAR])
@pytest.mark.parametrize("T", [1, 63, 64, 65, 200])
def test_gates_and_ragged_T(gate, T):
    w = gi.Workload("t", B=2, H=2, T=T, dk=128, dv=128, dtype=torch.bfloat16, gate=gate, s0_std=0.02)
    _check_full(w, seed=T + 10 * gate)


@pytest.mark.parametrize("dk,dv", [(64, 128), (128, 256), (256, 128), (256, 512)])
def test_head_shapes(dk, dv):
    w = gi.Workload("t", B=1, H=2, T=300, dk=dk, dv=dv, dtype=torch.bfloat16, gate=gi.GATE_PER_KEY, s0_std=0.02)
    _check_full(w, seed=dk + dv)


@pytest.mark.parametrize("nseg", [1, 2, 3, 7, 16])
def test_forced_segments(nseg):
    """The in-GPU sequence split with state correction gives the same result as one pass."""
    w = gi.Workload("t", B=1, H=2, T=1000, dk=128, dv=128, dtype=torch.bfloat16, gate=gi.GATE_PER_KEY, s0_std=0.02)
    _check_full(w, seed=3, force_segments=nseg)


@pytest.mark.parametrize("gate", [gi.GATE_NONE, gi.GATE_HEAD_SCALAR, gi.GATE_TOKEN_SCALAR])
def test_forced_segments_other_gates(gate):
    w = gi.Workload("t", B=1, H=2, T=700, dk=64, dv=128, dtype=torch.bfloat16, gate=gate, s0_std=0.02)
    _check_full(w, seed=4, force_segments=5)


@pytest.mark.parametrize("nseg,s0", [(2, 0.02), (3, 0.0), (3, 0.02)])
def test_state_pass_pieces(nseg, s0):
    """The split's state pass in pieces finer than the segments, over the chunks before the
    last segment only; the last segment's chunk pass writes S_T. 41 chunks (ragged last
    one), two dv tiles: 2 segments of 21 chunks take 3 pieces of 7 each, 3 segments of 14
    take 2 pieces of 7 each per segment (the last segment 13 chunks)."""
    import bench
    w = gi.Workload("t", B=1, H=2, T=64 * 40 + 17, dk=128, dv=256, dtype=torch.bfloat16,
                    gate=gi.GATE_PER_KEY, s0_std=s0)
    split = bench.planned_split(w, nseg, 148)
    assert split == ((2, 21, 3, 3, 7) if nseg == 2 else (3, 14, 2, 4, 7))
    _check_full(w, seed=11 + nseg, force_segments=nseg)


def test_steep_gate_stays_finite_and_exact():
    """log alpha ~ -U(0,4) per entry: a chunk-level reference would overflow; the
    sub-chunk references keep every factor bounded."""
    w = gi.Workload("t", B=1, H=2, T=256, dk=128, dv=128, dtype=torch.bfloat16, gate=gi.GATE_PER_KEY,
                    gate_dist="steep", s0_std=0.5)
    _check_full(w, seed=5)


def test_extreme_gate_uses_exact_fallback():
    """log alpha = -60 everywhere: each diagonal sub-chunk block falls back to
    pairwise log-space scores; the output is (q_t . k_t) v_t up to e^-60."""
    w = gi.Workload("t", B=1, H=1, T=128, dk=64, dv=128, dtype=torch.bfloat16, gate=gi.GATE_PER_KEY,
                    gate_dist="const:-60", s0_std=0.0)
    _check_full(w, seed=6)


def test_mixed_steep_columns():
    """A few key columns fall off a cliff inside one sub-chunk, the rest are mild."""
    w = gi.Workload("t", B=1, H=2, T=192, dk=128, dv=128, dtype=torch.bfloat16, gate=gi.GATE_PER_KEY, s0_std=0.1)
    x = gi.make_inputs(w, seed=7)
    x["log_g"][:, :, 70, ::9] = -80.0
    x["log_g"][:, 1, 150, 3] = -200.0
    c = _dev(x)
    O, ST = gla.forward(c["q"], c["k"], c["v"], c["log_g"], c["S0"], path=gla.GLA_PATH_TENSOR)
    torch.cuda.synchronize()
    Oref, STref = oracle.gla_forward(x["q"], x["k"], x["v"], x["log_g"], x["gate"], x["S0"])
    assert_close(to_np(O), Oref, torch.bfloat16, "O")
    assert_close(to_np(ST), STref, torch.bfloat16, "ST")


def test_matches_simt_path():
    w = gi.Workload("t", B=2, H=2, T=333, dk=128, dv=256, dtype=torch.bfloat16, gate=gi.GATE_PER_KEY, s0_std=0.02)
    x, O1, S1 = _run(w, seed=8, path=gla.GLA_PATH_TENSOR)
    _, O2, S2 = _run(w, seed=8, path=gla.GLA_PATH_SIMT)
    rf, _ = errors(to_np(O1), to_np(O2))
    assert rf < 5e-3


def test_deterministic_and_every_output_written():
    w = gi.Workload("t", B=2, H=2, T=250, dk=128, dv=256, dtype=torch.bfloat16, gate=gi.GATE_PER_KEY, s0_std=0.02)
    x = gi.make_inputs(w, seed=9)
    c = _dev(x)
    outs = []
    for _ in range(2):
        O = torch.full((2, 2, 250, 256), float("nan"), dtype=torch.bfloat16, device="cuda")
        ST = torch.full((2, 2, 128, 256), float("nan"), device="cuda")
        gla.forward(c["q"], c["k"], c["v"], c["log_g"], c["S0"], O=O, ST=ST, path=gla.GLA_PATH_TENSOR)
        torch.cuda.synchronize()
        assert torch.isfinite(O.float()).all() and torch.isfinite(ST).all()
        outs.append((O.clone(), ST.clone()))
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])


def test_in_place_state_carry_with_split():
    w = gi.Workload("t", B=1, H=2, T=640, dk=128, dv=128, dtype=torch.bfloat16, gate=gi.GATE_PER_KEY, s0_std=0.3)
    x = gi.make_inputs(w, seed=10)
    c = _dev(x)
    S = c["S0"].clone()
    O = torch.empty(1, 2, 640, 128, dtype=torch.bfloat16, device="cuda")
    gla.forward(c["q"], c["k"], c["v"], c["log_g"], S, O=O, ST=S, path=gla.GLA_PATH_TENSOR, force_segments=4)
    torch.cuda.synchronize()
    Oref, STref = oracle.gla_forward(x["q"], x["k"], x["v"], x["log_g"], x["gate"], x["S0"])
    assert_close(to_np(O), Oref, torch.bfloat16, "O")
    assert_close(to_np(S), STref, torch.bfloat16, "ST")


@pytest.mark.parametrize("gate", [gi.GATE_NONE, gi.GATE_HEAD_SCALAR])
def test_state_carried_in_place_across_calls(gate):
    """A long sequence fed as consecutive calls, each call's S_T written over the next call's
    S0 in one buffer, with no synchronisation in between: the scores formed in the chunk pass
    (dk <= 128), where no gate means no prep kernel ahead of the pass, so the pass itself must
    wait for the previous call's S_T before it reads S0. Equal to one call over the sequence."""
    w = gi.Workload("t", B=2, H=4, T=3 * 256, dk=128, dv=256, dtype=torch.bfloat16, gate=gate, s0_std=0.2)
    x = gi.make_inputs(w, seed=21 + gate)
    c = _dev(x)
    S = c["S0"].clone()
    parts = [tuple(c[n][:, :, 256 * i:256 * (i + 1)].contiguous() for n in ("q", "k", "v")) for i in range(3)]
    Os = [torch.empty(2, 4, 256, 256, dtype=torch.bfloat16, device="cuda") for _ in range(3)]
    for (q, k, v), Oi in zip(parts, Os):   # the calls' kernels back to back on the stream
        gla.forward(q, k, v, c["log_g"], S, O=Oi, ST=S, gate=x["gate"], path=gla.GLA_PATH_TENSOR)
    torch.cuda.synchronize()
    O = torch.cat(Os, dim=2)
    assert gla.gla_device_status() == 0
    Oref, STref = oracle.gla_forward(x["q"], x["k"], x["v"], x["log_g"], x["gate"], x["S0"])
    assert_close(to_np(O), Oref, torch.bfloat16, "O")
    assert_close(to_np(S), STref, torch.bfloat16, "ST")


def test_gla_fwd_public_signature():
    """gla_fwd(q,k,v,log_g,S0,O,ST,B,H,T,dk,dv,chunk,stream): per-key gate, stream-ordered workspace."""
    w = gi.Workload("t", B=2, H=2, T=130, dk=128, dv=128, dtype=torch.bfloat16, gate=gi.GATE_PER_KEY, s0_std=0.02)
    x = gi.make_inputs(w, seed=12)
    c = _dev(x)
    O = torch.empty(2, 2, 130, 128, dtype=torch.bfloat16, device="cuda")
    ST = torch.empty(2, 2, 128, 128, device="cuda")
    bnd.gla_fwd(c["q"], c["k"], c["v"], c["log_g"], c["S0"], O, ST, 2, 2, 130, 128, 128, 64)
    torch.cuda.synchronize()
    Oref, STref = oracle.gla_forward(x["q"], x["k"], x["v"], x["log_g"], x["gate"], x["S0"])
    assert_close(to_np(O), Oref, torch.bfloat16, "O")
    assert_close(to_np(ST), STref, torch.bfloat16, "ST")


# ---------------------------------------------------------------- full-size workloads, sampled heads

def _sampled(name, heads, seed=0):
    w = gi.WORKLOADS[name]
    x, O, ST = _run(w, seed=seed, path=gla.GLA_PATH_AUTO)
    ref = oracle.gla_forward_rows(x["q"], x["k"], x["v"], x["log_g"], x["gate"], x["S0"], heads)
    for (b, h), (Oref, STref) in ref.items():
        assert_close(to_np(O[b, h]), Oref, torch.bfloat16, f"{name} O[{b},{h}]")
        assert_close(to_np(ST[b, h]), STref, torch.bfloat16, f"{name} ST[{b},{h}]")


def test_full_linear_attention_sampled():
    _sampled("linear_attn", [(0, 0), (7, 15), (3, 9)])


def test_full_scalar_decay_sampled():
    _sampled("scalar_decay", [(0, 0), (3, 15), (1, 7)])


def test_full_gla_1p3b_sampled():
    _sampled("gla_1p3b", [(0, 0), (7, 3), (4, 1)])


def test_full_gla_long_sampled():
    _sampled("gla_long", [(0, 0), (0, 3)])


def test_full_token_gate_sampled():
    _sampled("token_gate", [(0, 0), (7, 3), (2, 1)])


# ---------------------------------------------------------------- per-token scalar gate

@pytest.mark.parametrize("dk", [64, 128, 256])
def test_token_gate_head_sizes(dk):
    w = gi.Workload("t", B=2, H=2, T=300, dk=dk, dv=256, dtype=torch.bfloat16, gate=gi.GATE_TOKEN_SCALAR,
                    s0_std=0.02)
    _check_full(w, seed=30 + dk)


@pytest.mark.parametrize("dist", ["steep", "const:-60", "zero"])
def test_token_gate_extremes(dist):
    """log gamma_t = -U(0,4), a constant -60 (every earlier token forgotten) and 0 (no decay):
    every factor stays <= 1, so the tensor path needs no fallback."""
    w = gi.Workload("t", B=1, H=2, T=200, dk=128, dv=128, dtype=torch.bfloat16, gate=gi.GATE_TOKEN_SCALAR,
                    gate_dist=dist, s0_std=0.3)
    _check_full(w, seed=35)


def test_token_gate_equals_per_key_broadcast():
    """The per-token gate through its own prep equals the per-key path fed the same gate on every key."""
    w = gi.Workload("t", B=2, H=2, T=190, dk=128, dv=128, dtype=torch.bfloat16, gate=gi.GATE_TOKEN_SCALAR,
                    s0_std=0.05)
    x = gi.make_inputs(w, seed=36)
    c = _dev(x)
    O1, S1 = gla.forward(c["q"], c["k"], c["v"], c["log_g"], c["S0"], path=gla.GLA_PATH_TENSOR)
    gk = c["log_g"][..., None].expand(*c["q"].shape).contiguous()
    O2, S2 = gla.forward(c["q"], c["k"], c["v"], gk, c["S0"], path=gla.GLA_PATH_TENSOR)
    torch.cuda.synchronize()
    assert_close(to_np(O1), to_np(O2).astype(np.float64), torch.bfloat16, "O token vs per-key")
    assert_close(to_np(S1), to_np(S2).astype(np.float64), torch.bfloat16, "ST token vs per-key")


# ---------------------------------------------------------------- degenerate and extreme shapes

def test_zero_per_key_gate_equals_no_gate():
    """log alpha = 0 through the per-key path is causal linear attention."""
    w = gi.Workload("t", B=1, H=2, T=200, dk=128, dv=128, dtype=torch.bfloat16, gate=gi.GATE_PER_KEY,
                    gate_dist="zero", s0_std=0.05)
    x = gi.make_inputs(w, seed=21)
    c = _dev(x)
    O1, S1 = gla.forward(c["q"], c["k"], c["v"], c["log_g"], c["S0"], path=gla.GLA_PATH_TENSOR)
    O2, S2 = gla.forward(c["q"], c["k"], c["v"], None, c["S0"], path=gla.GLA_PATH_TENSOR)
    torch.cuda.synchronize()
    assert_close(to_np(O1), to_np(O2), torch.bfloat16, "O per-key zero gate vs no gate")
    Oref, STref = oracle.gla_forward(x["q"], x["k"], x["v"], None, gi.GATE_NONE, x["S0"])
    assert_close(to_np(O1), Oref, torch.bfloat16, "O")
    assert_close(to_np(S1), STref, torch.bfloat16, "ST")


def test_wide_dv_eight_tiles():
    w = gi.Workload("t", B=1, H=1, T=257, dk=128, dv=1024, dtype=torch.bfloat16, gate=gi.GATE_PER_KEY, s0_std=0.02)
    _check_full(w, seed=22)


def test_many_small_heads():
    w = gi.Workload("t", B=32, H=8, T=70, dk=64, dv=128, dtype=torch.bfloat16, gate=gi.GATE_PER_KEY, s0_std=0.02)
    _check_full(w, seed=23)


def test_steep_scalar_decay():
    """lambda = e^-30: the closed-form scores lambda^(r-s) underflow to zero off the diagonal."""
    w = gi.Workload("t", B=1, H=2, T=150, dk=64, dv=128, dtype=torch.bfloat16, gate=gi.GATE_HEAD_SCALAR, s0_std=0.1)
    x = gi.make_inputs(w, seed=24)
    x["log_g"] = torch.tensor([-30.0, -0.5], dtype=torch.float32)
    c = _dev(x)
    O, ST = gla.forward(c["q"], c["k"], c["v"], c["log_g"], c["S0"], path=gla.GLA_PATH_TENSOR)
    torch.cuda.synchronize()
    Oref, STref = oracle.gla_forward(x["q"], x["k"], x["v"], x["log_g"], x["gate"], x["S0"])
    assert_close(to_np(O), Oref, torch.bfloat16, "O")
    assert_close(to_np(ST), STref, torch.bfloat16, "ST")


# ---------------------------------------------------------------- dk = 512 in two key halves

@pytest.mark.parametrize("gate", [gi.GATE_NONE, gi.GATE_HEAD_SCALAR, gi.GATE_PER_KEY, gi.GATE_TOKEN_SCALAR])
@pytest.mark.parametrize("T", [1, 65, 200])
def test_dk512_key_halves(gate, T):
    """dk = 512 on the tensor path: two chunk passes, each over 256 keys with its own rows of
    the state, the second adding the first's fp32 partial output; every gate mode but the
    bilinear one, ragged T, S0 given."""
    w = gi.Workload("t", B=1, H=2, T=T, dk=512, dv=256, dtype=torch.bfloat16, gate=gate, s0_std=0.02)
    x = gi.make_inputs(w, seed=50 + T + gate)
    c = _dev(x)
    O = torch.empty(x["v"].shape, dtype=torch.bfloat16, device="cuda")
    ST = torch.empty(1, 2, 512, 256, device="cuda")
    p = bnd.make_params(c["q"], c["k"], c["v"], c["log_g"], c["S0"], O, ST, gate=x["gate"],
                        path=bnd.GLA_PATH_TENSOR)
    assert [bnd.gla_fwd_stage_name(p, i) for i in range(bnd.gla_fwd_num_stages(p))][-2:] == \
        ["gla_chunk_fwd", "gla_chunk_fwd_keys_hi"]
    O, ST = gla.forward(c["q"], c["k"], c["v"], c["log_g"], c["S0"], gate=x["gate"], path=gla.GLA_PATH_TENSOR)
    torch.cuda.synchronize()
    assert gla.gla_device_status() == 0
    Oref, STref = oracle.gla_forward(x["q"], x["k"], x["v"], x["log_g"], x["gate"], x["S0"])
    assert_close(to_np(O), Oref, torch.bfloat16, "O")
    assert_close(to_np(ST), STref, torch.bfloat16, "ST")


def test_dk512_steep_gate_and_in_place_state():
    """dk = 512 with log alpha = -U(0,4) (the prep's sub-chunk form at 512 keys) and ST == S0
    (each key half updates its own rows of the state in place)."""
    w = gi.Workload("t", B=1, H=2, T=150, dk=512, dv=128, dtype=torch.bfloat16, gate=gi.GATE_PER_KEY,
                    gate_dist="steep", s0_std=0.3)
    x = gi.make_inputs(w, seed=58)
    c = _dev(x)
    S = c["S0"].clone()
    O, ST = gla.forward(c["q"], c["k"], c["v"], c["log_g"], S, path=gla.GLA_PATH_TENSOR, ST=S)
    torch.cuda.synchronize()
    assert gla.gla_device_status() == 0
    Oref, STref = oracle.gla_forward(x["q"], x["k"], x["v"], x["log_g"], x["gate"], x["S0"])
    assert_close(to_np(O), Oref, torch.bfloat16, "O")
    assert_close(to_np(S), STref, torch.bfloat16, "ST (in place)")


# ---------------------------------------------------------------- maximum sizes

def test_max_heads_grid_limit():
    """B*H = 65535, the most heads the tensor path takes (the chunk pass gives every head
    its own grid row): every output element written, sampled heads against the oracle."""
    w = gi.Workload("t", B=65535, H=1, T=3, dk=64, dv=128, dtype=torch.bfloat16, gate=gi.GATE_PER_KEY)
    x = gi.make_inputs(w, seed=61)
    c = _dev(x)
    O = torch.full(x["v"].shape, float("nan"), dtype=torch.bfloat16, device="cuda")
    gla.forward(c["q"], c["k"], c["v"], c["log_g"], None, path=gla.GLA_PATH_TENSOR, want_state=False, O=O)
    torch.cuda.synchronize()
    assert gla.gla_device_status() == 0
    assert not torch.isnan(O).any()
    heads = [(0, 0), (32767, 0), (65534, 0)]
    ref = oracle.gla_forward_rows(x["q"], x["k"], x["v"], x["log_g"], x["gate"], None, heads)
    for (b, h), (Oref, _) in ref.items():
        assert_close(to_np(O[b, h]), Oref, torch.bfloat16, f"O[{b},{h}]")


def test_long_sequence_many_chunks():
    """One head of T = 2^18 + 37 rows (4097 chunks with a ragged tail; the planner splits the
    sequence), per-key gate and S0, against the oracle over the whole sequence."""
    w = gi.Workload("t", B=1, H=1, T=(1 << 18) + 37, dk=64, dv=128, dtype=torch.bfloat16,
                    gate=gi.GATE_PER_KEY, s0_std=0.1)
    x, O, ST = _run(w, seed=62, path=gla.GLA_PATH_TENSOR)
    Oref, STref = oracle.gla_forward(x["q"], x["k"], x["v"], x["log_g"], x["gate"], x["S0"])
    assert_close(to_np(O), Oref, torch.bfloat16, "O")
    assert_close(to_np(ST), STref, torch.bfloat16, "ST")
