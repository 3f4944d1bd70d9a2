"""The sliding-window split (window_chunks > 0; off by default and not exact): each
segment after the first starts from the state that the window of chunks before it
leaves from a zero start, instead of the exact state the scan over earlier segments
gives (the FlashQLA talk's "sliding window" property of decaying gates).

Held to the fp64 oracle two ways:
  1. the GPU result equals, within the bf16 tolerance, the same windowed method
     evaluated with the oracle, segment by segment from the windowed start states;
  2. the windowed start states differ from the exact ones by at most the decayed
     influence of what the window drops, max_k Gamma_w[k] * |S_w|_F (S_w the exact
     state at the window's first token, Gamma_w the product of the gates over the
     window), and the GPU outputs differ from the exact ones by no more than that
     error can reach through the query rows, plus the bf16 tolerance."""
import numpy as np
import pytest
import torch

import oracle
import chunkwise_gated_linear_gla_gb300 as gla
from chunkwise_gated_linear_gla_gb300 import build as gbuild
from chunkwise_gated_linear_gla_gb300 import inputs as gi

from _util import TOL, assert_close, to_np

pytestmark = pytest.mark.gpu

C = 64


@pytest.fixture(scope="module", autouse=True)
def _built():
    gbuild.build()
    oracle.build()


def _segments(T, nseg_req):
    """The plan's split: nseg segments of ceil(nchunks / nseg) chunks (the last shorter)."""
    nch = -(-T // C)
    nseg = min(nseg_req, nch)
    cps = -(-nch // nseg)
    nseg = -(-nch // cps)
    return [min(T, s * cps * C) for s in range(nseg)] + [T]


def _tok(x, a, b):
    g = x["log_g"]
    if g is not None and x["gate"] != gi.GATE_HEAD_SCALAR:
        g = g[:, :, a:b]
    return x["q"][:, :, a:b], x["k"][:, :, a:b], x["v"][:, :, a:b], g


def _log_gamma(x, a, b, dk):
    """Sum over tokens [a, b) of log alpha, per (b, h, key)."""
    B, H = x["q"].shape[:2]
    g = x["log_g"]
    if x["gate"] == gi.GATE_HEAD_SCALAR:
        return np.broadcast_to((b - a) * g.double().numpy()[None, :, None], (B, H, dk))
    if x["gate"] == gi.GATE_TOKEN_SCALAR:
        return np.broadcast_to(g[:, :, a:b].double().numpy().sum(axis=2)[..., None], (B, H, dk))
    return g[:, :, a:b].double().numpy().sum(axis=2)


def _windowed_oracle(x, edges, wtok):
    """The windowed method in fp64: returns (O, S_T, windowed start states, window starts)."""
    Os, starts, wstarts = [], [], []
    S = x["S0"]
    for s, (a, b) in enumerate(zip(edges, edges[1:])):
        if s > 0:
            w = max(0, a - wtok)
            q, k, v, g = _tok(x, w, a)
            _, S = oracle.gla_forward(q, k, v, g, x["gate"], None)
            wstarts.append(w)
        starts.append(S)
        q, k, v, g = _tok(x, a, b)
        O, S = oracle.gla_forward(q, k, v, g, x["gate"], S)
        Os.append(O)
    return np.concatenate(Os, axis=2), S, starts, wstarts


CASES = [("per_key", gi.GATE_PER_KEY, 128, 256), ("head_scalar", gi.GATE_HEAD_SCALAR, 128, 128),
         ("token_scalar", gi.GATE_TOKEN_SCALAR, 64, 128)]


@pytest.mark.parametrize("name,gate,dk,dv", CASES, ids=[c[0] for c in CASES])
@pytest.mark.parametrize("wchunks", [1, 2, 4])
def test_window_split_matches_the_windowed_method_and_its_bound(name, gate, dk, dv, wchunks):
    T, nseg = 1000, 4
    w = gi.Workload("t", B=2, H=2, T=T, dk=dk, dv=dv, dtype=torch.bfloat16, gate=gate, s0_std=0.2)
    x = gi.make_inputs(w, seed=90 + wchunks)
    c = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    O, ST = gla.forward(c["q"], c["k"], c["v"], c["log_g"], c["S0"], gate=x["gate"], force_segments=nseg,
                        window_chunks=wchunks)
    torch.cuda.synchronize()
    assert gla.gla_device_status() == 0
    edges = _segments(T, nseg)
    assert len(edges) - 1 == nseg
    Ow, STw, starts, wstarts = _windowed_oracle(x, edges, wchunks * C)
    # 1. the implementation of the windowed method
    assert_close(to_np(O), Ow, torch.bfloat16, "O vs the windowed method")
    assert_close(to_np(ST), STw, torch.bfloat16, "S_T vs the windowed method")
    # 2. the method's error against the exact pass, within the decayed-influence bound
    Oex, _ = oracle.gla_forward(x["q"], x["k"], x["v"], x["log_g"], x["gate"], x["S0"])
    qn = np.linalg.norm(x["q"].double().numpy(), axis=3)   # [B,H,T]
    gotO = to_np(O)
    for s in range(1, nseg):
        a, b, wst = edges[s], edges[s + 1], wstarts[s - 1]
        q, k, v, g = _tok(x, 0, a)
        _, S_exact = oracle.gla_forward(q, k, v, g, x["gate"], x["S0"])
        q, k, v, g = _tok(x, 0, wst)
        _, S_w = oracle.gla_forward(q, k, v, g, x["gate"], x["S0"])
        gam = np.exp(_log_gamma(x, wst, a, dk)).max(axis=2)                       # [B,H]
        bound = gam * np.linalg.norm(S_w.reshape(*S_w.shape[:2], -1), axis=2)     # [B,H]
        err = np.linalg.norm((starts[s] - S_exact).reshape(*S_exact.shape[:2], -1), axis=2)
        assert np.all(err <= bound * (1 + 1e-9) + 1e-12), (s, err, bound)
        # through row r the start error reaches O at most |q_r| * bound (decays only shrink it)
        reach = qn[:, :, a:b].max(axis=2) * bound                                  # [B,H]
        dev = np.abs(gotO[:, :, a:b] - Oex[:, :, a:b]).max(axis=(2, 3))
        tol = TOL[torch.bfloat16]["max_abs"] * np.abs(Oex[:, :, a:b]).max()
        assert np.all(dev <= reach + tol), (s, dev, reach, tol)


def test_window_covering_everything_is_exact_without_s0():
    """A window at least as long as the sequence before each segment, and no S0: nothing is
    dropped, so the split gives the exact pass."""
    T = 700
    w = gi.Workload("t", B=1, H=2, T=T, dk=128, dv=128, dtype=torch.bfloat16, gate=gi.GATE_PER_KEY)
    x = gi.make_inputs(w, seed=95)
    c = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    O, ST = gla.forward(c["q"], c["k"], c["v"], c["log_g"], None, gate=x["gate"], force_segments=3,
                        window_chunks=64)
    torch.cuda.synchronize()
    Oex, STex = oracle.gla_forward(x["q"], x["k"], x["v"], x["log_g"], x["gate"], None)
    assert_close(to_np(O), Oex, torch.bfloat16, "O")
    assert_close(to_np(ST), STex, torch.bfloat16, "S_T")


def test_window_is_off_by_default_and_ignored_without_a_split():
    T = 400
    w = gi.Workload("t", B=1, H=2, T=T, dk=128, dv=128, dtype=torch.bfloat16, gate=gi.GATE_PER_KEY, s0_std=0.3)
    x = gi.make_inputs(w, seed=96)
    c = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    O1, S1 = gla.forward(c["q"], c["k"], c["v"], c["log_g"], c["S0"], force_segments=1, window_chunks=1)
    O2, S2 = gla.forward(c["q"], c["k"], c["v"], c["log_g"], c["S0"], force_segments=1)
    torch.cuda.synchronize()
    assert torch.equal(O1, O2) and torch.equal(S1, S2)
