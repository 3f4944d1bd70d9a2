"""Pins for the fp64 backward oracle (the adjoint of the recurrence of "Gated
Linear Attention Transformers with Hardware-Efficient Training", §4.1 Eq. 3).
None of them restates the adjoint recurrence:

* central finite differences of L = <dO, O> + <dST, S_T>, where O and S_T come
  from the forward oracle (itself pinned in test_oracle_pins.py);
* torch.autograd through a separately written fp64 recurrence in plain torch
  operations (a library's reverse mode, not this code);
* the closed form of causal linear attention (§2.1: O = ((Q K^T) (.) M) V gives
  dV = ((Q K^T) (.) M)^T dO, dQ = ((dO V^T) (.) M) K, dK = ((dO V^T) (.) M)^T Q).

All run on the CPU.
"""
import numpy as np
import pytest
import torch

import oracle
from chunkwise_gated_linear_gla_gb300 import inputs as gi

GATES = [gi.GATE_NONE, gi.GATE_HEAD_SCALAR, gi.GATE_PER_KEY, gi.GATE_TOKEN_SCALAR]


def _case(B, H, T, dk, dv, gate, seed, s0=True, dst=True, dist="logsigmoid16"):
    w = gi.Workload("pin", B=B, H=H, T=T, dk=dk, dv=dv, dtype=torch.float32, gate=gate,
                    s0_std=0.5 if s0 else 0.0, gate_dist=dist)
    x = gi.make_inputs(w, seed=seed)
    f = lambda t: None if t is None else t.to(torch.float64).numpy()
    rng = np.random.default_rng(seed)
    dO = rng.standard_normal((B, H, T, dv))
    dST = rng.standard_normal((B, H, dk, dv)) if dst else None
    return f(x["q"]), f(x["k"]), f(x["v"]), f(x["log_g"]), x["gate"], f(x["S0"]), dO, dST


def _loss(q, k, v, g, gate, S0, dO, dST):
    O, ST = oracle.gla_forward(q, k, v, g, gate, S0)
    L = float((O * dO).sum())
    if dST is not None:
        L += float((ST * dST).sum())
    return L


@pytest.mark.parametrize("gate", GATES)
def test_finite_differences(gate):
    q, k, v, g, gate, S0, dO, dST = _case(2, 2, 5, 3, 2, gate, seed=51)
    dq, dk, dv, dg, dS0 = oracle.gla_backward(q, k, v, g, gate, S0, dO, dST)
    args = dict(q=q, k=k, v=v, g=g, S0=S0)
    grads = dict(q=dq, k=dk, v=dv, g=dg, S0=dS0)
    h = 1e-6
    for name in ("q", "k", "v", "g", "S0"):
        if name == "g" and gate == gi.GATE_NONE:
            assert dg is None
            continue
        arr = args[name]
        fd = np.zeros_like(arr)
        for idx in np.ndindex(arr.shape):
            p, m = dict(args), dict(args)
            p[name] = arr.copy(); p[name][idx] += h
            m[name] = arr.copy(); m[name][idx] -= h
            fd[idx] = (_loss(p["q"], p["k"], p["v"], p["g"], gate, p["S0"], dO, dST)
                       - _loss(m["q"], m["k"], m["v"], m["g"], gate, m["S0"], dO, dST)) / (2 * h)
        scale = max(1.0, np.abs(fd).max())
        np.testing.assert_allclose(grads[name], fd, rtol=0, atol=1e-7 * scale, err_msg=name)


def _torch_recurrence(q, k, v, g, gate, S0):
    """Eq. 3 token by token in plain fp64 torch operations (O and S_T)."""
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    S = S0.clone() if S0 is not None else torch.zeros(B, H, dk, dv, dtype=torch.float64)
    outs = []
    for t in range(T):
        if gate == gi.GATE_NONE:
            a = torch.ones(B, H, dk, dtype=torch.float64)
        elif gate == gi.GATE_HEAD_SCALAR:
            a = torch.exp(g)[None, :, None].expand(B, H, dk)
        elif gate == gi.GATE_TOKEN_SCALAR:
            a = torch.exp(g[:, :, t])[..., None].expand(B, H, dk)
        else:
            a = torch.exp(g[:, :, t])
        S = a[..., None] * S + k[:, :, t, :, None] * v[:, :, t, None, :]
        outs.append(torch.einsum("bhk,bhkv->bhv", q[:, :, t], S))
    return torch.stack(outs, dim=2), S


@pytest.mark.parametrize("gate", GATES)
@pytest.mark.parametrize("T", [1, 40, 200])
def test_autograd_of_plain_recurrence(gate, T):
    """T = 200 spans several checkpoint blocks of the oracle's reverse sweep."""
    q, k, v, g, gate, S0, dO, dST = _case(2, 2, T, 8, 6, gate, seed=52 + T)
    t = lambda a: None if a is None else torch.tensor(a, dtype=torch.float64, requires_grad=True)
    tq, tk, tv, tg, tS0 = t(q), t(k), t(v), t(g), t(S0)
    O, ST = _torch_recurrence(tq, tk, tv, tg, gate, tS0)
    L = (O * torch.tensor(dO)).sum() + (ST * torch.tensor(dST)).sum()
    L.backward()
    dq, dk, dv, dg, dS0 = oracle.gla_backward(q, k, v, g, gate, S0, dO, dST)
    for name, got, ref in (("dq", dq, tq.grad), ("dk", dk, tk.grad), ("dv", dv, tv.grad), ("dS0", dS0, tS0.grad),
                           ("dlog_g", dg, None if tg is None else tg.grad)):
        if ref is None:
            continue
        ref = ref.numpy()
        np.testing.assert_allclose(got, ref, rtol=0, atol=1e-11 * max(1.0, np.abs(ref).max()), err_msg=name)


def test_linear_attention_closed_form():
    q, k, v, _, _, _, dO, _ = _case(2, 3, 37, 7, 5, gi.GATE_NONE, seed=53, s0=False, dst=False)
    dq, dk, dv, dg, dS0 = oracle.gla_backward(q, k, v, None, oracle.GATE_NONE, None, dO, None)
    M = np.tril(np.ones((37, 37)))
    P = (q @ np.swapaxes(k, -1, -2)) * M
    dP = (dO @ np.swapaxes(v, -1, -2)) * M
    np.testing.assert_allclose(dv, np.swapaxes(P, -1, -2) @ dO, rtol=0, atol=1e-12)
    np.testing.assert_allclose(dq, dP @ k, rtol=0, atol=1e-12)
    np.testing.assert_allclose(dk, np.swapaxes(dP, -1, -2) @ q, rtol=0, atol=1e-12)
    assert dg is None
    # with no S0 and no dST, dS0 = sum_t q_t^T do_t (alpha = 1)
    np.testing.assert_allclose(dS0, np.swapaxes(q, -1, -2) @ dO, rtol=0, atol=1e-12)


def test_empty_sequence():
    q = np.zeros((1, 2, 0, 4)); v = np.zeros((1, 2, 0, 3))
    dST = np.arange(24, dtype=np.float64).reshape(1, 2, 4, 3)
    dq, dk, dv, dg, dS0 = oracle.gla_backward(q, q, v, np.zeros((1, 2, 0, 4)), oracle.GATE_PER_KEY, None,
                                              np.zeros((1, 2, 0, 3)), dST)
    assert dq.shape == (1, 2, 0, 4) and dg.shape == (1, 2, 0, 4)
    np.testing.assert_array_equal(dS0, dST)


@pytest.mark.parametrize("mutant", [11, 12, 13, 14])
def test_pins_catch_planted_backward_mistakes(mutant):
    q, k, v, g, gate, S0, dO, dST = _case(1, 2, 30, 5, 4, gi.GATE_PER_KEY, seed=54)
    good = oracle.gla_backward(q, k, v, g, gate, S0, dO, dST)
    bad = oracle.gla_backward(q, k, v, g, gate, S0, dO, dST, mutant=mutant)
    t = lambda a: torch.tensor(a, dtype=torch.float64, requires_grad=True)
    tq, tk, tv, tg, tS0 = t(q), t(k), t(v), t(g), t(S0)
    O, ST = _torch_recurrence(tq, tk, tv, tg, gate, tS0)
    ((O * torch.tensor(dO)).sum() + (ST * torch.tensor(dST)).sum()).backward()
    refs = [tq.grad, tk.grad, tv.grad, tg.grad, tS0.grad]
    err_good = max(np.abs(a - r.numpy()).max() for a, r in zip(good, refs))
    err_bad = max(np.abs(a - r.numpy()).max() for a, r in zip(bad, refs))
    assert err_good < 1e-10
    assert err_bad > 1e-6, f"mutant {mutant} not caught"


# ---------------------------------------------------------------- bilinear gate (mode 4)

def _bil_case(B=1, H=2, T=5, dk=3, dv=2, seed=71, dist="logsigmoid16"):
    w = gi.Workload("pin", B=B, H=H, T=T, dk=dk, dv=dv, dtype=torch.float32, gate=gi.GATE_BILINEAR,
                    s0_std=0.5, gate_dist=dist)
    x = gi.make_inputs(w, seed=seed)
    f = lambda t: None if t is None else t.to(torch.float64).numpy()
    rng = np.random.default_rng(seed)
    dO = rng.standard_normal((B, H, T, dv))
    dST = rng.standard_normal((B, H, dk, dv))
    return f(x["q"]), f(x["k"]), f(x["v"]), f(x["log_g"]), f(x["log_b"]), f(x["S0"]), dO, dST


def _bil_loss(q, k, v, g, b, S0, dO, dST):
    O, ST = oracle.gla_forward(q, k, v, g, gi.GATE_BILINEAR, S0, log_b=b)
    return float((O * dO).sum()) + float((ST * dST).sum())


def test_bilinear_finite_differences():
    """Every gradient of the bilinear gate, log beta included, against central differences
    of the (pinned) forward oracle."""
    q, k, v, g, b, S0, dO, dST = _bil_case()
    dq, dk, dv, dg, dS0, db = oracle.gla_backward(q, k, v, g, gi.GATE_BILINEAR, S0, dO, dST, log_b=b)
    args = dict(q=q, k=k, v=v, g=g, b=b, S0=S0)
    grads = dict(q=dq, k=dk, v=dv, g=dg, b=db, S0=dS0)
    h = 1e-6
    for name, arr in args.items():
        fd = np.zeros_like(arr)
        for idx in np.ndindex(arr.shape):
            p, m = dict(args), dict(args)
            p[name] = arr.copy(); p[name][idx] += h
            m[name] = arr.copy(); m[name][idx] -= h
            fd[idx] = (_bil_loss(**p, dO=dO, dST=dST) - _bil_loss(**m, dO=dO, dST=dST)) / (2 * h)
        scale = max(1.0, np.abs(fd).max())
        np.testing.assert_allclose(grads[name], fd, rtol=0, atol=1e-7 * scale, err_msg=name)


@pytest.mark.parametrize("T", [1, 33, 150])
def test_bilinear_autograd_of_plain_recurrence(T):
    """torch.autograd through S_t = Diag(alpha_t) S_{t-1} Diag(beta_t) + k_t^T v_t written
    in plain fp64 torch operations (T = 150 spans checkpoint blocks)."""
    q, k, v, g, b, S0, dO, dST = _bil_case(B=2, H=1, T=T, dk=6, dv=5, seed=72 + T)
    t = lambda a: torch.tensor(a, dtype=torch.float64, requires_grad=True)
    tq, tk, tv, tg, tb, tS0 = t(q), t(k), t(v), t(g), t(b), t(S0)
    S = tS0
    outs = []
    for s in range(T):
        S = torch.exp(tg[:, :, s])[..., None] * S * torch.exp(tb[:, :, s])[..., None, :] + \
            tk[:, :, s, :, None] * tv[:, :, s, None, :]
        outs.append(torch.einsum("bhk,bhkv->bhv", tq[:, :, s], S))
    L = (torch.stack(outs, dim=2) * torch.tensor(dO)).sum() + (S * torch.tensor(dST)).sum()
    L.backward()
    got = oracle.gla_backward(q, k, v, g, gi.GATE_BILINEAR, S0, dO, dST, log_b=b)
    for name, x, ref in zip(("dq", "dk", "dv", "dlog_g", "dS0", "dlog_b"), got,
                            (tq.grad, tk.grad, tv.grad, tg.grad, tS0.grad, tb.grad)):
        ref = ref.numpy()
        np.testing.assert_allclose(x, ref, rtol=0, atol=1e-11 * max(1.0, np.abs(ref).max()), err_msg=name)


def test_bilinear_unit_beta_is_the_per_key_backward():
    """beta = 1: every gradient but dlog beta equals the per-key gate's."""
    q, k, v, g, b, S0, dO, dST = _bil_case(B=2, H=2, T=40, dk=4, dv=3, seed=73)
    got = oracle.gla_backward(q, k, v, g, gi.GATE_BILINEAR, S0, dO, dST, log_b=np.zeros_like(b))
    ref = oracle.gla_backward(q, k, v, g, gi.GATE_PER_KEY, S0, dO, dST)
    for name, x, y in zip(("dq", "dk", "dv", "dlog_g", "dS0"), got[:5], ref):
        np.testing.assert_allclose(x, y, rtol=0, atol=1e-12 * max(1.0, np.abs(y).max()), err_msg=name)


@pytest.mark.parametrize("dist", ["logsigmoid16", "steep"])
def test_bilinear_gate_gradients_closed_form(dist):
    """The gate gradients in closed form, from the other gradients and the outputs (what a
    chunked backward uses instead of the state products): with c_t the reverse cumulative
    sum over tokens t' >= t,
      dlog alpha_t = c_t( q (.) dq - k (.) dk ) + [t' = T-1] rowsum(dST (.) S_T),
      dlog beta_t  = c_t( o (.) do - v (.) dv ) + [t' = T-1] colsum(dST (.) S_T),
    where each term is the derivative through the cumulative decays b_t, b'_t that the
    parallel form O = ((Q (.) B)(K / B)^T (.) M (.) B'/B') V + (Q (.) B) S0 Diag(B') contains."""
    q, k, v, g, b, S0, dO, dST = _bil_case(B=1, H=2, T=70, dk=5, dv=4, seed=74, dist=dist)
    dq, dk, dv, dg, dS0, db = oracle.gla_backward(q, k, v, g, gi.GATE_BILINEAR, S0, dO, dST, log_b=b)
    O, ST = oracle.gla_forward(q, k, v, g, gi.GATE_BILINEAR, S0, log_b=b)
    ea = q * dq - k * dk
    eb = O * dO - v * dv
    ea[:, :, -1] += (dST * ST).sum(-1)
    eb[:, :, -1] += (dST * ST).sum(-2)
    rc = lambda x: np.flip(np.cumsum(np.flip(x, 2), 2), 2)
    for name, got, ref in (("dlog_g", dg, rc(ea)), ("dlog_b", db, rc(eb))):
        np.testing.assert_allclose(got, ref, rtol=0, atol=1e-10 * max(1.0, np.abs(ref).max()), err_msg=name)


@pytest.mark.parametrize("mutant", [15, 16])
def test_bilinear_pins_catch_planted_mistakes(mutant):
    """dlog beta without its factor beta_t (15) and D decayed by alpha only (16) each fail
    the finite-difference pin on some gradient."""
    q, k, v, g, b, S0, dO, dST = _bil_case(seed=75)
    bad = oracle.gla_backward(q, k, v, g, gi.GATE_BILINEAR, S0, dO, dST, log_b=b, mutant=mutant)
    args = dict(q=q, k=k, v=v, g=g, b=b, S0=S0)
    grads = dict(q=bad[0], k=bad[1], v=bad[2], g=bad[3], S0=bad[4], b=bad[5])
    h = 1e-6
    worst = 0.0
    for name, arr in args.items():
        for idx in np.ndindex(arr.shape):
            p, m = dict(args), dict(args)
            p[name] = arr.copy(); p[name][idx] += h
            m[name] = arr.copy(); m[name][idx] -= h
            fd = (_bil_loss(**p, dO=dO, dST=dST) - _bil_loss(**m, dO=dO, dST=dST)) / (2 * h)
            worst = max(worst, abs(grads[name][idx] - fd))
    assert worst > 1e-4
