"""Pins for the fp64 oracle: it is checked against forms and facts the pages
and the mathematics fix, none of which is the recurrence retyped.

Sources (page title, section):
  [GLA]   "Gated Linear Attention Transformers with Hardware-Efficient Training"
          (arXiv 2312.06635): §2.1 Eq. 1 and the masked parallel form,
          §2.2 Eq. 2 (chunkwise form, "C = L recovers the parallel form and
          C = 1 the recurrent form"), §4.1 Eq. 3 / parallel form / Eq. 4
          (log-space pairwise form), §4.2 (chunkwise GLA: Lambda, Gamma, gamma).
  [LA2]   "Lightning Attention-2: A Free Lunch for Handling Unlimited Sequence
          Lengths in Large Language Models", §3.2.1 Alg. 1 (decay mask
          M_ij = lambda^(i-j) for i >= j).
  [GLA Table 1] the data-dependent scalar gate G_t = gamma_t 1^T 1 (Mamba-2,
          mLSTM, Gated Retention rows): alpha_t has the same value gamma_t
          for every key; the bilinear gate G_t = alpha_t^T beta_t (DFW row).
All of these run on the CPU.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from chunkwise_gated_linear_gla_gb300 import inputs as gi

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _case(B=1, H=2, T=37, dk=8, dv=6, gate=gi.GATE_PER_KEY, dist="logsigmoid16",
          s0=0.5, seed=1, dtype=torch.float32):
    w = gi.Workload("pin", B=B, H=H, T=T, dk=dk, dv=dv, dtype=dtype, gate=gate,
                    s0_std=s0, gate_dist=dist)
    x = gi.make_inputs(w, seed=seed)
    f = lambda t: None if t is None else t.to(torch.float64).numpy()
    return f(x["q"]), f(x["k"]), f(x["v"]), f(x["log_g"]), x["gate"], f(x["S0"])


def _logb(log_g, gate, B, H, T, dk):
    """Inclusive cumulative log-decay log b_t = sum_{j<=t} log alpha_j, [B,H,T,dk]."""
    if gate == gi.GATE_NONE:
        return np.zeros((B, H, T, dk))
    if gate == gi.GATE_HEAD_SCALAR:
        steps = np.arange(1, T + 1, dtype=np.float64)
        return np.broadcast_to(log_g[None, :, None, None] * steps[None, None, :, None], (B, H, T, dk)).copy()
    if gate == gi.GATE_TOKEN_SCALAR:
        return np.broadcast_to(np.cumsum(log_g, axis=2)[..., None], (B, H, T, dk)).copy()
    return np.cumsum(log_g, axis=2)


def _gate_log(log_g, gate, B, H, T, dk):
    if gate == gi.GATE_NONE:
        return np.zeros((B, H, T, dk))
    if gate == gi.GATE_HEAD_SCALAR:
        return np.broadcast_to(log_g[None, :, None, None], (B, H, T, dk)).copy()
    if gate == gi.GATE_TOKEN_SCALAR:
        return np.broadcast_to(log_g[..., None], (B, H, T, dk)).copy()
    return log_g


# ---------------------------------------------------------------- golden

def _read_golden(name):
    rows = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, rest = line.split(None, 1)
            rows[key] = np.array([[float(x) for x in part.split()] for part in rest.split("|")])
    return rows


def test_golden_hand_worked_example():
    g = _read_golden("gla_hand_t3.txt")
    q, k, v = (g[n][None, None] for n in ("q", "k", "v"))
    log_g = np.log(g["alpha"])[None, None]
    S0 = g["S0"][None, None]
    O, ST = oracle.gla_forward(q, k, v, log_g, oracle.GATE_PER_KEY, S0)
    np.testing.assert_allclose(O[0, 0], g["O"], rtol=0, atol=1e-13)
    np.testing.assert_allclose(ST[0, 0], g["ST"], rtol=0, atol=1e-13)


# ---------------------------------------------------------------- brute force

def _brute_force(q, k, v, log_g, gate, S0):
    """Unrolled Eq. 3: S_t = sum_i (prod_{j=i+1..t} alpha_j)^T 1 (.) k_i^T v_i (+ prod_{j<=t} alpha_j (.) S0).

    Products of alpha are formed explicitly, one factor at a time.
    """
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    glog = _gate_log(log_g, gate, B, H, T, dk)
    alpha = np.exp(glog)
    O = np.zeros((B, H, T, dv))
    ST = np.zeros((B, H, dk, dv))
    for b in range(B):
        for h in range(H):
            for t in range(T):
                S = np.zeros((dk, dv))
                for i in range(t + 1):
                    p = np.ones(dk)
                    for j in range(i + 1, t + 1):
                        p = p * alpha[b, h, j]
                    S += p[:, None] * np.outer(k[b, h, i], v[b, h, i])
                if S0 is not None:
                    p = np.ones(dk)
                    for j in range(0, t + 1):
                        p = p * alpha[b, h, j]
                    S += p[:, None] * S0[b, h]
                O[b, h, t] = q[b, h, t] @ S
                if t == T - 1:
                    ST[b, h] = S
    return O, ST


@pytest.mark.parametrize("gate", [gi.GATE_NONE, gi.GATE_HEAD_SCALAR, gi.GATE_PER_KEY, gi.GATE_TOKEN_SCALAR])
def test_brute_force_tiny(gate):
    q, k, v, g, gate, S0 = _case(B=2, H=2, T=6, dk=3, dv=4, gate=gate, s0=0.7, seed=3)
    O, ST = oracle.gla_forward(q, k, v, g, gate, S0)
    Ob, STb = _brute_force(q, k, v, g, gate, S0)
    np.testing.assert_allclose(O, Ob, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(ST, STb, rtol=1e-13, atol=1e-13)


# ---------------------------------------------------------------- quadratic forms

def _quadratic_logspace(q, k, v, log_g, gate, S0):
    """[GLA] §4.1 Eq. 4: P_ij = sum_k Q_ik K_jk exp(logB_ik - logB_jk) for i >= j, O = (P (.) M) V.

    The S0 contribution follows from the same unrolling: o_t gains (q_t (.) b_t) S0,
    and S_T = sum_i (b_T / b_i)^T 1 (.) k_i^T v_i + (b_T^T 1) (.) S0.
    """
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    lb = _logb(log_g, gate, B, H, T, dk)
    O = np.zeros((B, H, T, dv))
    ST = np.zeros((B, H, dk, dv))
    for b in range(B):
        for h in range(H):
            L = lb[b, h]
            D = L[:, None, :] - L[None, :, :]               # [i, j, k] = logB_ik - logB_jk
            mask = np.tril(np.ones((T, T), dtype=bool))       # M_ij = 1 iff i >= j
            E = np.where(mask[:, :, None], np.exp(np.where(mask[:, :, None], D, 0.0)), 0.0)
            P = np.einsum("ik,jk,ijk->ij", q[b, h], k[b, h], E)
            O[b, h] = P @ v[b, h]
            if S0 is not None:
                O[b, h] += (q[b, h] * np.exp(L)) @ S0[b, h]
            w = np.exp(L[-1][None, :] - L)                   # (b_T / b_i), [T, dk]
            ST[b, h] = (k[b, h] * w).T @ v[b, h]
            if S0 is not None:
                ST[b, h] += np.exp(L[-1])[:, None] * S0[b, h]
    return O, ST


def _parallel_direct(q, k, v, log_g, gate, S0):
    """[GLA] §4.1 parallel form O = (((Q (.) B)(K / B)^T) (.) M) V, b_t = prod_{j<=t} alpha_j.

    Numerically usable only while b_t stays far from underflow (tiny T, mild gates).
    """
    B_, H, T, dk = q.shape
    lb = _logb(log_g, gate, B_, H, T, dk)
    Bm = np.exp(lb)
    O = np.zeros(v.shape[:-1] + (v.shape[-1],))
    for b in range(B_):
        for h in range(H):
            P = (q[b, h] * Bm[b, h]) @ (k[b, h] / Bm[b, h]).T
            O[b, h] = np.tril(P) @ v[b, h]
            if S0 is not None:
                O[b, h] += (q[b, h] * Bm[b, h]) @ S0[b, h]
    return O


@pytest.mark.parametrize("gate,dist", [(gi.GATE_NONE, "logsigmoid16"),
                                       (gi.GATE_HEAD_SCALAR, "logsigmoid16"),
                                       (gi.GATE_PER_KEY, "logsigmoid16"),
                                       (gi.GATE_PER_KEY, "steep"),
                                       (gi.GATE_TOKEN_SCALAR, "logsigmoid16"),
                                       (gi.GATE_TOKEN_SCALAR, "steep")])
def test_quadratic_logspace_form(gate, dist):
    q, k, v, g, gate, S0 = _case(B=1, H=3, T=96, dk=8, dv=5, gate=gate, dist=dist, s0=0.3, seed=5)
    O, ST = oracle.gla_forward(q, k, v, g, gate, S0)
    Oq, STq = _quadratic_logspace(q, k, v, g, gate, S0)
    scale = np.abs(Oq).max()
    np.testing.assert_allclose(O, Oq, rtol=0, atol=1e-12 * scale)
    np.testing.assert_allclose(ST, STq, rtol=0, atol=1e-12 * np.abs(STq).max())


def test_parallel_direct_form_tiny():
    q, k, v, g, gate, S0 = _case(B=2, H=1, T=24, dk=6, dv=7, s0=0.2, seed=7)
    O, _ = oracle.gla_forward(q, k, v, g, gate, S0)
    Op = _parallel_direct(q, k, v, g, gate, S0)
    np.testing.assert_allclose(O, Op, rtol=0, atol=1e-12 * np.abs(Op).max())


def test_ungated_is_causal_linear_attention():
    """[GLA] §2.1: alpha = 1 gives O = ((Q K^T) (.) M) V with M_ij = 1 iff i >= j."""
    q, k, v, _, _, _ = _case(B=2, H=2, T=70, dk=16, dv=9, gate=gi.GATE_NONE, s0=0.0, seed=9)
    O, ST = oracle.gla_forward(q, k, v, None, oracle.GATE_NONE, None)
    Ol = np.tril(q @ np.swapaxes(k, -1, -2)) @ v
    np.testing.assert_allclose(O, Ol, rtol=0, atol=1e-13 * np.abs(Ol).max())
    np.testing.assert_allclose(ST, np.swapaxes(k, -1, -2) @ v, rtol=0, atol=1e-12)


def test_scalar_decay_closed_form():
    """[LA2] §3.2.1: o_t = sum_{i<=t} lambda^(t-i) (q_t . k_i) v_i, plus lambda^t-weighted S0 term."""
    q, k, v, g, gate, S0 = _case(B=1, H=4, T=50, dk=5, dv=3, gate=gi.GATE_HEAD_SCALAR, s0=0.4, seed=11)
    O, ST = oracle.gla_forward(q, k, v, g, gate, S0)
    T = q.shape[2]
    for h in range(4):
        lam = math.exp(g[h])
        i = np.arange(T)
        M = np.where(i[:, None] >= i[None, :], lam ** (i[:, None] - i[None, :]).clip(min=0), 0.0)
        ref = ((q[0, h] @ k[0, h].T) * M) @ v[0, h]
        ref += (lam ** (i + 1))[:, None] * (q[0, h] @ S0[0, h])
        np.testing.assert_allclose(O[0, h], ref, rtol=0, atol=1e-12 * np.abs(ref).max())
        st = sum(lam ** (T - 1 - j) * np.outer(k[0, h, j], v[0, h, j]) for j in range(T)) + lam ** T * S0[0, h]
        np.testing.assert_allclose(ST[0, h], st, rtol=0, atol=1e-12 * np.abs(st).max())


def test_token_scalar_decay_matrix_form():
    """[GLA Table 1] with alpha_t = gamma_t 1: O = ((Q K^T) (.) L) V with the lower-triangular
    decay matrix L_ts = prod_{u=s+1..t} gamma_u, built here by explicit running products
    (no logarithms), plus the (prod_{u<=t} gamma_u) q_t S0 term; S_T likewise."""
    q, k, v, g, gate, S0 = _case(B=2, H=2, T=40, dk=5, dv=4, gate=gi.GATE_TOKEN_SCALAR, s0=0.4, seed=41)
    O, ST = oracle.gla_forward(q, k, v, g, gate, S0)
    T = q.shape[2]
    gam = np.exp(g)
    for b in range(2):
        for h in range(2):
            L = np.zeros((T, T))
            for t in range(T):
                p = 1.0
                L[t, t] = 1.0
                for s_ in range(t - 1, -1, -1):
                    p *= gam[b, h, s_ + 1]
                    L[t, s_] = p
            pre = np.cumprod(gam[b, h])                     # prod_{u<=t} gamma_u
            ref = ((q[b, h] @ k[b, h].T) * L) @ v[b, h] + pre[:, None] * (q[b, h] @ S0[b, h])
            np.testing.assert_allclose(O[b, h], ref, rtol=0, atol=1e-12 * np.abs(ref).max())
            st = (k[b, h] * L[T - 1][:, None]).T @ v[b, h] + pre[-1] * S0[b, h]
            np.testing.assert_allclose(ST[b, h], st, rtol=0, atol=1e-12 * np.abs(st).max())


def test_token_scalar_special_cases():
    """The per-token scalar gate is the per-key gate with every key's log alpha equal, and with a
    constant per head it is the fixed per-head decay: both reductions hold exactly."""
    q, k, v, g, gate, S0 = _case(B=2, H=3, T=50, dk=6, dv=5, gate=gi.GATE_TOKEN_SCALAR, s0=0.3, seed=43)
    O, ST = oracle.gla_forward(q, k, v, g, gate, S0)
    gk = np.broadcast_to(g[..., None], q.shape).copy()
    Ok, STk = oracle.gla_forward(q, k, v, gk, oracle.GATE_PER_KEY, S0)
    np.testing.assert_array_equal(O, Ok)
    np.testing.assert_array_equal(ST, STk)
    lam = np.array([-0.01, -0.2, -1.5])
    gc = np.broadcast_to(lam[None, :, None], g.shape).copy()
    Oc, STc = oracle.gla_forward(q, k, v, gc, oracle.GATE_TOKEN_SCALAR, S0)
    Oh, STh = oracle.gla_forward(q, k, v, lam, oracle.GATE_HEAD_SCALAR, S0)
    np.testing.assert_array_equal(Oc, Oh)
    np.testing.assert_array_equal(STc, STh)


# ---------------------------------------------------------------- bilinear gate

def _bilinear_case(B=1, H=2, T=37, dk=6, dv=5, seed=61, dist="logsigmoid16", s0=0.5):
    w = gi.Workload("pin", B=B, H=H, T=T, dk=dk, dv=dv, dtype=torch.float32, gate=gi.GATE_BILINEAR,
                    s0_std=s0, gate_dist=dist)
    x = gi.make_inputs(w, seed=seed)
    f = lambda t: None if t is None else t.to(torch.float64).numpy()
    return f(x["q"]), f(x["k"]), f(x["v"]), f(x["log_g"]), f(x["log_b"]), f(x["S0"])


def test_bilinear_brute_force():
    """[GLA Table 1, DFW] G_t = alpha_t^T beta_t: S_t = sum_i (prod alpha) x (prod beta) (.) k_i^T v_i
    (+ the same products over all steps (.) S0), products formed one factor at a time."""
    q, k, v, ga, gb, S0 = _bilinear_case(B=2, H=2, T=6, dk=3, dv=4, seed=61)
    O, ST = oracle.gla_forward(q, k, v, ga, gi.GATE_BILINEAR, S0, log_b=gb)
    al, be = np.exp(ga), np.exp(gb)
    for b in range(2):
        for h in range(2):
            for t in range(6):
                S = np.zeros((3, 4))
                for i in range(t + 1):
                    pa, pb = np.ones(3), np.ones(4)
                    for j in range(i + 1, t + 1):
                        pa = pa * al[b, h, j]
                        pb = pb * be[b, h, j]
                    S += np.outer(pa, pb) * np.outer(k[b, h, i], v[b, h, i])
                pa, pb = np.ones(3), np.ones(4)
                for j in range(t + 1):
                    pa = pa * al[b, h, j]
                    pb = pb * be[b, h, j]
                S += np.outer(pa, pb) * S0[b, h]
                np.testing.assert_allclose(O[b, h, t], q[b, h, t] @ S, rtol=1e-13, atol=1e-13)
                if t == 5:
                    np.testing.assert_allclose(ST[b, h], S, rtol=1e-13, atol=1e-13)


def _bilinear_quadratic(q, k, v, ga, gb, S0):
    """Log-space pairwise form: o_t[j] = sum_{s<=t} sum_k q_tk k_sk e^(B_tk - B_sk) v_sj e^(B'_tj - B'_sj)
    plus sum_k q_tk e^(B_tk) S0_kj e^(B'_tj); S_T likewise, with B, B' the cumulative log gates."""
    Bk, Bv = np.cumsum(ga, axis=2), np.cumsum(gb, axis=2)
    B_, H, T, dk = q.shape
    O = np.zeros(v.shape)
    ST = np.zeros((B_, H, dk, v.shape[-1]))
    for b in range(B_):
        for h in range(H):
            for t in range(T):
                for s_ in range(t + 1):
                    sc = np.sum(q[b, h, t] * k[b, h, s_] * np.exp(Bk[b, h, t] - Bk[b, h, s_]))
                    O[b, h, t] += sc * v[b, h, s_] * np.exp(Bv[b, h, t] - Bv[b, h, s_])
                O[b, h, t] += ((q[b, h, t] * np.exp(Bk[b, h, t])) @ S0[b, h]) * np.exp(Bv[b, h, t])
            wk = np.exp(Bk[b, h, -1][None, :] - Bk[b, h])
            wv = np.exp(Bv[b, h, -1][None, :] - Bv[b, h])
            ST[b, h] = (k[b, h] * wk).T @ (v[b, h] * wv)
            ST[b, h] += np.outer(np.exp(Bk[b, h, -1]), np.exp(Bv[b, h, -1])) * S0[b, h]
    return O, ST


@pytest.mark.parametrize("dist", ["logsigmoid16", "steep"])
def test_bilinear_quadratic_form(dist):
    q, k, v, ga, gb, S0 = _bilinear_case(B=1, H=2, T=50, dk=5, dv=6, seed=62, dist=dist, s0=0.3)
    O, ST = oracle.gla_forward(q, k, v, ga, gi.GATE_BILINEAR, S0, log_b=gb)
    Oq, STq = _bilinear_quadratic(q, k, v, ga, gb, S0)
    np.testing.assert_allclose(O, Oq, rtol=0, atol=1e-12 * np.abs(Oq).max())
    np.testing.assert_allclose(ST, STq, rtol=0, atol=1e-12 * np.abs(STq).max())


def test_bilinear_reductions():
    """beta = 1 is the per-key gate exactly; alpha = 1 is linear attention with a per-column decay,
    o_t[j] = sum_{s<=t} (q_t . k_s) v_s[j] prod_{u=s+1..t} beta_u[j]."""
    q, k, v, ga, gb, S0 = _bilinear_case(B=2, H=2, T=40, dk=6, dv=5, seed=63)
    O1, S1 = oracle.gla_forward(q, k, v, ga, gi.GATE_BILINEAR, S0, log_b=np.zeros_like(gb))
    O2, S2 = oracle.gla_forward(q, k, v, ga, gi.GATE_PER_KEY, S0)
    np.testing.assert_array_equal(O1, O2)
    np.testing.assert_array_equal(S1, S2)
    O3, _ = oracle.gla_forward(q, k, v, np.zeros_like(ga), gi.GATE_BILINEAR, None, log_b=gb)
    be = np.exp(gb)
    for b in range(2):
        for h in range(2):
            for t in range(40):
                ref = np.zeros(5)
                for s_ in range(t + 1):
                    p = np.ones(5)
                    for u in range(s_ + 1, t + 1):
                        p = p * be[b, h, u]
                    ref += (q[b, h, t] @ k[b, h, s_]) * v[b, h, s_] * p
                np.testing.assert_allclose(O3[b, h, t], ref, rtol=0, atol=1e-12 * max(1.0, np.abs(ref).max()))


@pytest.mark.parametrize("mutant", [1, 2, 3, 4, 5, 6, 7])
def test_bilinear_pins_catch_planted_mistakes(mutant):
    q, k, v, ga, gb, S0 = _bilinear_case(B=1, H=2, T=30, dk=5, dv=5, seed=64)
    O, ST = oracle.gla_forward(q, k, v, ga, gi.GATE_BILINEAR, S0, mutant=mutant, log_b=gb)
    Oq, STq = _bilinear_quadratic(q, k, v, ga, gb, S0)
    assert max(np.abs(O - Oq).max(), np.abs(ST - STq).max()) > 1e-6, f"mutant {mutant} not caught"


# ---------------------------------------------------------------- chunkwise form

def _chunked(q, k, v, log_g, gate, S0, C):
    """[GLA] §4.2 chunkwise form, in fp64, for any chunk size C (last chunk may be short).

    Lambda = b_{iC+j}/b_{iC}, Gamma = b_{(i+1)C}/b_{iC+j}, gamma = b_{(i+1)C}/b_{iC};
    S_[i+1] = (gamma^T 1) (.) S_[i] + (K (.) Gamma)^T V;
    O = (Q (.) Lambda) S_[i] + (((Q (.) Lambda)(K / Lambda)^T) (.) M) V.
    Ratios are taken as exp of differences of the cumulative log-decay.
    """
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    lb = _logb(log_g, gate, B, H, T, dk)
    O = np.zeros((B, H, T, dv))
    ST = np.zeros((B, H, dk, dv))
    for b in range(B):
        for h in range(H):
            S = np.zeros((dk, dv)) if S0 is None else S0[b, h].copy()
            for s in range(0, T, C):
                e = min(s + C, T)
                base = lb[b, h, s - 1] if s > 0 else np.zeros(dk)
                L = lb[b, h, s:e] - base             # log Lambda, rows of this chunk
                Lend = lb[b, h, e - 1] - base         # log gamma
                Qc, Kc, Vc = q[b, h, s:e], k[b, h, s:e], v[b, h, s:e]
                Lam = np.exp(L)
                Gam = np.exp(Lend[None, :] - L)
                O[b, h, s:e] = (Qc * Lam) @ S + np.tril((Qc * Lam) @ (Kc / Lam).T) @ Vc
                S = np.exp(Lend)[:, None] * S + (Kc * Gam).T @ Vc
            ST[b, h] = S
    return O, ST


@pytest.mark.parametrize("C", [1, 2, 3, 7, 16, 64, 100])
@pytest.mark.parametrize("gate", [gi.GATE_NONE, gi.GATE_HEAD_SCALAR, gi.GATE_PER_KEY, gi.GATE_TOKEN_SCALAR])
def test_chunk_size_invariance(C, gate):
    """[GLA] §2.2 / §4.2: the chunkwise form equals the recurrence for every C (C=1 and C=T are its limits)."""
    q, k, v, g, gate, S0 = _case(B=1, H=2, T=100, dk=8, dv=6, gate=gate, s0=0.5, seed=13)
    O, ST = oracle.gla_forward(q, k, v, g, gate, S0)
    Oc, STc = _chunked(q, k, v, g, gate, S0, C)
    np.testing.assert_allclose(O, Oc, rtol=0, atol=1e-12 * np.abs(Oc).max())
    np.testing.assert_allclose(ST, STc, rtol=0, atol=1e-12 * np.abs(STc).max())


# ---------------------------------------------------------------- invariants and limits

def test_steep_gate_limit():
    """Eq. 3 with log alpha = -60 everywhere: S_t = k_t^T v_t + O(e^-60), so o_t = (q_t . k_t) v_t."""
    q, k, v, _, _, _ = _case(B=1, H=2, T=40, dk=8, dv=5, s0=0.0, seed=17)
    g = np.full(q.shape, -60.0)
    O, ST = oracle.gla_forward(q, k, v, g, oracle.GATE_PER_KEY, None)
    ref = np.sum(q * k, axis=-1, keepdims=True) * v
    # e^-60 ~ 9e-27: far below rounding of the dot product itself
    np.testing.assert_allclose(O, ref, rtol=0, atol=1e-14 * np.abs(ref).max())
    np.testing.assert_allclose(ST, np.einsum("bhk,bhv->bhkv", k[:, :, -1], v[:, :, -1]), rtol=0, atol=1e-15)


@pytest.mark.parametrize("gate", [gi.GATE_NONE, gi.GATE_HEAD_SCALAR, gi.GATE_PER_KEY, gi.GATE_TOKEN_SCALAR])
def test_initial_state_linearity(gate):
    """O(S0) - O(0) = (Q (.) B) S0 and S_T(S0) - S_T(0) = Diag(b_T) S0."""
    q, k, v, g, gate, S0 = _case(B=2, H=2, T=45, dk=7, dv=4, gate=gate, s0=1.0, seed=19)
    O1, ST1 = oracle.gla_forward(q, k, v, g, gate, S0)
    O0, ST0 = oracle.gla_forward(q, k, v, g, gate, None)
    lb = _logb(g, gate, *q.shape)
    np.testing.assert_allclose(O1 - O0, np.einsum("bhtk,bhkv->bhtv", q * np.exp(lb), S0), rtol=0, atol=1e-12)
    np.testing.assert_allclose(ST1 - ST0, np.exp(lb[:, :, -1])[..., None] * S0, rtol=0, atol=1e-12)


@pytest.mark.parametrize("T1", [1, 17, 64])
def test_segment_composition(T1):
    """[GLA] §2.2: S_[0] may come from the previous segment; running T1 steps and then
    the rest from S_T1 equals one run over all T steps."""
    q, k, v, g, gate, S0 = _case(B=1, H=2, T=90, dk=6, dv=5, s0=0.3, seed=23)
    O, ST = oracle.gla_forward(q, k, v, g, gate, S0)
    Oa, STa = oracle.gla_forward(q[:, :, :T1], k[:, :, :T1], v[:, :, :T1], g[:, :, :T1], gate, S0)
    Ob, STb = oracle.gla_forward(q[:, :, T1:], k[:, :, T1:], v[:, :, T1:], g[:, :, T1:], gate, STa)
    np.testing.assert_allclose(np.concatenate([Oa, Ob], axis=2), O, rtol=0, atol=1e-12)
    np.testing.assert_allclose(STb, ST, rtol=0, atol=1e-12)


def test_linearity_in_v_and_column_subsets():
    q, k, v, g, gate, _ = _case(B=1, H=1, T=33, dk=5, dv=8, s0=0.0, seed=29)
    O, _ = oracle.gla_forward(q, k, v, g, gate, None)
    O2, _ = oracle.gla_forward(q, k, 2.0 * v, g, gate, None)
    np.testing.assert_allclose(O2, 2.0 * O, rtol=1e-14, atol=1e-14)
    cols = [6, 1, 3]
    Os, _ = oracle.gla_forward(q, k, v[..., cols], g, gate, None)
    np.testing.assert_allclose(Os, O[..., cols], rtol=0, atol=1e-14)


def test_empty_sequence_returns_initial_state():
    q = np.zeros((1, 2, 0, 4)); v = np.zeros((1, 2, 0, 3))
    S0 = np.arange(24, dtype=np.float64).reshape(1, 2, 4, 3)
    O, ST = oracle.gla_forward(q, q, v, np.zeros((1, 2, 0, 4)), oracle.GATE_PER_KEY, S0)
    assert O.shape == (1, 2, 0, 3)
    np.testing.assert_array_equal(ST, S0)


def test_threads_do_not_change_result():
    q, k, v, g, gate, S0 = _case(B=2, H=2, T=64, dk=8, dv=130, s0=0.2, seed=31)
    O1, ST1 = oracle.gla_forward(q, k, v, g, gate, S0, nthreads=1)
    O8, ST8 = oracle.gla_forward(q, k, v, g, gate, S0, nthreads=8)
    np.testing.assert_array_equal(O1, O8)
    np.testing.assert_array_equal(ST1, ST8)


# ---------------------------------------------------------------- planted mistakes

@pytest.mark.parametrize("mutant", [1, 2, 3, 4, 5, 6, 7])
def test_pins_catch_planted_mistakes(mutant):
    """Each deliberate mistake planted in the oracle must fail at least one pin."""
    q, k, v, g, gate, S0 = _case(B=1, H=2, T=40, dk=6, dv=6, s0=0.5, seed=37)
    if mutant != 3:
        # the same mistakes under the per-token scalar gate (where rows and columns of the
        # gate coincide, so mutant 3 is no mistake there)
        qt, kt, vt, gt, gatet, S0t = _case(B=1, H=2, T=40, dk=6, dv=6, gate=gi.GATE_TOKEN_SCALAR, s0=0.5, seed=38)
        Ot, STt = oracle.gla_forward(qt, kt, vt, gt, gatet, S0t, mutant=mutant)
        Oqt, STqt = _quadratic_logspace(qt, kt, vt, gt, gatet, S0t)
        assert max(np.abs(Ot - Oqt).max(), np.abs(STt - STqt).max()) > 1e-6, f"mutant {mutant} (token gate)"
    O, ST = oracle.gla_forward(q, k, v, g, gate, S0, mutant=mutant)
    Oq, STq = _quadratic_logspace(q, k, v, g, gate, S0)
    Oc, STc = _chunked(q, k, v, g, gate, S0, 16)
    err = max(np.abs(O - Oq).max(), np.abs(ST - STq).max(), np.abs(O - Oc).max())
    assert err > 1e-6, f"mutant {mutant} not caught (err {err})"
    # the golden example catches the mutants that touch the gate, S0 or the output order
    gd = _read_golden("gla_hand_t3.txt")
    if mutant != 3:
        Og, STg = oracle.gla_forward(gd["q"][None, None], gd["k"][None, None], gd["v"][None, None],
                                     np.log(gd["alpha"])[None, None], oracle.GATE_PER_KEY,
                                     gd["S0"][None, None], mutant=mutant)
        assert max(np.abs(Og[0, 0] - gd["O"]).max(), np.abs(STg[0, 0] - gd["ST"]).max()) > 1e-6


# ---------------------------------------------------------------- the sequence exchange pair

@pytest.mark.parametrize("gate", [gi.GATE_PER_KEY, gi.GATE_HEAD_SCALAR, gi.GATE_TOKEN_SCALAR, gi.GATE_NONE])
def test_segment_pair_is_the_segments_affine_map(gate):
    """[GLA] §2.2: a segment run from any S0 ends in Diag(Gamma) S0 + S*, Gamma the product of
    the gates and S* the zero-start state. Checked against the recurrence run from two
    different S0 (so a wrong Gamma, e.g. a dropped token or a sign, fails)."""
    q, k, v, g, gt, S0 = _case(B=2, H=2, T=45, dk=6, dv=5, gate=gate, s0=0.7, seed=41)
    lg, Sst = oracle.segment_pair(k, v, g, gt)
    for s0 in (S0, -2.0 * S0 + 0.25):
        _, ST = oracle.gla_forward(q, k, v, g, gt, s0)
        np.testing.assert_allclose(ST, np.exp(lg)[..., None] * s0 + Sst, rtol=0, atol=1e-12)
    # the zero-start state does not depend on q
    _, ST0 = oracle.gla_forward(np.zeros_like(q), k, v, g, gt, None)
    np.testing.assert_array_equal(ST0, Sst)


def test_segment_pair_of_an_empty_segment_is_the_identity():
    k = np.zeros((1, 2, 0, 4)); v = np.zeros((1, 2, 0, 3))
    lg, Sst = oracle.segment_pair(k, v, np.zeros((1, 2, 0, 4)), oracle.GATE_PER_KEY)
    np.testing.assert_array_equal(lg, 0.0)
    np.testing.assert_array_equal(Sst, 0.0)


@pytest.mark.parametrize("cuts", [[], [1], [17, 64], [5, 6, 40, 77]])
def test_pair_scan_chains_segments_into_the_whole_sequence(cuts):
    """Pairs of consecutive segments, chained by the scan, give the recurrence's state at
    every segment boundary of the whole sequence (the FlashQLA talk, "core technical
    principles": one correction per segment after a serial recurrence over segments)."""
    q, k, v, g, gt, S0 = _case(B=1, H=2, T=90, dk=6, dv=5, s0=0.4, seed=43)
    edges = [0] + cuts + [90]
    pairs = [oracle.segment_pair(k[:, :, a:b], v[:, :, a:b], g[:, :, a:b], gt) for a, b in zip(edges, edges[1:])]
    S_in, S_T = oracle.pair_scan([p[0] for p in pairs], [p[1] for p in pairs], S0)
    for d, a in enumerate(edges[:-1]):
        _, S_a = oracle.gla_forward(q[:, :, :a], k[:, :, :a], v[:, :, :a], g[:, :, :a], gt, S0)
        np.testing.assert_allclose(S_in[d], S_a, rtol=0, atol=1e-12)
    _, ST = oracle.gla_forward(q, k, v, g, gt, S0)
    np.testing.assert_allclose(S_T, ST, rtol=0, atol=1e-12)
