"""fp64 CPU oracle for the chunkwise GLA forward pass (test infrastructure).

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` import this package. The CUDA library never does, and this
package imports nothing from the library: inputs arrive as plain tensors or
arrays drawn by the seeded generator.

The oracle is the token-by-token recurrence of "Gated Linear Attention
Transformers with Hardware-Efficient Training", §4.1 Eq. 3, written in C
(``gla_oracle.c``) and evaluated in fp64 on exactly the values the GPU sees
(bf16 inputs are widened losslessly). Its backward is the same recurrence's
adjoint (reverse-mode differentiation written out), also in C and fp64.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gla_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libgla_oracle.so")
_lock = threading.Lock()
_lib = None

GATE_NONE, GATE_HEAD_SCALAR, GATE_PER_KEY, GATE_TOKEN_SCALAR, GATE_BILINEAR = 0, 1, 2, 3, 4


def build(force: bool = False) -> str:
    """Compile the C oracle (gcc -O2, no fast-math) into oracle/_build."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-pthread",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            d = ctypes.POINTER(ctypes.c_double)
            lib.gla_oracle_fwd.restype = ctypes.c_int
            lib.gla_oracle_fwd.argtypes = [d, d, d, d, d, ctypes.c_int, d, d, d,
                                           ctypes.c_long, ctypes.c_long, ctypes.c_long,
                                           ctypes.c_long, ctypes.c_long, ctypes.c_int, ctypes.c_int]
            lib.gla_oracle_bwd.restype = ctypes.c_int
            lib.gla_oracle_bwd.argtypes = [d, d, d, d, ctypes.c_int, d, d, d, d, d, d, d, d,
                                           ctypes.c_long, ctypes.c_long, ctypes.c_long,
                                           ctypes.c_long, ctypes.c_long, ctypes.c_int, ctypes.c_int, d, d]
            _lib = lib
    return _lib


def _f64(x):
    """Widen a tensor/array to a contiguous fp64 numpy array (lossless for bf16/fp32)."""
    if x is None:
        return None
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().to("cpu", torch.float64).numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def default_threads() -> int:
    return max(1, len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count() or 1)


def gla_forward(q, k, v, log_g=None, gate=None, S0=None, want_state=True,
                nthreads=None, mutant=0, log_b=None):
    """Run the fp64 recurrence. Returns (O, ST) as fp64 numpy arrays (ST None if not wanted).

    q, k: [B,H,T,dk]; v: [B,H,T,dv]; log_g: [B,H,T,dk] (per-key), [H] (per-head
    scalar), [B,H,T] (per-token scalar) or None (alpha = 1); S0: [B,H,dk,dv] or None.
    The bilinear gate (gate = GATE_BILINEAR) also takes log_b: [B,H,T,dv].
    """
    qa, ka, va = _f64(q), _f64(k), _f64(v)
    B, H, T, dk = qa.shape
    dv = va.shape[-1]
    if gate is None:
        if log_g is None:
            gate = GATE_NONE
        else:
            gate = {1: GATE_HEAD_SCALAR, 3: GATE_TOKEN_SCALAR}.get(np.ndim(_f64(log_g)), GATE_PER_KEY)
    ga = _f64(log_g) if gate != GATE_NONE else None
    ba = _f64(log_b) if gate == GATE_BILINEAR else None
    sa = _f64(S0)
    O = np.empty((B, H, T, dv), dtype=np.float64)
    ST = np.empty((B, H, dk, dv), dtype=np.float64) if want_state else None
    rc = _load().gla_oracle_fwd(_ptr(qa), _ptr(ka), _ptr(va), _ptr(ga), _ptr(ba), int(gate), _ptr(sa),
                                _ptr(O), _ptr(ST), B, H, T, dk, dv,
                                int(nthreads or default_threads()), int(mutant))
    if rc != 0:
        raise RuntimeError(f"gla_oracle_fwd failed with status {rc}")
    return O, ST


def gla_backward(q, k, v, log_g, gate, S0, dO, dST=None, want_dS0=True, nthreads=None, mutant=0, log_b=None):
    """Gradients of L = <dO, O> + <dST, S_T> through the recurrence (the adjoint
    recurrence, fp64). Returns (dq, dk, dv, dlog_g, dS0) as numpy arrays;
    dlog_g is shaped like log_g (None without a gate), dS0 None unless wanted.
    The bilinear gate (gate = GATE_BILINEAR, log_b [B,H,T,dv]) appends dlog_b."""
    qa, ka, va = _f64(q), _f64(k), _f64(v)
    B, H, T, dk = qa.shape
    dv = va.shape[-1]
    if gate is None:
        if log_g is None:
            gate = GATE_NONE
        else:
            gate = {1: GATE_HEAD_SCALAR, 3: GATE_TOKEN_SCALAR}.get(np.ndim(_f64(log_g)), GATE_PER_KEY)
    ga = _f64(log_g) if gate != GATE_NONE else None
    sa, doa, dsta = _f64(S0), _f64(dO), _f64(dST)
    lba = _f64(log_b) if gate == GATE_BILINEAR else None
    dlb = np.empty((B, H, T, dv)) if gate == GATE_BILINEAR else None
    dq = np.empty((B, H, T, dk)); dk_ = np.empty((B, H, T, dk)); dv_ = np.empty((B, H, T, dv))
    dg = None if gate == GATE_NONE else np.empty(ga.shape)
    dS0 = np.empty((B, H, dk, dv)) if want_dS0 else None
    rc = _load().gla_oracle_bwd(_ptr(qa), _ptr(ka), _ptr(va), _ptr(ga), int(gate), _ptr(sa), _ptr(doa),
                                _ptr(dsta), _ptr(dq), _ptr(dk_), _ptr(dv_), _ptr(dg), _ptr(dS0),
                                B, H, T, dk, dv, int(nthreads or default_threads()), int(mutant),
                                _ptr(lba), _ptr(dlb))
    if rc != 0:
        raise RuntimeError(f"gla_oracle_bwd failed with status {rc}")
    if gate == GATE_BILINEAR:
        return dq, dk_, dv_, dg, dS0, dlb
    return dq, dk_, dv_, dg, dS0


def gla_forward_rows(q, k, v, log_g, gate, S0, bh_list, nthreads=None, log_b=None):
    """Oracle restricted to a subset of (b,h) pairs; returns {bh: (O[T,dv], ST[dk,dv])}.

    Used to check full-size launches on sampled heads: each (b,h) is an
    independent problem, so running the recurrence on one head alone gives
    that head's exact result.
    """
    out = {}
    qa, ka, va = _f64(q), _f64(k), _f64(v)
    B, H, T, dk = qa.shape
    ga = None if gate == GATE_NONE else _f64(log_g)
    sa = _f64(S0)
    for (b, h) in bh_list:
        g1 = None
        if gate in (GATE_PER_KEY, GATE_TOKEN_SCALAR):
            g1 = ga[b:b + 1, h:h + 1]
        elif gate == GATE_HEAD_SCALAR:
            g1 = ga[h:h + 1]
        s1 = None if sa is None else sa[b:b + 1, h:h + 1]
        b1 = None if gate != GATE_BILINEAR else _f64(log_b)[b:b + 1, h:h + 1]
        if gate == GATE_BILINEAR:
            g1 = ga[b:b + 1, h:h + 1]
        O, ST = gla_forward(qa[b:b + 1, h:h + 1], ka[b:b + 1, h:h + 1], va[b:b + 1, h:h + 1],
                            g1, gate, s1, True, nthreads, log_b=b1)
        out[(b, h)] = (O[0, 0], ST[0, 0])
    return out


def segment_pair(k, v, log_g=None, gate=None):
    """The exchange pair of one sequence segment ("Gated Linear Attention Transformers
    with Hardware-Efficient Training", §2.2: the state a segment hands to the next).

    log_Gamma [B,H,dk]: the sum over the segment's tokens of log alpha_t per key (the
    log of the product of the gates; T log lambda_h for a per-head gate, 0 without one).
    S_star [B,H,dk,dv]: the recurrence's final state from S0 = 0 (q does not enter it).
    Both fp64 numpy arrays; not for the bilinear gate.
    """
    ka, va = _f64(k), _f64(v)
    B, H, T, dk = ka.shape
    if gate is None:
        gate = GATE_NONE if log_g is None else {1: GATE_HEAD_SCALAR, 3: GATE_TOKEN_SCALAR}.get(
            np.ndim(_f64(log_g)), GATE_PER_KEY)
    if gate == GATE_BILINEAR:
        raise ValueError("the bilinear gate's decay is a dk x dv matrix, not a key vector")
    _, S_star = gla_forward(ka, ka, va, log_g, gate, None)
    ga = None if gate == GATE_NONE else _f64(log_g)
    if gate == GATE_NONE:
        lg = np.zeros((B, H, dk))
    elif gate == GATE_HEAD_SCALAR:
        lg = np.broadcast_to((T * ga)[None, :, None], (B, H, dk)).copy()
    elif gate == GATE_PER_KEY:
        lg = ga.sum(axis=2)
    else:
        lg = np.broadcast_to(ga.sum(axis=2)[..., None], (B, H, dk)).copy()
    return lg, S_star


def pair_scan(log_Gammas, S_stars, S0=None):
    """The states entering P consecutive segments and the state after the last, from
    their pairs in sequence order: S = S0 (or 0); for each segment d, S_in[d] = S and
    S = Diag(exp(log_Gamma_d)) S + S*_d. Returns (S_in [P,B,H,dk,dv], S_T), fp64."""
    lgs = [_f64(x) for x in log_Gammas]
    sss = [_f64(x) for x in S_stars]
    S = np.zeros_like(sss[0]) if S0 is None else _f64(S0).copy()
    S_in = []
    for lg, ss in zip(lgs, sss):
        S_in.append(S.copy())
        S = np.exp(lg)[..., None] * S + ss
    return np.stack(S_in), S
