"""Shared helpers for the tests: tolerances and comparisons against the oracle."""
import numpy as np
import torch

# Tolerances of the contract: bf16 inputs with fp32 accumulation must reach
# relative Frobenius error <= 5e-3 and max-abs error <= 1e-2 * max|ref|; fp32
# inputs must hold 1e-5 on both measures. Applied to O and to S_T.
TOL = {
    torch.bfloat16: dict(rel_fro=5e-3, max_abs=1e-2),
    torch.float32: dict(rel_fro=1e-5, max_abs=1e-5),
}


def errors(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    diff = got - ref
    nref = np.linalg.norm(ref)
    rel_fro = np.linalg.norm(diff) / (nref if nref > 0 else 1.0)
    mref = np.abs(ref).max() if ref.size else 0.0
    max_abs = np.abs(diff).max() / (mref if mref > 0 else 1.0) if ref.size else 0.0
    return float(rel_fro), float(max_abs)


def assert_close(got, ref, dtype, what=""):
    t = TOL[dtype]
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    rf, ma = errors(got, ref)
    assert rf <= t["rel_fro"] and ma <= t["max_abs"], (
        f"{what}: rel_fro={rf:.3e} (tol {t['rel_fro']:.0e}), max_abs/max|ref|={ma:.3e} (tol {t['max_abs']:.0e})")
    return rf, ma


def to_np(t):
    return t.detach().to("cpu", torch.float64).numpy()
