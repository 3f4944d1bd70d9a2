"""Seeded synthetic inputs for the chunkwise GLA forward pass.

This module only draws random tensors. It holds none of the method's
arithmetic (no cumulative gates, no state, no outputs), so both the CUDA
path and the fp64 oracle can be fed from it without sharing any of the
computation they are compared on.

Workloads follow the shapes and distributions the GLA and Lightning
Attention-2 pages use:

* gate distribution: alpha = sigmoid(x)^(1/tau) with tau = 16
  ("Gated Linear Attention Transformers with Hardware-Efficient Training",
  §4.4), i.e. log alpha = logsigmoid(N(0,1)) / 16 for a standard-normal
  pre-activation;
* head shapes of the 1.3B GLA layer, d_model = 2048, d_k = d/2, d_v = d,
  4 heads (same paper, §4.4 and §5.1);
* the fixed per-head decay of Lightning Attention-2 / RetNet,
  lambda_h = 1 - 2^-(5 + 5h/H) ("Lightning Attention-2", §3.2.1);
* the data-dependent scalar gate, one gamma_t per token and head shared by
  every key (the Mamba-2, mLSTM and Gated Retention rows of Table 1 in the
  GLA paper, §4.1), drawn like Gated Retention's sigmoid(x)^(1/tau) with
  tau = 16: log gamma_t = logsigmoid(N(0,1)) / 16;
* the bilinear gate G_t = alpha_t^T beta_t (Table 1's DFW row, alpha and beta
  sigmoids of projections of x), drawn like the GLA gate on both sides:
  log alpha = logsigmoid(N(0,1)) / 16 per key and log beta likewise per value
  column.

Draw order is fixed: q, k, v, gate pre-activation, S0 (all fp32 from one
``torch.Generator('cpu')``), then each tensor is cast to its dtype (bf16 by
round-to-nearest-even), so the oracle sees exactly the values the GPU sees.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Optional

import torch

GATE_NONE = 0
GATE_HEAD_SCALAR = 1
GATE_PER_KEY = 2
GATE_TOKEN_SCALAR = 3
GATE_BILINEAR = 4

_GATE_NAMES = {"none": GATE_NONE, "scalar": GATE_HEAD_SCALAR, "per_key": GATE_PER_KEY,
               "token_scalar": GATE_TOKEN_SCALAR, "bilinear": GATE_BILINEAR}


@dataclass
class Workload:
    """Shape and distribution of one synthetic workload."""

    name: str
    B: int
    H: int
    T: int
    dk: int
    dv: int
    dtype: torch.dtype          # dtype of q, k, v and O
    gate: int                   # GATE_NONE / HEAD_SCALAR / PER_KEY / TOKEN_SCALAR / BILINEAR
    qkv_scale: str = "all"      # "all": q,k,v * dk^-0.5 ; "q": only q
    k_l2norm: bool = False      # k normalised to unit L2 norm per row
    s0_std: float = 0.0         # 0 => S0 absent (zero state)
    gate_dist: str = "logsigmoid16"  # or "steep" (log alpha = -U(0,4)) or "const:<x>"
    chunk: int = 64
    notes: str = ""
    extra: dict = field(default_factory=dict)

    def with_(self, **kw) -> "Workload":
        d = dict(self.__dict__)
        d.update(kw)
        return Workload(**d)

    @property
    def tokens(self) -> int:
        return self.B * self.T


# The five workloads. Sizes are per head.
WORKLOADS = {
    "fp32_small": Workload(
        "fp32_small", B=1, H=2, T=256, dk=64, dv=64, dtype=torch.float32,
        gate=GATE_PER_KEY, qkv_scale="q", notes="fp32 GLA, parity only"),
    "linear_attn": Workload(
        "linear_attn", B=8, H=16, T=2048, dk=128, dv=128, dtype=torch.bfloat16,
        gate=GATE_NONE, k_l2norm=True, notes="ungated causal linear attention"),
    "scalar_decay": Workload(
        "scalar_decay", B=4, H=16, T=8192, dk=128, dv=128, dtype=torch.bfloat16,
        gate=GATE_HEAD_SCALAR, notes="fixed per-head decay (Lightning Attention-2 / RetNet)"),
    "gla_1p3b": Workload(
        "gla_1p3b", B=8, H=4, T=2048, dk=256, dv=512, dtype=torch.bfloat16,
        gate=GATE_PER_KEY, s0_std=0.02, notes="GLA layer shaped like the 1.3B model"),
    "token_gate": Workload(
        "token_gate", B=8, H=4, T=2048, dk=256, dv=512, dtype=torch.bfloat16,
        gate=GATE_TOKEN_SCALAR, s0_std=0.02,
        notes="data-dependent scalar gate per token and head (Mamba-2 / mLSTM form), 1.3B layer shape"),
    "bilinear": Workload(
        "bilinear", B=8, H=4, T=2048, dk=256, dv=512, dtype=torch.bfloat16,
        gate=GATE_BILINEAR, s0_std=0.02,
        notes="bilinear gate alpha_t^T beta_t (DFW form), 1.3B layer shape"),
    "gla_wide_heads": Workload(
        "gla_wide_heads", B=8, H=2, T=2048, dk=512, dv=1024, dtype=torch.bfloat16,
        gate=GATE_PER_KEY, s0_std=0.02,
        notes="the 1.3B layer (d_model 2048, dk = d/2, dv = d) cut into 2 heads instead of 4: "
              "larger head dimensions, as in the head-count ablation; keys wider than 256"),
    "gla_long": Workload(
        "gla_long", B=1, H=4, T=65536, dk=256, dv=512, dtype=torch.bfloat16,
        gate=GATE_PER_KEY, notes="long sequence, low B*H"),
}


def scalar_log_decay(H: int) -> torch.Tensor:
    """log(lambda_h) for lambda_h = 1 - 2^-(5 + 5h/H), computed in fp64, returned fp32."""
    vals = [math.log1p(-(2.0 ** -(5.0 + 5.0 * h / H))) for h in range(H)]
    return torch.tensor(vals, dtype=torch.float64).to(torch.float32)


def make_inputs(w: Workload, seed: int = 0) -> dict:
    """Draw the inputs of workload ``w`` on the CPU.

    Returns a dict with q, k, v (``w.dtype``), log_g (fp32 or None), S0 (fp32 or
    None) and the shape fields. Layouts: q, k, log_g are [B,H,T,dk]; v is
    [B,H,T,dv]; S0 is [B,H,dk,dv]; for the per-head scalar gate log_g is [H],
    for the per-token scalar gate [B,H,T]. The bilinear gate adds log_b
    [B,H,T,dv] (drawn after log_g); log_b is None in every other mode.
    """
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    B, H, T, dk, dv = w.B, w.H, w.T, w.dk, w.dv
    q = torch.randn((B, H, T, dk), generator=g, dtype=torch.float32)
    k = torch.randn((B, H, T, dk), generator=g, dtype=torch.float32)
    v = torch.randn((B, H, T, dv), generator=g, dtype=torch.float32)
    scale = dk ** -0.5
    if w.qkv_scale == "all":
        q, k, v = q * scale, k * scale, v * scale
    elif w.qkv_scale == "q":
        q = q * scale
    if w.k_l2norm:
        k = k / k.norm(dim=-1, keepdim=True).clamp_min(1e-12)

    def draw_gate(shape):
        if w.gate_dist == "logsigmoid16":
            pre = torch.randn(shape, generator=g, dtype=torch.float32)
            return torch.nn.functional.logsigmoid(pre) / 16.0
        if w.gate_dist == "steep":
            u = torch.rand(shape, generator=g, dtype=torch.float32)
            return -4.0 * u
        if w.gate_dist.startswith("const:"):
            return torch.full(shape, float(w.gate_dist[6:]), dtype=torch.float32)
        if w.gate_dist == "zero":
            return torch.zeros(shape, dtype=torch.float32)
        raise ValueError(f"unknown gate distribution {w.gate_dist!r}")

    log_g = log_b = None
    if w.gate in (GATE_PER_KEY, GATE_TOKEN_SCALAR, GATE_BILINEAR):
        log_g = draw_gate((B, H, T, dk) if w.gate != GATE_TOKEN_SCALAR else (B, H, T))
        if w.gate == GATE_BILINEAR:
            log_b = draw_gate((B, H, T, dv))
    elif w.gate == GATE_HEAD_SCALAR:
        log_g = scalar_log_decay(H)

    S0 = None
    if w.s0_std > 0.0:
        S0 = torch.randn((B, H, dk, dv), generator=g, dtype=torch.float32) * w.s0_std

    return dict(
        q=q.to(w.dtype).contiguous(), k=k.to(w.dtype).contiguous(),
        v=v.to(w.dtype).contiguous(),
        log_g=None if log_g is None else log_g.contiguous(),
        log_b=None if log_b is None else log_b.contiguous(),
        S0=None if S0 is None else S0.contiguous(),
        gate=w.gate, B=B, H=H, T=T, dk=dk, dv=dv, chunk=w.chunk, dtype=w.dtype,
    )


def small(name: str = "gla_1p3b", **kw) -> Workload:
    """A copy of a named workload with some fields replaced (used for small parity cases)."""
    return WORKLOADS[name].with_(**kw)


def gate_from_name(s: str) -> int:
    return _GATE_NAMES[s]
