"""torch.autograd glue: gated linear attention whose forward runs gla_fwd_ex and whose
backward runs gla_bwd, both through the C ABI. Argument marshalling only: every step of
both passes runs in the library's kernels.

    O, ST = gla_attention(q, k, v, log_g, S0)   # q, k, v bf16 or fp32; log_g, S0 fp32

Gradients reach q, k, v (in their dtype: the library returns fp32 gradients, cast here),
log_g and S0 (fp32), for every gate mode but the bilinear one. Nothing is kept from the
forward pass but its inputs: the backward recomputes the chunk states (gla_bwd's design).
"""
from __future__ import annotations

from . import binding as _b


def _function():
    import torch

    class GLAFunction(torch.autograd.Function):
        @staticmethod
        def forward(ctx, q, k, v, log_g, S0, gate):
            O, ST = _b.forward(q, k, v, log_g, S0, gate=gate)
            ctx.gate = gate
            ctx.save_for_backward(q, k, v, log_g, S0)
            return O, ST

        @staticmethod
        def backward(ctx, dO, dST):
            q, k, v, log_g, S0 = ctx.saved_tensors
            if dO is None:
                dO = torch.zeros((q.shape[0], q.shape[1], q.shape[2], v.shape[-1]), dtype=q.dtype, device=q.device)
            dO = dO.to(q.dtype).contiguous()
            dST = None if dST is None else dST.to(torch.float32).contiguous()
            want = ctx.needs_input_grad
            dq, dk, dv, dg, dS0 = _b.backward(q, k, v, log_g, S0, dO, dST, gate=ctx.gate,
                                              want_dS0=S0 is not None and want[4])
            cast = lambda g, like, need: g.to(like.dtype) if need and g is not None else None
            return (cast(dq, q, want[0]), cast(dk, k, want[1]), cast(dv, v, want[2]),
                    cast(dg, log_g, want[3]) if log_g is not None else None,
                    cast(dS0, S0, want[4]) if S0 is not None else None, None)

    return GLAFunction


_FN = None


def gla_attention(q, k, v, log_g=None, S0=None, gate=None):
    """(O, S_T) of the forward pass, differentiable in q, k, v, log_g and S0. Shapes and gate
    modes as for binding.forward; the inputs must be contiguous device tensors."""
    global _FN
    if _FN is None:
        _FN = _function()
    return _FN.apply(q, k, v, log_g, S0, gate)
