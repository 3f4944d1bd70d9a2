"""Sequence parallelism: one long sequence per (b, h) cut into consecutive
segments, one per rank of a torch.distributed group, in rank order.

A segment started from the state S_in leaves Diag(Gamma) S_in + S*, where
Gamma is the product of the gate over the segment and S* what the segment
leaves from a zero start ("Gated Linear Attention Transformers with
Hardware-Efficient Training", §2.2, the state carried between segments; the
FlashQLA talk, "core technical principles": each wrongly started segment is
corrected by one matrix per rank after a short serial recurrence over ranks).
So the ranks exchange one pair (log Gamma, S*) each, B*H*dk*(dv+1)*4 bytes,
and nothing else:

  1. every rank: its pair from a zero start (gla_segment_pair); rank 0 folds
     the sequence's initial state S0 into its own pair (gla_pair_combine);
  2. all ranks: all-gather of the pairs (the one collective);
  3. rank r: S_in = the scan over the pairs of ranks 0..r-1 (gla_pair_scan);
  4. rank r: its part of O and the state after its segment from S_in (gla_fwd_ex).

All arithmetic runs in the library's kernels; this module only orders the
calls and moves the pairs.
"""
from __future__ import annotations

from . import binding as _b


def exchange_pairs(log_Gamma, S_star, group=None):
    """All-gather every rank's pair; returns (log_Gamma [P,B,H,dk], S_star [P,B,H,dk,dv])
    stacked in group-rank order, which is the segments' order along the sequence."""
    import torch
    import torch.distributed as dist
    world = dist.get_world_size(group)
    log_Gamma, S_star = log_Gamma.contiguous(), S_star.contiguous()
    gl = [torch.empty_like(log_Gamma) for _ in range(world)]
    gs = [torch.empty_like(S_star) for _ in range(world)]
    dist.all_gather(gl, log_Gamma, group=group)
    dist.all_gather(gs, S_star, group=group)
    return torch.stack(gl), torch.stack(gs)


def entering_state(log_Gammas, S_stars, rank, stream=None):
    """The state entering segment `rank`, from the stacked pairs of the segments before
    it (the first already holding the sequence's initial state)."""
    import torch
    if rank == 0:
        B, H, dk, dv = S_stars.shape[1:]
        return torch.zeros((B, H, dk, dv), dtype=torch.float32, device=S_stars.device)
    _, S_in = _b.pair_scan(log_Gammas[:rank], S_stars[:rank], None, want_S_in=False, stream=stream)
    return S_in


def forward_sequence_parallel(q, k, v, log_g=None, S0=None, gate=None, group=None, rank=None,
                              exchange=None, path=_b.GLA_PATH_AUTO, stream=None):
    """This rank's segment of the forward pass of a sequence split over the group's ranks.

    q, k, v, log_g: this rank's tokens ([B,H,T_r,...]; a per-head gate log_g [H] is the
    same on every rank). S0: the sequence's initial state, read on rank 0 only (None:
    zero). Returns (O_r, S_r): this segment's outputs and the state after it (on the last
    rank, the sequence's final state). `rank` and `exchange(log_Gamma, S_star) -> stacked
    pairs` default to the group's rank and exchange_pairs.
    """
    if rank is None:
        import torch.distributed as dist
        rank = dist.get_rank(group)
    if exchange is None:
        def exchange(lg, ss):
            return exchange_pairs(lg, ss, group)
    log_G, S_star = _b.segment_pair(k, v, log_g, gate, q=q, path=path, stream=stream)
    if rank == 0 and S0 is not None:
        import torch
        # (log Gamma_0, S*_0) o (0, S0) = (log Gamma_0, Diag(Gamma_0) S0 + S*_0)
        lg0 = torch.zeros_like(log_G)
        s0 = S0.to(torch.float32).clone()
        _b.pair_combine(log_G, S_star, lg0, s0, stream=stream)
        log_G, S_star = lg0, s0
    log_Gs, S_stars = exchange(log_G, S_star)
    if rank == 0:
        S_in = S0
    else:
        S_in = entering_state(log_Gs, S_stars, rank, stream=stream)
    return _b.forward(q, k, v, log_g, S_in, gate=gate, path=path, stream=stream)
