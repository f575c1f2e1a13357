"""Selective scan with the time axis cut over the ranks of a torch.distributed group.

Rank r of P holds steps [t_r, t_{r+1}) of every sequence: its own slices of
x, delta, z, Bm, Cm (and dy in the backward), each [B, L_r, ...], with L_r free
to differ between ranks.  The recurrence over a piece is an affine map of the
state entering it, h -> exp(A * sum delta) h + h_end, so one all-gather of
every rank's (h_end [B, D, N], sum of delta [B, D]) lets each rank compose the
maps of the pieces before it and start its own piece from the state the whole
sequence has there.  The backward runs the same exchange on the adjoint, from
the last piece towards the first, and adds one all-reduce of the parameter
gradients (dA, dD, d_dt_bias), which each rank sums over its own steps only.

The arithmetic runs in libssscan (ss_scan_fwd_summary, ss_scan_bwd_summary,
ss_scan_carries, ss_scan_fwd, ss_scan_bwd); this module only moves the
summaries between ranks.  With NCCL the exchange stays on the device; with any
other backend (gloo) it passes through host memory.
"""

from __future__ import annotations

import torch
import torch.distributed as dist

from . import ops


def _device_collectives(group) -> bool:
    return dist.get_backend(group) == "nccl"


def all_gather_pieces(t: torch.Tensor, group=None) -> torch.Tensor:
    """Every rank's ``t`` stacked in rank order: [P, *t.shape], on ``t``'s device."""
    world = dist.get_world_size(group)
    if _device_collectives(group):
        t = t.contiguous()
        flat = torch.empty((world * t.numel(),), device=t.device, dtype=t.dtype)  # the ranks' tensors back to back
        dist.all_gather_into_tensor(flat, t.reshape(-1), group=group)
        return flat.view((world,) + tuple(t.shape))
    h = t.detach().to("cpu").contiguous()
    parts = [torch.empty_like(h) for _ in range(world)]
    dist.all_gather(parts, h, group=group)
    return torch.stack(parts).to(t.device)


def all_reduce_sum_(t: torch.Tensor, group=None) -> torch.Tensor:
    """Sum ``t`` over the ranks, in place."""
    if _device_collectives(group):
        dist.all_reduce(t, group=group)
        return t
    h = t.detach().to("cpu")
    dist.all_reduce(h, group=group)
    t.copy_(h)
    return t


def ss_scan_fwd_sharded(x, delta, A, Bm, Cm, Dv, z, h0=None, chunk: int = 64, group=None, want_h_last: bool = True,
                        dt_bias=None, delta_softplus: bool = False):
    """Forward of this rank's piece -> ``(y, ckpt, h_last, h_in)``.

    ``h0`` is the state entering the whole sequence: the same tensor on every
    rank, or None on every rank.  ``h_in`` is the state this piece starts from
    (``h0`` on rank 0); ``ckpt`` are the piece's own checkpoints for
    :func:`ss_scan_bwd_sharded`; ``h_last`` is the state after the piece (the
    whole sequence's final state on the last rank).
    """
    rank, world = dist.get_rank(group), dist.get_world_size(group)
    h_in = h0
    if world > 1:
        h_end, dsum = ops.ss_scan_fwd_summary(x, delta, A, Bm, dt_bias=dt_bias, delta_softplus=delta_softplus)
        carry = ops.ss_scan_carries(A, all_gather_pieces(dsum, group), all_gather_pieces(h_end, group), init=h0)
        h_in = carry[rank]
    y, ckpt, h_last = ops.ss_scan_fwd(x, delta, A, Bm, Cm, Dv, z, h0=h_in, chunk=chunk, want_h_last=want_h_last,
                                      dt_bias=dt_bias, delta_softplus=delta_softplus)
    return y, ckpt, h_last, h_in


def ss_scan_bwd_sharded(x, delta, A, Bm, Cm, Dv, z, ckpt, dy, dh_last=None, chunk: int = 64, group=None, dA=None,
                        dD=None, dt_bias=None, delta_softplus: bool = False, d_dt_bias=None):
    """Backward of this rank's piece -> dict as :func:`ops.ss_scan_bwd`.

    ``dh_last`` is the gradient on the whole sequence's final state: the same
    tensor on every rank, or None on every rank.  ``dx``, ``ddelta``, ``dz``,
    ``dB``, ``dC`` are the piece's own.  ``dA``, ``dD`` (and ``d_dt_bias``) are
    the whole sequence's, the same on every rank: given accumulators must hold
    the same value on every rank (replicated parameters), and the sum over all
    pieces is added to them.  ``dh0`` is the adjoint leaving the piece's first
    step: on rank 0 the gradient of ``h0``.  ``g_in`` is the carry that arrived
    at the piece's end.
    """
    rank, world = dist.get_rank(group), dist.get_world_size(group)
    g_in = dh_last
    if world > 1:
        g_start, dsum = ops.ss_scan_bwd_summary(delta, A, Cm, z, dy, dt_bias=dt_bias, delta_softplus=delta_softplus)
        carry = ops.ss_scan_carries(A, all_gather_pieces(dsum, group), all_gather_pieces(g_start, group),
                                    init=dh_last, reverse=True)
        g_in = carry[rank]
    fused = dt_bias is not None or delta_softplus
    acc = {"dA": dA, "dD": dD, "d_dt_bias": d_dt_bias}
    # rank 0 accumulates onto the given tensors, the others start from zero; the all-reduce then gives
    # every rank (given value) + (sum over the pieces)
    own = {k: (v if rank == 0 else None) for k, v in acc.items()}
    out = ops.ss_scan_bwd(x, delta, A, Bm, Cm, Dv, z, ckpt, dy, dh_last=g_in, chunk=chunk, dA=own["dA"], dD=own["dD"],
                          dt_bias=dt_bias, delta_softplus=delta_softplus, d_dt_bias=own["d_dt_bias"])
    if world > 1:
        for k in ("dA", "dD") + (("d_dt_bias",) if fused else ()):
            all_reduce_sum_(out[k], group)
            if rank != 0 and acc[k] is not None:
                acc[k].copy_(out[k])
                out[k] = acc[k]
    out["g_in"] = g_in
    return out
