"""Head-sharded execution of exact attention over several GPUs, one process (rank) per GPU.

Every (batch, head) pair is an independent attention problem in both passes: O = softmax(scale Q K^T) V
is defined head by head (the Attention(Q,K,V) formula of the FlashAttention fable on ckw19810413.github.io,
section 概念揭曉), and the backward of one head reads only that head's tensors.  So the B*H heads of a call
split into contiguous ranges, one per rank; each rank runs the ordinary single-GPU entry points on its own
range, in its own device memory, and no data crosses between ranks while computing.  The only collective
is the optional gather that reassembles full outputs on every rank for a caller who wants them there.

The heads of a contiguous [B, H, N, d] tensor are contiguous [N, d] blocks in b-major order, so a range of
flattened heads is a contiguous slice: shards are views, never copies.
"""
from __future__ import annotations

from typing import Callable, Sequence

import torch


def head_ranges(total_heads: int, world: int) -> list[tuple[int, int]]:
    """Contiguous [start, stop) ranges of flattened heads, one per rank, in rank order.  Sizes differ by at
    most one; the first ``total_heads % world`` ranks get the larger size, and ranks beyond the head count
    get an empty range."""
    if total_heads < 0 or world < 1:
        raise ValueError("need total_heads >= 0 and world >= 1")
    base, extra = divmod(total_heads, world)
    out, start = [], 0
    for r in range(world):
        stop = start + base + (1 if r < extra else 0)
        out.append((start, stop))
        start = stop
    return out


def local_heads(t: torch.Tensor, rank: int, world: int) -> torch.Tensor:
    """This rank's heads of a contiguous [B, H, N, ...] tensor as a [1, h, N, ...] view (h may be 0)."""
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    B, H = t.shape[0], t.shape[1]
    start, stop = head_ranges(B * H, world)[rank]
    return t.reshape(B * H, *t.shape[2:])[start:stop].unsqueeze(0)


def _gather_heads(local: torch.Tensor, full_shape: Sequence[int], world: int, group=None) -> torch.Tensor:
    """All-gathers every rank's [1, h_r, ...] shard into the full [B, H, ...] tensor on every rank.  Shards are
    padded to the largest range for the collective and trimmed after it."""
    import torch.distributed as dist
    B, H = full_shape[0], full_shape[1]
    ranges = head_ranges(B * H, world)
    hmax = max(stop - start for start, stop in ranges)
    rest = tuple(full_shape[2:])
    padded = torch.zeros((hmax, *rest), dtype=local.dtype, device=local.device)
    h = local.shape[1]
    if h:
        padded[:h] = local[0]
    parts = [torch.empty_like(padded) for _ in range(world)]
    dist.all_gather(parts, padded, group=group)
    heads = [parts[r][: stop - start] for r, (start, stop) in enumerate(ranges)]
    return torch.cat(heads, dim=0).reshape(B, H, *rest)


def sharded_forward(q, k, v, scale=None, *, rank: int, world: int, gather: bool = False, group=None,
                    fwd: Callable | None = None, lse_dtype: torch.dtype = torch.float32):
    """Forward of this rank's heads.  q, k, v: full contiguous [B, H, N, d] tensors on this rank's device
    (only this rank's heads are read).  Returns (o, lse): this rank's [1, h, N, d] and [1, h, N] shards, or
    with ``gather`` the full [B, H, N, d] and [B, H, N] tensors on every rank.  ``fwd`` is the per-shard
    forward (default: the library's fa_fwd) and ``lse_dtype`` the dtype of the LSE it returns (the library's
    is float32), which a rank without heads needs for its empty shard."""
    if fwd is None:
        from . import fa_fwd as fwd
    B, H, N, d = q.shape
    lq, lk, lv = (local_heads(t, rank, world) for t in (q, k, v))
    if lq.shape[1]:
        o, lse = fwd(lq, lk, lv, scale)
    else:
        o = torch.empty((1, 0, N, d), dtype=q.dtype, device=q.device)
        lse = torch.empty((1, 0, N), dtype=lse_dtype, device=q.device)
    if not gather:
        return o, lse
    return (_gather_heads(o, (B, H, N, d), world, group), _gather_heads(lse, (B, H, N), world, group))


def sharded_backward(q, k, v, o, do, lse, scale=None, *, rank: int, world: int, gather: bool = False, group=None,
                     bwd: Callable | None = None):
    """Backward of this rank's heads.  All inputs are full contiguous tensors on this rank's device (o and lse
    as the forward produced them, full or gathered); only this rank's heads are read.  Returns (dq, dk, dv)
    shards [1, h, N, d], or with ``gather`` the full [B, H, N, d] gradients on every rank.  ``bwd`` is the
    per-shard backward (default: the library's fa_bwd)."""
    if bwd is None:
        from . import fa_bwd as bwd
    B, H, N, d = q.shape
    parts = [local_heads(t, rank, world) for t in (q, k, v, o, do, lse)]
    if parts[0].shape[1]:
        grads = bwd(*parts, scale)
    else:
        grads = tuple(torch.empty((1, 0, N, d), dtype=q.dtype, device=q.device) for _ in range(3))
    if not gather:
        return grads
    return tuple(_gather_heads(g, (B, H, N, d), world, group) for g in grads)


__all__ = ["head_ranges", "local_heads", "sharded_forward", "sharded_backward"]
