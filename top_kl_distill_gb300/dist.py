"""Host side of running the row losses on several GPUs of one node.

One process per GPU (torchrun sets RANK, LOCAL_RANK, WORLD_SIZE).  Rows are
independent units -- every per-row output (loss, lse, gradient row, top-k)
depends on its own row only -- so a batch is split into contiguous row shards
and no collective touches the per-row data.  The one exchange step is the mean
over the loss window, which spans the shards: each rank takes the mean over its
part of the window (vl_window_mean, or the mean output of the loss call) and one
all-reduce of mean x count gives the batch's mean.
"""
from __future__ import annotations

import os


def world() -> tuple[int, int, int]:
    """(world size, rank, local rank) from the launcher's environment; (1, 0, 0) when alone."""
    return (int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")),
            int(os.environ.get("LOCAL_RANK", "0")))


def shard(ntok: int, rank: int, ws: int) -> tuple[int, int]:
    """Rows [r0, r1) of rank `rank` out of `ws`: contiguous, sizes differing by at most one."""
    if ws < 1 or not 0 <= rank < ws or ntok < 0:
        raise ValueError(f"shard({ntok}, {rank}, {ws})")
    q, r = divmod(ntok, ws)
    r0 = rank * q + min(rank, r)
    return r0, r0 + q + (1 if rank < r else 0)


def max_over_ranks(value: float, device: str = "cuda") -> float:
    """The largest `value` over all ranks (the identity when not distributed)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t[0])


def window_shard(ntok: int, rank: int, ws: int, loss_start: int, loss_end: int) -> tuple[int, int, int, int]:
    """Rows [r0, r1) of rank `rank` and the part of the loss window [loss_start, loss_end)
    that falls inside them, relative to r0 (an empty window when none does)."""
    if not 0 <= loss_start <= loss_end <= ntok:
        raise ValueError(f"window [{loss_start}, {loss_end}) not inside [0, {ntok}]")
    r0, r1 = shard(ntok, rank, ws)
    ls = min(max(loss_start - r0, 0), r1 - r0)
    le = min(max(loss_end - r0, 0), r1 - r0)
    return r0, r1, ls, le


def global_window_mean(local_mean, local_count: int, total_count: int):
    """The mean over the whole loss window from this rank's mean over its part of it
    (a one-element tensor) and that part's row count: one all-reduce (sum) of
    local_mean x local_count in float64, divided by the window's total row count; 0 for
    an empty window, as the page's read_loss gives.  Returns a float64 one-element
    tensor on local_mean's device, the same on every rank."""
    import torch
    import torch.distributed as dist
    t = local_mean.detach().reshape(1).to(torch.float64) * float(local_count)
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        dist.all_reduce(t, op=dist.ReduceOp.SUM)
    if total_count <= 0:
        return torch.zeros_like(t)
    return t / float(total_count)
