"""Host side of running the row losses on several GPUs of one node.

One process per GPU (torchrun sets RANK, LOCAL_RANK, WORLD_SIZE).  Rows are
independent units -- every per-row output (loss, lse, gradient row, top-k)
depends on its own row only -- so a batch is split into contiguous row shards
and no collective touches the data path.  The only cross-rank step is the
reduction of a scalar (the slowest rank's time, or a loss sum) on the host side.
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
