"""Host-side helpers for running the decode path on several GPUs.

The path has no exchange step: sequences and heads are independent, so each
rank owns a disjoint set of sequences (its own checkpoints, buffers, counts
and read copies) and no collective touches the data. The only cross-rank
traffic is for timing: a barrier around the timed region, then the maximum
elapsed time and the total number of processed tokens.
"""
from __future__ import annotations


def shard_range(total: int, rank: int, world: int) -> tuple[int, int]:
    """Contiguous, balanced split of `total` sequences over `world` ranks;
    returns [start, stop) for `rank` (the first total % world ranks get one
    more)."""
    if world < 1 or not 0 <= rank < world or total < 0:
        raise ValueError("bad shard request")
    base, extra = divmod(total, world)
    start = rank * base + min(rank, extra)
    return start, start + base + (1 if rank < extra else 0)


def aggregate(units: float, elapsed_ms: float, dist=None, device=None) -> tuple[float, float]:
    """Whole-job (units, time): the units summed over ranks, and the slowest
    rank's elapsed time. With no process group, the local values."""
    if dist is None or not dist.is_available() or not dist.is_initialized():
        return float(units), float(elapsed_ms)
    import torch
    t = torch.tensor([float(units), float(elapsed_ms)], dtype=torch.float64,
                     device=device if device is not None else "cpu")
    u = t[:1].clone()
    m = t[1:].clone()
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    dist.all_reduce(m, op=dist.ReduceOp.MAX)
    return float(u.item()), float(m.item())
