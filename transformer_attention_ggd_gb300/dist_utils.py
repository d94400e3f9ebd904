"""Cross-rank helpers for data-parallel use of the attention path.

The path shards by (b, h): forward, decode and dQ/dK/dV need no exchange.
A data-parallel training step over a batch split across ranks has one real
exchange, the sum of the per-head scalar gradients (dalpha, dbeta, dmu, ds:
4*H floats), done here as one flat all-reduce.  Timing across ranks takes
the slowest rank.
"""

from __future__ import annotations


def shard_batch(B: int, rank: int, world: int) -> tuple[int, int]:
    """[start, stop) of the batch rows owned by `rank` (contiguous, balanced)."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError("bad rank/world")
    base, extra = divmod(B, world)
    start = rank * base + min(rank, extra)
    return start, start + base + (1 if rank < extra else 0)


def allreduce_head_grads(grads, dist, group=None):
    """Sum the per-head scalar gradients over ranks, in place (one collective)."""
    import torch
    flat = torch.cat([g.reshape(-1) for g in grads])
    dist.all_reduce(flat, op=dist.ReduceOp.SUM, group=group)
    off = 0
    for g in grads:
        n = g.numel()
        g.copy_(flat[off:off + n].view_as(g))
        off += n
    return grads


def max_over_ranks(value: float, dist, device=None) -> float:
    """The largest `value` over all ranks (the job's time is the slowest rank's)."""
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())
