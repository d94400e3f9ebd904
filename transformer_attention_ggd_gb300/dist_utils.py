"""Cross-rank helpers for sharded use of the attention path.

The path shards by (b, h): forward, decode and dQ/dK/dV need no exchange.
Batch rows split across data-parallel ranks share the per-head prior and
SSMax parameters, so a training step has one real exchange, the sum of the
per-head scalar gradients (dalpha, dbeta, dmu, ds: 4*H floats of the heads
the rank holds), done here as one flat all-reduce over the data-parallel
group.  Heads split across tensor-parallel ranks (each rank holds the q, k, v
columns of its heads, as a column-split QKV projection gives them) need no
exchange at all: a head's scalar gradients come from that rank alone.  On a
dp x tp mesh the reduction runs over the ranks that hold the same heads.
Timing across ranks takes the slowest rank.
"""

from __future__ import annotations


def shard_batch(B: int, rank: int, world: int) -> tuple[int, int]:
    """[start, stop) of the batch rows owned by `rank` (contiguous, balanced)."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError("bad rank/world")
    base, extra = divmod(B, world)
    start = rank * base + min(rank, extra)
    return start, start + base + (1 if rank < extra else 0)


def shard_heads(H: int, rank: int, world: int) -> tuple[int, int]:
    """[start, stop) of the heads owned by tensor-parallel `rank`."""
    return shard_batch(H, rank, world)


def mesh_groups(dist, dp: int, tp: int):
    """Process groups of a dp x tp mesh, rank = d * tp + t (every rank must
    call this, in the same order).  Returns (dp_group, tp_group, d, t): the
    ranks holding the same heads (t fixed) and the ranks holding the same
    batch rows (d fixed)."""
    world = dist.get_world_size()
    if dp * tp != world:
        raise ValueError(f"dp * tp = {dp * tp} != world size {world}")
    rank = dist.get_rank()
    d, t = divmod(rank, tp)
    dp_group = tp_group = None
    for tt in range(tp):
        g = dist.new_group([dd * tp + tt for dd in range(dp)])
        if tt == t:
            dp_group = g
    for dd in range(dp):
        g = dist.new_group([dd * tp + tt for tt in range(tp)])
        if dd == d:
            tp_group = g
    return dp_group, tp_group, d, t


def sharded_attention_backward(q, k, v, o, lse, dO, alpha, beta, mu, s=None, *, dist=None,
                               dp_group=None, backward=None, **kw):
    """Backward of this rank's shard: q, k, v, o, lse, dO hold its batch rows
    and heads, alpha, beta, mu, s its heads.  dq, dk, dv come back final; the
    per-head scalar gradients are summed over `dp_group` (skipped when `dist`
    is None or the group has one rank).  `backward` computes one shard; it
    defaults to the library's ``attention_backward`` (keyword options such
    as causal, ssmax, prior and eps pass through)."""
    if backward is None:
        from .bam_attn import attention_backward as backward
    dq, dk, dv, *g = backward(q, k, v, o, lse, dO, alpha, beta, mu, s, **kw)
    if dist is not None and dist.get_world_size(dp_group) > 1:
        allreduce_head_grads(g, dist, dp_group)
    return (dq, dk, dv, *g)


def allreduce_head_grads(grads, dist, group=None):
    """Sum the per-head scalar gradients over ranks, in place (one collective
    of 4 H floats).  With the gloo backend, device tensors are reduced
    through one host copy (gloo reduces host memory)."""
    import torch
    flat = torch.cat([g.reshape(-1) for g in grads])
    if flat.is_cuda and dist.get_backend(group) == "gloo":
        host = flat.cpu()
        dist.all_reduce(host, op=dist.ReduceOp.SUM, group=group)
        flat.copy_(host)
    else:
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
