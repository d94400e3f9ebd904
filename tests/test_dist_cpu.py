"""Cross-rank helpers on CPU (gloo): the reductions, the shardings, and a dp x tp
mesh of 2 and 4 ranks whose sharded backward equals the full problem."""

import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from transformer_attention_ggd_gb300.dist_utils import (allreduce_head_grads, max_over_ranks,
                                                        shard_batch)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        H = 3
        grads = [torch.full((H,), float(rank + 1) * (w + 1)) for w in range(4)]
        allreduce_head_grads(grads, dist)
        t = max_over_ranks(10.0 + rank, dist)
        q.put((rank, [g.tolist() for g in grads], t))
    finally:
        dist.destroy_process_group()


def test_two_rank_reductions():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, grads, t in out:
        for w, g in enumerate(grads):
            assert g == [3.0 * (w + 1)] * 3   # (1 + 2) * (w + 1)
        assert t == 11.0


@pytest.mark.parametrize("B,world", [(8, 2), (7, 2), (64, 8), (1, 1), (5, 8)])
def test_shard_batch_covers_every_row_once(B, world):
    seen = []
    for r in range(world):
        a, b = shard_batch(B, r, world)
        assert 0 <= a <= b <= B
        seen.extend(range(a, b))
    assert seen == list(range(B))


# ---------------------------------------------------------------- dp x tp mesh

def _oracle_backward(q, k, v, o, lse, dO, alpha, beta, mu, s, causal=True, ssmax=True, prior=0,
                     eps=1e-5):
    """One shard's backward by the fp64 oracle (stands in for the GPU on CPU)."""
    import oracle
    r = oracle.bwd(q.numpy(), k.numpy(), v.numpy(), dO.numpy(), alpha.numpy(), beta.numpy(),
                   mu.numpy(), s.numpy(), eps=eps, causal=causal, ssmax=ssmax, prior=prior)
    return tuple(torch.from_numpy(r[n]) for n in ("dq", "dk", "dv", "dalpha", "dbeta", "dmu",
                                                  "ds"))


def _mesh_inputs(prior):
    g = torch.Generator().manual_seed(11)
    B, H, T, D = 4, 4, 9, 8
    x = {n: torch.randn(B, H, T, D, generator=g, dtype=torch.float64) for n in ("q", "k", "v", "do")}
    if prior:
        x["alpha"] = torch.tensor([0.2, -0.7, 1.1, -2.0], dtype=torch.float64)
        x["mu"] = torch.tensor([0.15, -0.4, 0.33, 0.0], dtype=torch.float64)
    else:
        x["alpha"] = torch.tensor([0.8, 2.5, 6.0, 30.0], dtype=torch.float64)
        x["mu"] = torch.tensor([0.37, 0.74, 1.5, 0.0], dtype=torch.float64)
    x["beta"] = torch.tensor([1.6, 0.6, -0.5, 1.0], dtype=torch.float64)
    x["s"] = torch.tensor([0.5, 0.8, 1.1, 0.9], dtype=torch.float64)
    return x


def _mesh_worker(rank, world, port, dp, tp, prior, q):
    from transformer_attention_ggd_gb300.dist_utils import (mesh_groups, shard_heads,
                                                            sharded_attention_backward)
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dp_group, tp_group, d, t = mesh_groups(dist, dp, tp)
        x = _mesh_inputs(prior)
        B, H = x["q"].shape[:2]
        b0, b1 = shard_batch(B, d, dp)
        h0, h1 = shard_heads(H, t, tp)
        loc = {n: x[n][b0:b1, h0:h1].contiguous() for n in ("q", "k", "v", "do")}
        hp = {n: x[n][h0:h1].contiguous() for n in ("alpha", "beta", "mu", "s")}
        res = sharded_attention_backward(loc["q"], loc["k"], loc["v"], None, None, loc["do"],
                                         hp["alpha"], hp["beta"], hp["mu"], hp["s"], dist=dist,
                                         dp_group=dp_group, backward=_oracle_backward,
                                         causal=True, ssmax=True, prior=prior)
        q.put((rank, b0, b1, h0, h1, [r.numpy() for r in res]))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("dp,tp,prior", [(2, 1, 0), (1, 2, 0), (2, 2, 0), (2, 2, 1)])
def test_sharded_step_matches_the_full_problem(dp, tp, prior):
    """Each rank of a dp x tp mesh takes its batch rows and heads; tensor
    gradients are its slice of the full ones, and after the one all-reduce
    over the data-parallel group its heads' scalar gradients are the full
    batch sums."""
    import oracle
    world, port = dp * tp, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_mesh_worker, args=(r, world, port, dp, tp, prior, q))
             for r in range(world)]
    for p in procs:
        p.start()
    out = [q.get(timeout=180) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    x = _mesh_inputs(prior)
    ref = oracle.bwd(*(x[n].numpy() for n in ("q", "k", "v", "do")),
                     *(x[n].numpy() for n in ("alpha", "beta", "mu", "s")), causal=True,
                     ssmax=True, prior=prior)
    names = ("dq", "dk", "dv", "dalpha", "dbeta", "dmu", "ds")
    for rank, b0, b1, h0, h1, res in out:
        for n, got in zip(names[:3], res[:3]):
            np.testing.assert_allclose(got, ref[n][b0:b1, h0:h1], rtol=1e-12, atol=1e-14)
        for n, got in zip(names[3:], res[3:]):
            np.testing.assert_allclose(got, ref[n][h0:h1], rtol=1e-10, atol=1e-13,
                                       err_msg=f"rank {rank} {n}")


@pytest.mark.parametrize("H,world", [(12, 2), (12, 5), (3, 4), (1, 1)])
def test_shard_heads_covers_every_head_once(H, world):
    from transformer_attention_ggd_gb300.dist_utils import shard_heads
    seen = []
    for r in range(world):
        a, b = shard_heads(H, r, world)
        seen.extend(range(a, b))
    assert seen == list(range(H))
