"""World-size-2 checks of the cross-rank helpers on CPU (gloo)."""

import os
import socket

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
