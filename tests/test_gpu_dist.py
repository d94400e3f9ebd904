"""The sharded backward over the library's own CUDA path.

Two processes, each a gloo rank on the one GPU, take a shard of a B x H
problem: with dp = 2 each holds half the batch rows (the per-head scalar
gradients are then summed over the two ranks, the step's one exchange); with
tp = 2 each holds half the heads (no exchange).  Each rank runs the
library's forward and `sharded_attention_backward` with the library's
`attention_backward`, and its dq, dk, dv slice and its heads' scalar
gradients must match the fp64 oracle's backward of the full problem at the
parity tolerances.  The ranks' kernels never wait on one another: the only
exchange is the host-side all-reduce of 4 H floats.
"""

import os
import socket

import numpy as np
import pytest

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

B, H, T = 4, 4, 200


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _inputs():
    from transformer_attention_ggd_gb300.inputs import bf16_bits, random_params
    rng = np.random.default_rng(2024)
    bits = {n: bf16_bits(rng.standard_normal((B, H, T, 64), dtype=np.float32))
            for n in ("q", "k", "v", "do")}
    prm = random_params(H, rng, mu_hi=5.0)
    prm["beta"][1] = -0.4
    return bits, prm


def _rank(rank, world, port, dp, tp, out):
    import torch.distributed as dist
    from transformer_attention_ggd_gb300 import bam_attn as ba
    from transformer_attention_ggd_gb300.dist_utils import (mesh_groups, shard_batch, shard_heads,
                                                            sharded_attention_backward)
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ba.load_library()
        dp_group, _, d, t = mesh_groups(dist, dp, tp)
        bits, prm = _inputs()
        b0, b1 = shard_batch(B, d, dp)
        h0, h1 = shard_heads(H, t, tp)

        def dev(n):
            x = np.ascontiguousarray(bits[n][b0:b1, h0:h1])
            return torch.from_numpy(x.view(np.int16)).cuda().view(torch.bfloat16)

        q, k, v, do = (dev(n) for n in ("q", "k", "v", "do"))
        hp = {n: torch.from_numpy(np.ascontiguousarray(prm[n][h0:h1])).cuda()
              for n in ("alpha", "beta", "mu", "s")}
        o, lse = ba.attention_forward(q, k, v, hp["alpha"], hp["beta"], hp["mu"], hp["s"],
                                      causal=True, ssmax=True)
        res = sharded_attention_backward(q, k, v, o, lse, do, hp["alpha"], hp["beta"], hp["mu"],
                                         hp["s"], dist=dist, dp_group=dp_group, causal=True,
                                         ssmax=True)
        torch.cuda.synchronize()
        out.put((rank, b0, b1, h0, h1, [r.float().cpu().numpy() for r in res]))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("dp,tp", [(2, 1), (1, 2)])
def test_sharded_backward_on_the_gpu_matches_the_full_problem(dp, tp):
    import torch.multiprocessing as mp

    import oracle
    from transformer_attention_ggd_gb300.inputs import bf16_to_f64
    from _gpu_helpers import GRAD_RTOL, scalar_rel_err, tensor_rel_err

    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    world, port = dp * tp, _free_port()
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    procs = [ctx.Process(target=_rank, args=(r, world, port, dp, tp, out)) for r in range(world)]
    for p in procs:
        p.start()
    got = [out.get(timeout=600) for _ in range(world)]
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    bits, prm = _inputs()
    ref = oracle.bwd(*(bf16_to_f64(bits[n]) for n in ("q", "k", "v", "do")), prm["alpha"],
                     prm["beta"], prm["mu"], prm["s"], causal=True, ssmax=True)
    names = ("dq", "dk", "dv", "dalpha", "dbeta", "dmu", "ds")
    for rank, b0, b1, h0, h1, res in got:
        for n, g in zip(names[:3], res[:3]):
            err = tensor_rel_err(g, ref[n][b0:b1, h0:h1])
            assert err < GRAD_RTOL, (rank, n, err)
        for w, (n, g) in enumerate(zip(names[3:], res[3:])):
            err = scalar_rel_err(g, ref[n][h0:h1], ref["absg"][w][h0:h1], ref["absp"][w][h0:h1])
            assert (err < GRAD_RTOL).all(), (rank, n, err)
