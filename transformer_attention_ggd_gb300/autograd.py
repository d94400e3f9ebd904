"""PyTorch autograd wrapper of the C ABI (argument marshalling only).

``bam_attention`` is differentiable in q, k, v, the three per-head prior
parameters and the SSMax scale s: its forward calls ``bam_attn_fwd`` and
keeps O and the LSE, its backward calls ``bam_attn_bwd``.  Both run in the
library's CUDA kernels; nothing here computes a step of the method.

With ``prior=BAM_PRIOR_THETA`` the prior tensors are the BAM README's
theta_alpha, theta_beta, theta_mu ("Implementation Details":
b = -exp(theta_alpha) (|d - mu| + eps)^theta_beta, mu = 2 sinh(theta_mu)),
so the module's parameters can be trained as the authors parameterise them.
"""

from __future__ import annotations

import torch

from . import bam_attn as ba


class BamAttention(torch.autograd.Function):
    @staticmethod
    def forward(ctx, q, k, v, alpha, beta, mu, s, causal, ssmax, prior, eps, o_dtype):
        o, lse = ba.attention_forward(q, k, v, alpha, beta, mu, s, eps=eps, causal=causal,
                                      ssmax=ssmax, o_dtype=o_dtype, prior=prior)
        ctx.save_for_backward(q, k, v, o, lse, alpha, beta, mu, s)
        ctx.cfg = (causal, ssmax, prior, eps)
        return o

    @staticmethod
    def backward(ctx, dO):
        q, k, v, o, lse, alpha, beta, mu, s = ctx.saved_tensors
        causal, ssmax, prior, eps = ctx.cfg
        dO = dO.to(torch.bfloat16).contiguous()
        dq, dk, dv, da, db, dm, ds = ba.attention_backward(
            q, k, v, o, lse, dO, alpha, beta, mu, s, eps=eps, causal=causal, ssmax=ssmax,
            prior=prior)
        return (dq, dk, dv, da, db, dm, ds if s is not None else None,
                None, None, None, None, None)


def bam_attention(q, k, v, alpha, beta, mu, s=None, *, causal=True, ssmax=False,
                  prior=ba.BAM_PRIOR_ALPHA, eps=1e-5, o_dtype=None):
    """GGD-BAM attention with autograd.

    q, k, v: bf16 CUDA tensors [B, H, T, 64] (contiguous).  alpha, beta, mu
    (and s when ssmax): fp32 CUDA tensors [H].  Returns O [B, H, T, 64] in
    ``o_dtype`` (default bf16; fp32 keeps the parity-grade output).  The
    incoming gradient of O is rounded to bf16 for the backward kernel.
    """
    if ssmax and s is None:
        raise ValueError("ssmax needs the per-head scale s")
    o_dtype = o_dtype or torch.bfloat16
    return BamAttention.apply(q, k, v, alpha, beta, mu, s if ssmax else None, bool(causal),
                              bool(ssmax), int(prior), float(eps), o_dtype)
