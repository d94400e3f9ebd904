"""Shared helpers for the GPU parity tests (device upload, oracle inputs)."""

import numpy as np
import torch

from transformer_attention_ggd_gb300.inputs import bf16_bits, bf16_to_f64

# Tolerances: O is compared in fp32 output mode with a max-abs bound of 1e-2;
# gradients (dq, dk, dv) and the per-head scalar gradients with a relative
# bound of 2e-2.  "Relative" for a tensor: max|g - g*| / max(max|g*|, 1e-3);
# for a scalar: |g - g*| / max(|g*|, 1e-2 * sum|dS X|, 1e-4 * sum P(|dP|+|Delta|)|X|).
# The last two terms only matter where the reference cancels: dS = P(dP -
# Delta) is a difference, and an fp32 evaluation with hardware exp2 (relative
# error ~2^-22) carries noise of a few 1e-7 of P(|dP| + |Delta|), which a large
# table value X (db/dbeta of an eps-clamped head) multiplies; a row with a
# single key has dS = 0 exactly.  With the 2e-2 factor the floor is 2e-6 of
# the pre-cancellation magnitude.  The tensor floor likewise keeps an
# all-zero reference (T = 1) from dividing fp32 noise by zero.
O_ATOL = 1e-2
GRAD_RTOL = 2e-2
GRAD_FLOOR = 1e-3
SCALAR_NOISE = 1e-4
# LSE is not bounded by the method's stated tolerances.  Logits are fp32 dot
# products of bf16 inputs plus an fp32 table value, so LSE carries the fp32
# representation error of the logit itself (relative ~6e-8; an eps-clamped
# bias can reach -1e6) plus the bf16 rounding of the weights in the row sum
# (relative 2^-9 per weight, averaging out): 2e-3 absolute + 1e-6 relative.
LSE_ATOL = 2e-3
LSE_RTOL = 1e-6


def dev_bf16(bits: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(device).view(
        torch.bfloat16)


def host_bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def dev_f32(x, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.asarray(x, dtype=np.float32)).to(device)


def normal_bits(rng, shape) -> np.ndarray:
    return bf16_bits(rng.standard_normal(shape, dtype=np.float32))


def params_dev(prm):
    return {n: dev_f32(prm[n]) for n in ("alpha", "beta", "mu", "s")}


def f64(bits):
    return bf16_to_f64(bits)


def scalar_rel_err(got, ref, absg, absp):
    den = np.maximum(np.maximum(np.abs(ref), 1e-2 * absg), SCALAR_NOISE * absp)
    den = np.maximum(den, 1e-30)
    return np.abs(got - ref) / den


def tensor_rel_err(got, ref):
    return np.abs(got - ref).max() / max(np.abs(ref).max(), GRAD_FLOOR)
