"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle.

This module holds no part of the attention arithmetic: it draws random
numbers with numpy's PCG64 generator, rounds them to bfloat16 (round to
nearest even, done on the bit pattern) and widens them back exactly.  The GPU
path receives the bf16 bit patterns; the oracle receives the same values
widened to float64.

The five workloads follow the shapes of the pages' experiments: training at
T=512 (BAM README, training command; the gist summary, "Resultats
Empiriques"), long-context evaluation up to 32k tokens and 512x the training
length (README, "Evaluation"; summary, passkey retrieval), and decode against
a 32k cache.  The datasets (FineWeb, passkey prompts) are not available, so
N(0,1) tensors of those shapes stand in for activations, and per-head
parameters are drawn from the stated ranges.
"""

from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

D_HEAD = 64


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns (uint16), round to nearest even; a NaN
    stays a (quiet) NaN instead of rounding into the infinity pattern."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    rounded = np.where(np.isnan(x), (u >> 16) | 0x40, rounded)
    return rounded.astype(np.uint16)


def bf16_to_f32(b: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> float32 (exact)."""
    b = np.ascontiguousarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


def bf16_to_f64(b: np.ndarray) -> np.ndarray:
    return bf16_to_f32(b).astype(np.float64)


@dataclass
class Workload:
    name: str
    B: int
    H: int
    T: int                 # sequence length (Tkv for decode)
    D: int = D_HEAD
    causal: bool = True
    ssmax: bool = True
    op: str = "fwd"        # "fwd", "train" (fwd+bwd) or "decode"
    eps: float = 1e-5
    desc: str = ""
    params: dict = field(default_factory=dict)


def _loguniform(rng, lo, hi, n):
    return np.exp(rng.uniform(np.log(lo), np.log(hi), n))


def head_params(cfg: int, H: int, rng: np.random.Generator) -> dict:
    """Per-head alpha, beta, mu, s (float32) for workload `cfg` (1..5)."""
    if cfg == 1:
        assert H == 4
        a = np.array([2.0, 8.0, 32.0, 128.0])
        b = np.array([1.0, 0.5, 1.5, 2.0])
        m = np.zeros(H)
        s = np.ones(H)
    elif cfg == 3:
        a = _loguniform(rng, 1.0, 1e4, H)
        half = H // 2
        b = np.concatenate([rng.uniform(-1.0, 0.0, half), rng.uniform(0.0, 2.0, H - half)])
        m = rng.uniform(0.0, 64.0, H)
        s = rng.uniform(0.3, 1.0, H)
    else:  # 2, 4, 5: alpha log-U[1,1e3], beta U[-1,2], mu = 0, s U[0.3,1]
        a = _loguniform(rng, 1.0, 1e3, H)
        b = rng.uniform(-1.0, 2.0, H)
        m = np.zeros(H)
        s = rng.uniform(0.3, 1.0, H)
    return {k: np.asarray(val, dtype=np.float32) for k, val in
            (("alpha", a), ("beta", b), ("mu", m), ("s", s))}


WORKLOADS = {
    1: Workload("fwd_B2_H4_T256", 2, 4, 256, ssmax=False, op="fwd",
                desc="forward, no SSMax, B=2 H=4 T=256 D=64 causal"),
    2: Workload("train_B8_H12_T512", 8, 12, 512, op="train",
                desc="training step fwd+bwd, B=8 H=12 T=512 D=64 causal, BAM+SSMax"),
    3: Workload("prefill_B1_H12_T32768", 1, 12, 32768, op="fwd",
                desc="long-context prefill, B=1 H=12 T=32768 causal, BAM+SSMax"),
    4: Workload("prefill_B1_H8_T262144", 1, 8, 262144, op="fwd",
                desc="extreme extrapolation prefill, B=1 H=8 T=262144 causal, BAM+SSMax"),
    5: Workload("decode_B64_H12_Tkv32768", 64, 12, 32768, op="decode",
                desc="decode, one query per sequence, B=64 H=12 Tkv=32768, BAM+SSMax"),
}


def workload(cfg: int) -> Workload:
    return WORKLOADS[cfg]


def make_inputs(cfg: int, seed: int | None = None, B: int | None = None,
                H: int | None = None, T: int | None = None) -> dict:
    """Inputs for workload `cfg` (sizes may be overridden for small tests).

    Returns bf16 bit arrays 'q', 'k', 'v' (and 'do' for training) shaped
    [B,H,T,D] ('q' is [B,H,D] for decode), plus float32 'alpha', 'beta',
    'mu', 's' of length H.
    """
    w = WORKLOADS[cfg]
    B = w.B if B is None else B
    H = w.H if H is None else H
    T = w.T if T is None else T
    rng = np.random.default_rng(1000 + cfg if seed is None else seed)
    out = head_params(cfg, H, rng) if not (cfg == 1 and H != 4) else head_params(2, H, rng)
    D = w.D

    def normal(shape):
        return bf16_bits(rng.standard_normal(shape, dtype=np.float32))

    if w.op == "decode":
        out["q"] = normal((B, H, D))
    else:
        out["q"] = normal((B, H, T, D))
    out["k"] = normal((B, H, T, D))
    out["v"] = normal((B, H, T, D))
    if w.op == "train":
        out["do"] = normal((B, H, T, D))
    out.update(B=B, H=H, T=T, D=D, causal=w.causal, ssmax=w.ssmax, eps=w.eps)
    return out


def random_params(H: int, rng: np.random.Generator, beta_lo=-1.0, beta_hi=2.0,
                  mu_hi=0.0) -> dict:
    """Generic per-head parameters for edge-case tests."""
    return {
        "alpha": _loguniform(rng, 1.0, 1e3, H).astype(np.float32),
        "beta": rng.uniform(beta_lo, beta_hi, H).astype(np.float32),
        "mu": rng.uniform(0.0, mu_hi, H).astype(np.float32) if mu_hi > 0
        else np.zeros(H, np.float32),
        "s": rng.uniform(0.3, 1.0, H).astype(np.float32),
    }


def random_theta_params(H: int, rng: np.random.Generator) -> dict:
    """Per-head thetas of the README parameterisation (values held in the
    alpha, beta, mu slots): theta_alpha ~ U[-3, 1] (exp(theta_alpha) from
    0.05 to 2.7, around the README's "slope" and "sampled" initialisations),
    theta_beta ~ U[-1, 2] (both signs, and around its "linear" [0, 1] init),
    theta_mu ~ U[-1, 1] (mu = 2 sinh(theta_mu) within +-2.4), s ~ U[0.3, 1]."""
    return {
        "alpha": rng.uniform(-3.0, 1.0, H).astype(np.float32),
        "beta": rng.uniform(-1.0, 2.0, H).astype(np.float32),
        "mu": rng.uniform(-1.0, 1.0, H).astype(np.float32),
        "s": rng.uniform(0.3, 1.0, H).astype(np.float32),
    }
