"""Pins of the oracle's theta prior (the BAM repository README's own
parameterisation, "Implementation Details": b = -exp(theta_alpha) *
(|d - mu| + eps)^theta_beta with mu = exp(theta_mu) - exp(-theta_mu)).

Each check compares against something other than that formula: dense ALiBi
and plain softmax attention (special cases), the independently pinned
(alpha, beta, mu) prior through the change of variables
alpha = exp(-theta_alpha / theta_beta), beta = theta_beta, mu = 2 sinh(theta_mu)
(exact when eps = 0), and central finite differences of the loss.
"""

import math

import numpy as np
import pytest
from scipy.special import softmax

import oracle
from oracle.oracle import PRIOR_THETA


def _p2_slopes(n):
    # "ALiBi: Attention with Linear Biases", "Code": start = 2^(-2^-(log2 n - 3)),
    # slope_h = start^(h+1)
    start = 2.0 ** (-(2.0 ** -(math.log2(n) - 3)))
    return np.array([start ** (h + 1) for h in range(n)])


def _dense(q, k, v, bias, causal):
    B, H, T, D = q.shape
    s = np.einsum("bhid,bhjd->bhij", q, k) / math.sqrt(D) + bias[None]
    if causal:
        s = np.where(np.tril(np.ones((T, T), bool))[None, None], s, -np.inf)
    m = s.max(-1, keepdims=True)
    lse = (m + np.log(np.exp(s - m).sum(-1, keepdims=True)))[..., 0]
    return np.einsum("bhij,bhjd->bhid", softmax(s, axis=-1), v), lse


@pytest.mark.parametrize("H", [4, 8])
@pytest.mark.parametrize("causal", [True, False])
def test_theta_alibi_special_case(H, causal):
    """theta_beta = 1, theta_mu = 0, theta_alpha = ln(slope): the bias is
    -slope * (|d| + eps), ALiBi plus a per-head constant that the softmax
    removes (the LSE moves by exactly -slope * eps)."""
    rng = np.random.default_rng(31 + H)
    B, T, D, eps = 2, 23, 16, 1e-5
    q, k, v = (rng.standard_normal((B, H, T, D)) for _ in range(3))
    slopes = _p2_slopes(H)
    pos = np.arange(T)
    rel = np.abs(pos[None, :] - pos[:, None]).astype(float)
    ref, ref_lse = _dense(q, k, v, -slopes[:, None, None] * rel[None], causal)
    o, lse = oracle.fwd(q, k, v, alpha=np.log(slopes), beta=np.ones(H), mu=np.zeros(H),
                        eps=eps, causal=causal, prior=PRIOR_THETA)
    np.testing.assert_allclose(o, ref, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(lse, ref_lse - (slopes * eps)[None, :, None], rtol=1e-12,
                               atol=1e-12)


@pytest.mark.parametrize("causal", [True, False])
def test_theta_nope_when_beta_zero(causal):
    """theta_beta = 0: the bias is the constant -exp(theta_alpha)."""
    rng = np.random.default_rng(41)
    B, H, T, D = 2, 3, 19, 8
    q, k, v = (rng.standard_normal((B, H, T, D)) for _ in range(3))
    ta = np.array([-1.0, 0.0, 1.3])
    ref, ref_lse = _dense(q, k, v, np.zeros((H, T, T)), causal)
    o, lse = oracle.fwd(q, k, v, alpha=ta, beta=np.zeros(H), mu=[0.0, 0.4, -1.1],
                        causal=causal, prior=PRIOR_THETA)
    np.testing.assert_allclose(o, ref, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(lse, ref_lse - np.exp(ta)[None, :, None], rtol=1e-12,
                               atol=1e-12)


def test_theta_is_the_alpha_form_under_the_change_of_variables():
    """With eps = 0 and theta_beta > 0, exp(ta) w^tb = (w / exp(-ta/tb))^tb."""
    for ta, tb, tm in [(0.3, 1.5, 0.2), (-2.0, 0.7, -0.9), (1.1, 2.5, 1.4), (0.0, 1.0, 0.0)]:
        alpha, mu = math.exp(-ta / tb), 2.0 * math.sinh(tm)
        for d in [-40, -7, -1, 0, 1, 2, 5, 33, 500]:
            bt = oracle.bias(d, ta, tb, tm, eps=0.0, prior=PRIOR_THETA)
            ba = oracle.bias(d, alpha, tb, mu, eps=1e-5)
            assert bt == pytest.approx(ba, rel=1e-12, abs=1e-300)
    rng = np.random.default_rng(43)
    B, H, T, D = 1, 3, 17, 8
    q, k, v = (rng.standard_normal((B, H, T, D)) for _ in range(3))
    ta, tb, tm = np.array([0.3, -0.5, 1.2]), np.array([1.5, 0.8, 2.0]), np.array([0.1, 0.7, -0.3])
    for causal in (True, False):
        o_t, lse_t = oracle.fwd(q, k, v, alpha=ta, beta=tb, mu=tm, eps=0.0, causal=causal,
                                ssmax=True, s=[0.5, 0.9, 1.2], prior=PRIOR_THETA)
        o_a, lse_a = oracle.fwd(q, k, v, alpha=np.exp(-ta / tb), beta=tb, mu=2 * np.sinh(tm),
                                causal=causal, ssmax=True, s=[0.5, 0.9, 1.2])
        np.testing.assert_allclose(o_t, o_a, rtol=1e-11, atol=1e-12)
        np.testing.assert_allclose(lse_t, lse_a, rtol=1e-11, atol=1e-12)


def test_theta_bias_grad_matches_finite_differences():
    for (d, ta, tb, tm) in [(5.0, 0.3, 1.5, 0.2), (1.0, -1.2, -0.8, 0.9), (3.0, 2.0, 0.5, -1.3),
                            (10.0, 0.0, 2.0, 0.0), (0.0, 0.5, 0.0, 0.4)]:
        g = oracle.bias_grad(d, ta, tb, tm, prior=PRIOR_THETA)
        fd = []
        for pos in range(3):
            x = [ta, tb, tm]
            hh = 1e-6 * max(1.0, abs(x[pos]))
            xp, xm = list(x), list(x)
            xp[pos] += hh
            xm[pos] -= hh
            fd.append((oracle.bias(d, *xp, prior=PRIOR_THETA) -
                       oracle.bias(d, *xm, prior=PRIOR_THETA)) / (2 * hh))
        np.testing.assert_allclose(g, fd, rtol=1e-7, atol=1e-10)


@pytest.mark.parametrize("causal,ssmax,T", [(True, True, 8), (False, True, 6), (True, False, 7)])
def test_theta_gradients_match_finite_differences(causal, ssmax, T):
    rng = np.random.default_rng(51 + T)
    B, H, D = 1, 3, 4
    q, k, v, dO = (rng.standard_normal((B, H, T, D)) for _ in range(4))
    # theta_mu non-zero and non-integer mu, so |d - mu| > 0 everywhere
    prm = {"alpha": np.array([0.2, -0.7, 1.1]), "beta": np.array([1.6, 0.6, -0.5]),
           "mu": np.array([0.15, -0.4, 0.33]), "s": np.array([0.5, 0.8, 1.1])}
    g = oracle.bwd(q, k, v, dO, causal=causal, ssmax=ssmax, prior=PRIOR_THETA, **prm)

    def f():
        o, _ = oracle.fwd(q, k, v, causal=causal, ssmax=ssmax, prior=PRIOR_THETA, **prm)
        return float(np.sum(o * dO))

    def fd_at(x, idx):
        h = 1e-6 * max(1.0, abs(x[idx]))
        old = x[idx]
        x[idx] = old + h
        fp = f()
        x[idx] = old - h
        fm = f()
        x[idx] = old
        return (fp - fm) / (2 * h)

    scale = max(1.0, max(np.abs(g[n]).max() for n in ("dq", "dk", "dv")))
    for name, x in (("dq", q), ("dk", k), ("dv", v)):
        fd = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            fd[idx] = fd_at(x, idx)
        np.testing.assert_allclose(g[name], fd, rtol=1e-6, atol=1e-7 * scale)
    for name, key in (("dalpha", "alpha"), ("dbeta", "beta"), ("dmu", "mu"), ("ds", "s")):
        x = prm[key]
        fd = np.array([fd_at(x, (h,)) for h in range(H)])
        np.testing.assert_allclose(g[name], fd, rtol=1e-6, atol=1e-8, err_msg=name)
