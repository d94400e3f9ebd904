"""Pins of the fp64 oracle against what the pages and the mathematics fix.

Every check here compares the oracle with something other than itself: a
number the pages print, a closed form, a special case that reduces to a
textbook formula or a scipy routine, an invariant, or central finite
differences.  Chosen so that a dropped term, a wrong sign or index, or a
transposed operand in the oracle fails at least one of them.
"""

import math
import os

import numpy as np
import pytest
from scipy import stats
from scipy.special import softmax

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *rest = line.split()
            vals[key] = [float(x) for x in rest]
    return vals


def _p5_slopes(H):
    # "NNX ALiBi-Style Attention", "One fixed slope per head": 2^(-8(h+1)/H)
    return np.array([2.0 ** (-8.0 * (h + 1) / H) for h in range(H)])


def _p2_slopes(n):
    # "ALiBi: Attention with Linear Biases", "Code": start = 2^(-2^-(log2 n - 3)),
    # slope_h = start^(h+1)
    start = 2.0 ** (-(2.0 ** -(math.log2(n) - 3)))
    return np.array([start ** (h + 1) for h in range(n)])


def _dense_attention(q, k, v, bias, causal):
    """Plain softmax attention with an additive [H,T,T] bias, numpy fp64."""
    B, H, T, D = q.shape
    s = np.einsum("bhid,bhjd->bhij", q, k) / math.sqrt(D) + bias[None]
    if causal:
        s = np.where(np.tril(np.ones((T, T), bool))[None, None], s, -np.inf)
    w = softmax(s, axis=-1)
    return np.einsum("bhij,bhjd->bhid", w, v), w


# --------------------------------------------------------------------------
# Worked example (printed numbers)
# --------------------------------------------------------------------------

def test_worked_example_printed_values():
    g = _read_golden("alibi_worked_example.txt")
    H, T = int(g["H"][0]), int(g["T"][0])
    m = _p5_slopes(H)
    np.testing.assert_allclose(m, [1 / 4, 1 / 16, 1 / 64, 1 / 256], rtol=0, atol=0)
    q = np.zeros((1, H, T, 1))
    k = np.zeros((1, H, T, 1))
    v = np.zeros((1, H, T, 1))
    v[..., :, 0] = g["values"]
    o, _ = oracle.fwd(q, k, v, alpha=1.0 / m, beta=np.ones(H), mu=np.zeros(H),
                      causal=False, ssmax=False)
    tol = 0.5 * 10.0 ** (-g["printed_decimals"][0])
    np.testing.assert_allclose(o[0, 0, :, 0], g["head0_outputs"], rtol=0, atol=tol)
    expected = 1.0 / (1.0 + np.exp(m))
    np.testing.assert_allclose(o[0, :, 0, 0], expected, rtol=1e-14)
    np.testing.assert_allclose(o[0, :, 1, 0], 1.0 - expected, rtol=1e-14)
    # Zero content: SSMax changes nothing.
    o2, _ = oracle.fwd(q, k, v, alpha=1.0 / m, beta=np.ones(H), mu=np.zeros(H),
                       s=np.full(H, 0.7), causal=False, ssmax=True)
    np.testing.assert_allclose(o2, o, rtol=1e-15, atol=0)


def test_worked_example_causal_row0_is_value0():
    H = 4
    m = _p5_slopes(H)
    v = np.zeros((1, H, 2, 1))
    v[..., 1, 0] = 1.0
    o, _ = oracle.fwd(np.zeros_like(v), np.zeros_like(v), v, alpha=1 / m, beta=np.ones(H),
                      mu=np.zeros(H), causal=True)
    # A causal mask forbids position 0 from seeing position 1 (same section).
    assert np.all(o[0, :, 0, 0] == 0.0)


# --------------------------------------------------------------------------
# Special cases that reduce to textbook attention
# --------------------------------------------------------------------------

@pytest.mark.parametrize("H", [4, 8, 12])
@pytest.mark.parametrize("causal", [True, False])
def test_alibi_special_case(H, causal):
    rng = np.random.default_rng(7 + H)
    B, T, D = 2, 37, 16
    q, k, v = (rng.standard_normal((B, H, T, D)) for _ in range(3))
    slopes = _p2_slopes(H)
    np.testing.assert_allclose(slopes, _p5_slopes(H), rtol=1e-14)
    pos = np.arange(T)
    rel = np.abs(pos[None, :] - pos[:, None]).astype(float)
    ref, _ = _dense_attention(q, k, v, -slopes[:, None, None] * rel[None], causal)
    o, lse = oracle.fwd(q, k, v, alpha=1.0 / slopes, beta=np.ones(H), mu=np.zeros(H),
                        causal=causal)
    np.testing.assert_allclose(o, ref, rtol=1e-11, atol=1e-12)


@pytest.mark.parametrize("causal", [True, False])
def test_nope_when_beta_zero(causal):
    rng = np.random.default_rng(11)
    B, H, T, D = 2, 3, 29, 8
    q, k, v = (rng.standard_normal((B, H, T, D)) for _ in range(3))
    ref, w = _dense_attention(q, k, v, np.zeros((H, T, T)), causal)
    # beta = 0 with arbitrary alpha, mu (integer and fractional, so u = 0 occurs)
    o, lse = oracle.fwd(q, k, v, alpha=[0.5, 3.0, 70.0], beta=np.zeros(H),
                        mu=[0.0, 2.0, 5.3], causal=causal)
    np.testing.assert_allclose(o, ref, rtol=1e-11, atol=1e-12)
    # LSE of the biased logits: log-sum-exp of scores plus the constant -1.
    s = np.einsum("bhid,bhjd->bhij", q, k) / math.sqrt(D)
    if causal:
        s = np.where(np.tril(np.ones((T, T), bool))[None, None], s, -np.inf)
    ref_lse = np.log(np.exp(s).sum(-1)) - 1.0
    np.testing.assert_allclose(lse, ref_lse, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("beta", [0.5, 1.0, 1.5, 2.0, 3.0])
def test_zero_content_weights_are_the_ggd_prior(beta, causal):
    """With q = 0 the weights are the generalized normal density of d = i - j.

    scipy.stats.gennorm(beta, loc=mu, scale=alpha) has density proportional
    to exp(-|(x - mu)/alpha|^beta): the GGD prior of the gist summary,
    "Solution Proposee : GGD-BAM".  V = identity exposes the weights.
    """
    T = 12
    H = 3
    alpha = np.array([0.7, 3.0, 10.0])
    mu = np.array([0.0, 2.5, 4.0])
    q = np.zeros((1, H, T, T))
    k = np.random.default_rng(3).standard_normal((1, H, T, T))
    v = np.broadcast_to(np.eye(T), (1, H, T, T)).copy()
    o, _ = oracle.fwd(q, k, v, alpha=alpha, beta=np.full(H, beta), mu=mu, causal=causal)
    for h in range(H):
        for i in range(T):
            js = np.arange(i + 1 if causal else T)
            pdf = stats.gennorm.pdf(i - js, beta, loc=mu[h], scale=alpha[h])
            np.testing.assert_allclose(o[0, h, i, js], pdf / pdf.sum(), rtol=1e-10,
                                       atol=1e-300)
            if causal:
                assert np.all(o[0, h, i, i + 1:] == 0.0)


def test_alibi_unit_distance_ratio():
    """Each extra unit of distance multiplies the weight ratio by exp(-slope)."""
    H, T = 4, 9
    m = _p5_slopes(H)
    q = np.zeros((1, H, T, T))
    v = np.broadcast_to(np.eye(T), (1, H, T, T)).copy()
    o, _ = oracle.fwd(q, q.copy(), v, alpha=1 / m, beta=np.ones(H), mu=np.zeros(H),
                      causal=True)
    for h in range(H):
        for i in range(1, T):
            r = o[0, h, i, :i] / o[0, h, i, 1:i + 1]
            np.testing.assert_allclose(r, np.exp(-m[h]), rtol=1e-12)


def test_negative_beta_inverts_the_prior():
    """beta < 0: mass is pushed away from the query (summary, GGD-BAM bullets).

    With zero content, weights grow with |d - mu|; at d = mu the eps clamp
    (eps = 1e-5, README "Implementation Details") makes the key negligible.
    """
    T, H = 16, 2
    q = np.zeros((1, H, T, T))
    v = np.broadcast_to(np.eye(T), (1, H, T, T)).copy()
    beta = np.array([-0.5, -1.0])
    mu = np.array([3.0, 0.0])
    o, _ = oracle.fwd(q, q.copy(), v, alpha=np.array([1.0, 2.0]), beta=beta, mu=mu,
                      causal=True)
    for h in range(H):
        i = T - 1
        w = o[0, h, i, : i + 1]
        dist = np.abs((i - np.arange(i + 1)) - mu[h])
        order = np.argsort(dist, kind="stable")
        assert np.all(np.diff(w[order]) >= -1e-15), "weights must grow with |d - mu|"
        j0 = int(i - mu[h])
        assert w[j0] < 1e-100 * w.max()


def test_mu_moves_the_peak_into_the_past():
    """Reading of the offset: d = i - j and u = |d - mu|; the prior peaks at j = i - mu."""
    T, H = 20, 1
    q = np.zeros((1, H, T, T))
    v = np.broadcast_to(np.eye(T), (1, H, T, T)).copy()
    for mu in [3.0, 7.0]:
        o, _ = oracle.fwd(q, q.copy(), v, alpha=[2.0], beta=[2.0], mu=[mu], causal=True)
        for i in range(int(mu), T):
            assert int(np.argmax(o[0, 0, i, : i + 1])) == i - int(mu)


# --------------------------------------------------------------------------
# Closed-form rows, SSMax, decode
# --------------------------------------------------------------------------

def test_closed_form_rows():
    rng = np.random.default_rng(5)
    B, H, T, D = 1, 2, 7, 8
    q, k, v = (rng.standard_normal((B, H, T, D)) for _ in range(3))
    prm = dict(alpha=[3.0, 0.5], beta=[1.3, -0.4], mu=[0.0, 1.5], s=[0.6, 0.9])
    for ssmax in (False, True):
        o, _ = oracle.fwd(q, k, v, causal=True, ssmax=ssmax, **prm)
        np.testing.assert_array_equal(o[:, :, 0], v[:, :, 0])  # causal row 0 sees only key 0
    vc = np.broadcast_to(rng.standard_normal(D), (B, H, T, D)).copy()
    o, _ = oracle.fwd(q, k, vc, causal=False, ssmax=True, **prm)
    np.testing.assert_allclose(o, vc, rtol=1e-14)           # constant V
    o1, lse1 = oracle.fwd(q[:, :, :1], k[:, :, :1], v[:, :, :1], causal=True, **prm)
    np.testing.assert_array_equal(o1, v[:, :, :1])           # T = 1
    # beta > 0, mu = 0 -> b(0) = 0, so the LSE of T=1 is the scaled score
    np.testing.assert_allclose(lse1[0, 0, 0], q[0, 0, 0] @ k[0, 0, 0] / math.sqrt(D),
                               rtol=1e-14)


@pytest.mark.parametrize("causal", [True, False])
def test_ssmax_is_plain_attention_on_rescaled_queries(causal):
    rng = np.random.default_rng(9)
    B, H, T, D = 2, 3, 23, 8
    q, k, v = (rng.standard_normal((B, H, T, D)) for _ in range(3))
    prm = dict(alpha=[3.0, 40.0, 0.9], beta=[0.7, -0.8, 2.0], mu=[0.0, 4.0, 1.25])
    s = np.array([0.3, 0.75, 1.0])
    o, lse = oracle.fwd(q, k, v, s=s, causal=causal, ssmax=True, **prm)
    n = (np.arange(T) + 1) if causal else np.full(T, T)
    qs = q * (s[None, :, None, None] * np.log(n)[None, None, :, None])
    o2, lse2 = oracle.fwd(qs, k, v, causal=causal, ssmax=False, **prm)
    np.testing.assert_allclose(o, o2, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(lse, lse2, rtol=1e-12, atol=1e-13)


def test_decode_is_the_last_prefill_row():
    rng = np.random.default_rng(13)
    B, H, T, D = 3, 4, 41, 16
    q, k, v = (rng.standard_normal((B, H, T, D)) for _ in range(3))
    prm = dict(alpha=[1.5, 20.0, 300.0, 2.0], beta=[-0.7, 0.4, 1.9, 1.0],
               mu=[0.0, 3.0, 10.5, 0.0], s=[0.4, 0.5, 0.9, 1.0])
    for ssmax in (False, True):
        o, lse = oracle.fwd(q, k, v, causal=True, ssmax=ssmax, **prm)
        od, lsed = oracle.decode(q[:, :, -1], k, v, ssmax=ssmax, **prm)
        np.testing.assert_allclose(od, o[:, :, -1], rtol=1e-13, atol=1e-14)
        np.testing.assert_allclose(lsed, lse[:, :, -1], rtol=1e-13, atol=1e-14)


def test_fwd_rows_matches_full():
    rng = np.random.default_rng(17)
    B, H, T, D = 2, 3, 50, 8
    q, k, v = (rng.standard_normal((B, H, T, D)) for _ in range(3))
    prm = dict(alpha=[1.5, 20.0, 3.0], beta=[-0.7, 0.4, 1.9], mu=[0.0, 3.0, 10.5],
               s=[0.4, 0.5, 0.9])
    o, lse = oracle.fwd(q, k, v, causal=True, ssmax=True, **prm)
    rows = np.array([0, 7, 49, 50, 199, 299])
    orow, lrow = oracle.fwd_rows(q, k, v, rows, causal=True, ssmax=True, **prm)
    np.testing.assert_array_equal(orow, o.reshape(-1, D)[rows])
    np.testing.assert_array_equal(lrow, lse.reshape(-1)[rows])


# --------------------------------------------------------------------------
# Gradients against central finite differences
# --------------------------------------------------------------------------

def _loss(q, k, v, dO, prm, causal, ssmax):
    o, _ = oracle.fwd(q, k, v, causal=causal, ssmax=ssmax, **prm)
    return float(np.sum(o * dO))


def _fd(f, x, idx):
    h = 1e-6 * max(1.0, abs(x[idx]))
    old = x[idx]
    x[idx] = old + h
    fp = f()
    x[idx] = old - h
    fm = f()
    x[idx] = old
    return (fp - fm) / (2 * h)


@pytest.mark.parametrize("causal,ssmax,T,mu0,beta", [
    (True, True, 9, 0.37, (1.7, 0.5, -0.6)),
    (False, True, 6, 0.37, (1.7, 0.5, -0.6)),
    # Integer mu: u = 0 occurs.  beta >= 1 there (a central difference across
    # the cusp of |x|^beta, beta < 1, is not a derivative), and beta < 0 where
    # the eps clamp is active (db/dmu = 0 inside the clamp).
    (True, False, 7, 1.0, (1.7, 1.0, -0.6)),
])
def test_gradients_match_finite_differences(causal, ssmax, T, mu0, beta):
    rng = np.random.default_rng(21 + T)
    B, H, D = 1, 3, 4
    q, k, v, dO = (rng.standard_normal((B, H, T, D)) for _ in range(4))
    prm = {"alpha": np.array([0.8, 2.5, 6.0]), "beta": np.array(beta),
           "mu": np.array([mu0, 2 * mu0, mu0]), "s": np.array([0.5, 0.8, 1.1])}
    g = oracle.bwd(q, k, v, dO, causal=causal, ssmax=ssmax, **prm)

    def f():
        return _loss(q, k, v, dO, prm, causal, ssmax)

    scale = max(1.0, max(np.abs(g[n]).max() for n in ("dq", "dk", "dv")))
    for name, x in (("dq", q), ("dk", k), ("dv", v)):
        fd = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            fd[idx] = _fd(f, x, idx)
        np.testing.assert_allclose(g[name], fd, rtol=1e-6, atol=1e-7 * scale)
    for name, key in (("dalpha", "alpha"), ("dbeta", "beta"), ("dmu", "mu"), ("ds", "s")):
        x = prm[key]
        fd = np.array([_fd(f, x, (h,)) for h in range(H)])
        np.testing.assert_allclose(g[name], fd, rtol=1e-6, atol=1e-8, err_msg=name)
    if not ssmax:
        assert np.all(g["ds"] == 0.0)
    # Invariant: softmax weights sum to one, so sum_j dv_j = sum_i dO_i.
    np.testing.assert_allclose(g["dv"].sum(axis=2), dO.sum(axis=2), rtol=1e-12, atol=1e-12)
    # absg bounds each scalar gradient, and absp bounds absg
    # (|dS X| = P |dP - Delta| |X| <= P (|dP| + |Delta|) |X|).
    for w, name in enumerate(("dalpha", "dbeta", "dmu", "ds")):
        assert np.all(np.abs(g[name]) <= g["absg"][w] * (1 + 1e-12) + 1e-300)
        assert np.all(g["absg"][w] <= g["absp"][w] * (1 + 1e-12) + 1e-300)


def test_bias_grad_matches_finite_differences():
    for (d, a, b, m) in [(5.0, 2.0, 1.5, 0.3), (1.0, 7.0, -0.8, 2.6), (3.0, 0.5, 0.5, 4.2),
                         (10.0, 30.0, 2.0, 0.0)]:
        g = oracle.bias_grad(d, a, b, m)
        fd = []
        for pos in range(3):
            x = [a, b, m]
            hh = 1e-6 * max(1.0, abs(x[pos]))
            xp = list(x)
            xm = list(x)
            xp[pos] += hh
            xm[pos] -= hh
            fd.append((oracle.bias(d, *xp) - oracle.bias(d, *xm)) / (2 * hh))
        np.testing.assert_allclose(g, fd, rtol=1e-7, atol=1e-10)
