"""GPU parity of the theta prior (the BAM README's parameterisation,
"Implementation Details": b = -exp(theta_alpha) (|d - mu| + eps)^theta_beta,
mu = 2 sinh(theta_mu)) through the C ABI, and of the autograd wrapper, against
the oracle's theta prior."""

import math

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
from oracle.oracle import PRIOR_ALPHA, PRIOR_THETA
from transformer_attention_ggd_gb300 import bam_attn as ba
from transformer_attention_ggd_gb300.inputs import make_inputs, random_theta_params

from _gpu_helpers import (GRAD_RTOL, LSE_ATOL, LSE_RTOL, O_ATOL, dev_bf16, f64, normal_bits,
                          params_dev, scalar_rel_err, tensor_rel_err)

pytestmark = pytest.mark.gpu
TH = ba.BAM_PRIOR_THETA


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    ba.load_library()


THETAS = {"alpha": np.array([0.3, -1.5, 1.0, -3.0, 0.0, 0.7], np.float32),
          "beta": np.array([1.5, -0.5, 2.0, 0.0, 1.0, -1.0], np.float32),
          "mu": np.array([0.0, 0.37, -0.8, 1.2, 0.05, -0.3], np.float32),
          "s": np.ones(6, np.float32)}


def _table_tol(d, tb, tm, plane):
    """1e-6 relative, plus the effect of mu = 2 sinh(theta_mu) being formed
    in fp32 (a few ulp of mu, dmu) on w = |d - mu| + eps: relative dmu / w
    through w^theta_beta and 1/w, and dmu / (w |ln w|) through ln w."""
    mu = 2.0 * math.sinh(float(tm))
    w = np.abs(d - mu) + 1e-5
    dmu = 8.0 * float(np.spacing(np.float32(abs(mu) + 1e-30)))
    amp = abs(float(tb)) + 1.0
    if plane == "db/dtheta_beta":
        amp = amp + 1.0 / np.maximum(np.abs(np.log(w)), 1e-30)
    return 1e-6 + amp * dmu / w


@pytest.mark.parametrize("causal", [True, False])
def test_theta_tables_match_oracle(causal):
    """Forward plane (b log2 e) and the backward planes (db/dtheta_beta,
    db/dtheta_mu), copy 0 of each, entry by entry."""
    T, H = 700, 6
    prm = THETAS
    z = dev_bf16(np.zeros((1, H, T, 64), np.uint16))
    t = params_dev(prm)
    ws_f = ba.workspace(ba.BAM_OP_FWD, 1, H, T)
    o, lse = ba.attention_forward(z, z, z, t["alpha"], t["beta"], t["mu"], t["s"],
                                  causal=causal, ws=ws_f, prior=TH)
    ws_b = ba.workspace(ba.BAM_OP_BWD, 1, H, T)
    ba.attention_backward(z, z, z, o, lse, z, t["alpha"], t["beta"], t["mu"], t["s"],
                          causal=causal, ws=ws_b, prior=TH)
    torch.cuda.synchronize()
    t256 = (T + 255) // 256 * 256
    off = 256 if causal else t256 + 256
    length = off + t256 + 256
    fwd = ws_f[256:256 + 4 * H * length * 4].cpu().numpy().view(np.float32)
    fwd = fwd.reshape(4, H, length)
    bwd = ws_b[256:256 + 3 * 4 * H * length * 4].cpu().numpy().view(np.float32)
    bwd = bwd.reshape(3, 4, H, length)
    log2e = 1.0 / math.log(2.0)
    d = np.arange(length) - off
    for h in range(H):
        a, b, m = prm["alpha"][h], prm["beta"][h], prm["mu"][h]
        ref_b = np.array([oracle.bias(x, a, b, m, prior=PRIOR_THETA) for x in d]) * log2e
        ref_g = np.array([oracle.bias_grad(x, a, b, m, prior=PRIOR_THETA) for x in d])
        for got, ref, name in ((fwd[0, h, ::-1], ref_b, "b"), (bwd[0, 0, h, ::-1], ref_b, "b"),
                               (bwd[1, 0, h, ::-1], ref_g[:, 1], "db/dtheta_beta"),
                               (bwd[2, 0, h, ::-1], ref_g[:, 2], "db/dtheta_mu")):
            ref = np.clip(ref, -3.0e38, 3.0e38)
            err = np.abs(got - ref) / np.maximum(np.abs(ref), 1e-30)
            bad = err > _table_tol(d, b, m, name)
            # entries whose reference is exactly 0 (d = mu never occurs with
            # eps > 0, so only db/dtheta_beta at w = 1) compare absolutely
            bad &= ~((ref == 0.0) & (np.abs(got) <= 1e-6))
            assert not bad.any(), (name, h, int(d[bad.argmax()]), got[bad.argmax()],
                                   ref[bad.argmax()])


def _fwd_pair(bits, prm, causal, ssmax):
    t = params_dev(prm)
    q, k, v = (dev_bf16(bits[n]) for n in "qkv")
    o, lse = ba.attention_forward(q, k, v, t["alpha"], t["beta"], t["mu"], t["s"],
                                  causal=causal, ssmax=ssmax, prior=TH)
    torch.cuda.synchronize()
    oref, lref = oracle.fwd(f64(bits["q"]), f64(bits["k"]), f64(bits["v"]), prm["alpha"],
                            prm["beta"], prm["mu"], prm["s"], causal=causal, ssmax=ssmax,
                            prior=PRIOR_THETA)
    return o.cpu().numpy(), lse.cpu().numpy(), oref, lref


@pytest.mark.parametrize("T", [1, 17, 129, 300])
@pytest.mark.parametrize("causal,ssmax", [(True, True), (False, True), (True, False)])
def test_theta_forward_small_ragged(T, causal, ssmax):
    rng = np.random.default_rng(300 + T + 7 * causal + 3 * ssmax)
    bits = {n: normal_bits(rng, (2, 3, T, 64)) for n in "qkv"}
    prm = random_theta_params(3, rng)
    prm["beta"][0] = -0.7
    o, lse, oref, lref = _fwd_pair(bits, prm, causal, ssmax)
    np.testing.assert_allclose(o, oref, rtol=0, atol=O_ATOL)
    np.testing.assert_allclose(lse, lref, rtol=LSE_RTOL, atol=LSE_ATOL)


@pytest.mark.parametrize("T", [513, 2048])
@pytest.mark.parametrize("causal", [True, False])
def test_theta_forward_long_sequence_kernel(T, causal):
    """The theta prior through the long-sequence forward (256-row CTAs, which
    run when they fill two waves of the SMs): two heads repeated over 160
    batch rows, every row against the oracle's two heads."""
    rng = np.random.default_rng(T + 5 * causal)
    bits = {n: normal_bits(rng, (1, 2, T, 64)) for n in "qkv"}
    prm = random_theta_params(2, rng)
    prm["beta"][0] = -0.6
    t = params_dev(prm)
    rep = {n: dev_bf16(np.ascontiguousarray(np.repeat(b, 160, axis=0))) for n, b in bits.items()}
    o, lse = ba.attention_forward(rep["q"], rep["k"], rep["v"], t["alpha"], t["beta"], t["mu"],
                                  t["s"], causal=causal, ssmax=True, prior=TH)
    torch.cuda.synchronize()
    oref, lref = oracle.fwd(f64(bits["q"]), f64(bits["k"]), f64(bits["v"]), prm["alpha"],
                            prm["beta"], prm["mu"], prm["s"], causal=causal, ssmax=True,
                            prior=PRIOR_THETA)
    o, lse = o.cpu().numpy(), lse.cpu().numpy()
    np.testing.assert_allclose(o, np.repeat(oref, 160, axis=0), rtol=0, atol=O_ATOL)
    np.testing.assert_allclose(lse, np.repeat(lref, 160, axis=0), rtol=LSE_RTOL, atol=LSE_ATOL)


def _bwd_compare(bits, prm, causal, ssmax):
    t = params_dev(prm)
    q, k, v, g = (dev_bf16(bits[n]) for n in ("q", "k", "v", "do"))
    o, lse = ba.attention_forward(q, k, v, t["alpha"], t["beta"], t["mu"], t["s"],
                                  causal=causal, ssmax=ssmax, prior=TH)
    out = ba.attention_backward(q, k, v, o, lse, g, t["alpha"], t["beta"], t["mu"], t["s"],
                                causal=causal, ssmax=ssmax, prior=TH)
    torch.cuda.synchronize()
    names = ("dq", "dk", "dv", "dalpha", "dbeta", "dmu", "ds")
    got = {n: x.float().cpu().numpy() for n, x in zip(names, out)}
    ref = oracle.bwd(f64(bits["q"]), f64(bits["k"]), f64(bits["v"]), f64(bits["do"]),
                     prm["alpha"], prm["beta"], prm["mu"], prm["s"], causal=causal,
                     ssmax=ssmax, prior=PRIOR_THETA)
    for n in ("dq", "dk", "dv"):
        rel = tensor_rel_err(got[n], ref[n])
        assert rel <= GRAD_RTOL, f"{n}: relative error {rel:.3e}"
    for w, n in enumerate(("dalpha", "dbeta", "dmu", "ds")):
        if n == "ds" and not ssmax:
            assert np.all(got[n] == 0.0)
            continue
        err = scalar_rel_err(got[n], ref[n], ref["absg"][w], ref["absp"][w])
        assert err.max() <= GRAD_RTOL, f"{n}: {got[n]} vs {ref[n]} (err {err.max():.3e})"


@pytest.mark.parametrize("T", [2, 129, 300])
@pytest.mark.parametrize("causal,ssmax", [(True, True), (False, True), (True, False)])
def test_theta_backward_small_ragged(T, causal, ssmax):
    rng = np.random.default_rng(400 + T + 7 * causal + 3 * ssmax)
    bits = {n: normal_bits(rng, (2, 3, T, 64)) for n in ("q", "k", "v", "do")}
    prm = random_theta_params(3, rng)
    prm["beta"][1] = -0.5
    _bwd_compare(bits, prm, causal, ssmax)


def test_theta_training_step_full_size():
    """The B=8 H=12 T=512 training step with theta parameters."""
    d = make_inputs(2)
    bits = {n: d[n] for n in ("q", "k", "v", "do")}
    prm = random_theta_params(12, np.random.default_rng(2024))
    _bwd_compare(bits, prm, True, True)


@pytest.mark.parametrize("Tkv", [1, 65, 4097])
def test_theta_decode(Tkv):
    rng = np.random.default_rng(500 + Tkv)
    B, H = 2, 3
    q = normal_bits(rng, (B, H, 64))
    kc, vc = normal_bits(rng, (B, H, Tkv, 64)), normal_bits(rng, (B, H, Tkv, 64))
    prm = random_theta_params(H, rng)
    t = params_dev(prm)
    o, lse = ba.attention_decode(dev_bf16(q), dev_bf16(kc), dev_bf16(vc), t["alpha"], t["beta"],
                                 t["mu"], t["s"], ssmax=True, prior=TH)
    torch.cuda.synchronize()
    oref, lref = oracle.decode(f64(q), f64(kc), f64(vc), prm["alpha"], prm["beta"], prm["mu"],
                               prm["s"], ssmax=True, prior=PRIOR_THETA)
    np.testing.assert_allclose(o.cpu().numpy(), oref, rtol=0, atol=O_ATOL)
    np.testing.assert_allclose(lse.cpu().numpy(), lref, rtol=LSE_RTOL, atol=LSE_ATOL)


@pytest.mark.parametrize("prior", [PRIOR_ALPHA, PRIOR_THETA])
def test_autograd_wrapper_matches_oracle(prior):
    from transformer_attention_ggd_gb300.autograd import bam_attention
    rng = np.random.default_rng(600 + prior)
    B, H, T = 2, 3, 200
    bits = {n: normal_bits(rng, (B, H, T, 64)) for n in ("q", "k", "v", "do")}
    if prior == PRIOR_THETA:
        prm = random_theta_params(H, rng)
    else:
        from transformer_attention_ggd_gb300.inputs import random_params
        prm = random_params(H, rng, mu_hi=3.0)
    q, k, v = (dev_bf16(bits[n]).requires_grad_() for n in "qkv")
    t = {n: x.requires_grad_() for n, x in params_dev(prm).items()}
    o = bam_attention(q, k, v, t["alpha"], t["beta"], t["mu"], t["s"], causal=True, ssmax=True,
                      prior=prior, o_dtype=torch.float32)
    dO = dev_bf16(bits["do"]).float()
    (o * dO).sum().backward()
    torch.cuda.synchronize()
    oref, _ = oracle.fwd(f64(bits["q"]), f64(bits["k"]), f64(bits["v"]), prm["alpha"],
                         prm["beta"], prm["mu"], prm["s"], causal=True, ssmax=True,
                         prior=prior)
    np.testing.assert_allclose(o.detach().cpu().numpy(), oref, rtol=0, atol=O_ATOL)
    ref = oracle.bwd(f64(bits["q"]), f64(bits["k"]), f64(bits["v"]), f64(bits["do"]),
                     prm["alpha"], prm["beta"], prm["mu"], prm["s"], causal=True, ssmax=True,
                     prior=prior)
    for n, x in (("dq", q), ("dk", k), ("dv", v)):
        rel = tensor_rel_err(x.grad.float().cpu().numpy(), ref[n])
        assert rel <= GRAD_RTOL, f"{n}: relative error {rel:.3e}"
    for w, (n, key) in enumerate((("dalpha", "alpha"), ("dbeta", "beta"), ("dmu", "mu"),
                                  ("ds", "s"))):
        err = scalar_rel_err(t[key].grad.cpu().numpy(), ref[n], ref["absg"][w], ref["absp"][w])
        assert err.max() <= GRAD_RTOL, f"{n} (err {err.max():.3e})"
