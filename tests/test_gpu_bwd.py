"""GPU backward parity: dq, dk, dv and the per-head scalar gradients through
the C ABI against the fp64 oracle's chain-rule backward."""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
from transformer_attention_ggd_gb300 import bam_attn as ba
from transformer_attention_ggd_gb300.inputs import make_inputs, random_params

from _gpu_helpers import (GRAD_RTOL, dev_bf16, f64, normal_bits, params_dev, scalar_rel_err,
                          tensor_rel_err)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    ba.load_library()


def _gpu(bits, prm, causal, ssmax, o_dtype=torch.float32):
    q, k, v, g = (dev_bf16(bits[n]) for n in ("q", "k", "v", "do"))
    t = params_dev(prm)
    o, lse = ba.attention_forward(q, k, v, t["alpha"], t["beta"], t["mu"], t["s"],
                                  causal=causal, ssmax=ssmax, o_dtype=o_dtype)
    out = ba.attention_backward(q, k, v, o, lse, g, t["alpha"], t["beta"], t["mu"], t["s"],
                                causal=causal, ssmax=ssmax)
    torch.cuda.synchronize()
    names = ("dq", "dk", "dv", "dalpha", "dbeta", "dmu", "ds")
    return {n: x.float().cpu().numpy() for n, x in zip(names, out)}


def _ref(bits, prm, causal, ssmax):
    return oracle.bwd(f64(bits["q"]), f64(bits["k"]), f64(bits["v"]), f64(bits["do"]),
                      prm["alpha"], prm["beta"], prm["mu"], prm["s"], causal=causal,
                      ssmax=ssmax)


def _compare(got, ref, ssmax):
    for n in ("dq", "dk", "dv"):
        rel = tensor_rel_err(got[n], ref[n])
        assert rel <= GRAD_RTOL, f"{n}: relative error {rel:.3e}"
    for w, n in enumerate(("dalpha", "dbeta", "dmu", "ds")):
        if n == "ds" and not ssmax:
            assert np.all(got[n] == 0.0)
            continue
        err = scalar_rel_err(got[n], ref[n], ref["absg"][w], ref["absp"][w])
        assert err.max() <= GRAD_RTOL, f"{n}: {got[n]} vs {ref[n]} (err {err.max():.3e})"


@pytest.mark.parametrize("T", [1, 2, 17, 128, 129, 300])
@pytest.mark.parametrize("causal,ssmax", [(True, True), (True, False), (False, True)])
def test_small_ragged(T, causal, ssmax):
    rng = np.random.default_rng(100 + T * 5 + causal * 2 + ssmax)
    B, H = 2, 3
    bits = {n: normal_bits(rng, (B, H, T, 64)) for n in ("q", "k", "v", "do")}
    prm = random_params(H, rng, mu_hi=4.0)
    prm["beta"][0] = -0.6
    prm["mu"][1] = 2.5
    got = _gpu(bits, prm, causal, ssmax)
    ref = _ref(bits, prm, causal, ssmax)
    _compare(got, ref, ssmax)


def test_bf16_forward_output_as_input():
    rng = np.random.default_rng(8)
    B, H, T = 1, 4, 257
    bits = {n: normal_bits(rng, (B, H, T, 64)) for n in ("q", "k", "v", "do")}
    prm = random_params(H, rng, mu_hi=3.0)
    got = _gpu(bits, prm, True, True, o_dtype=torch.bfloat16)
    _compare(got, _ref(bits, prm, True, True), True)


def test_config2_training_step_full():
    d = make_inputs(2)
    bits = {n: d[n] for n in ("q", "k", "v", "do")}
    got = _gpu(bits, d, True, True)
    ref = _ref(bits, d, True, True)
    _compare(got, ref, True)


def test_training_shape_noncausal_full():
    """The training workload's shape without the causal mask: 384 items of
    four query tiles each, dealt over the CTAs round-robin (several rounds),
    every output against the oracle."""
    d = make_inputs(2)
    bits = {n: d[n] for n in ("q", "k", "v", "do")}
    got = _gpu(bits, d, False, True)
    _compare(got, _ref(bits, d, False, True), True)


@pytest.mark.parametrize("B,H,T", [(16, 16, 512), (7, 11, 520)])
def test_packed_schedules_full(B, H, T):
    """Shapes whose work items run in host-packed per-CTA lists (1024 items,
    the largest the kernel parameter holds, and a ragged T with few heads):
    every output against the oracle."""
    assert ba.bam_attn_bwd_schedule(B, H, T, True, 152) is not None
    rng = np.random.default_rng(B * 1000 + T)
    bits = {n: normal_bits(rng, (B, H, T, 64)) for n in ("q", "k", "v", "do")}
    prm = random_params(H, rng, mu_hi=4.0)
    prm["beta"][0] = -0.6
    got = _gpu(bits, prm, True, True)
    _compare(got, _ref(bits, prm, True, True), True)


def test_dk_dv_deterministic():
    rng = np.random.default_rng(4)
    bits = {n: normal_bits(rng, (1, 2, 400, 64)) for n in ("q", "k", "v", "do")}
    prm = random_params(2, rng)
    a = _gpu(bits, prm, True, True)
    b = _gpu(bits, prm, True, True)
    np.testing.assert_array_equal(a["dk"], b["dk"])
    np.testing.assert_array_equal(a["dv"], b["dv"])
    # dq and the scalar sums are accumulated with atomics: order may differ.
    np.testing.assert_allclose(a["dq"], b["dq"], rtol=1e-2, atol=1e-3)


@pytest.mark.parametrize("ssmax", [True, False])
def test_scalar_outputs_overwritten_not_accumulated(ssmax):
    """dalpha, dbeta, dmu and ds are summed into by the kernels after the
    call's first kernel zeroes them: outputs pre-filled with NaN come out
    right, and a second call into the same outputs (same workspace) gives the
    same values instead of twice them."""
    rng = np.random.default_rng(31 + ssmax)
    B, H, T = 2, 3, 300
    bits = {n: normal_bits(rng, (B, H, T, 64)) for n in ("q", "k", "v", "do")}
    prm = random_params(H, rng, mu_hi=3.0)
    q, k, v, g = (dev_bf16(bits[n]) for n in ("q", "k", "v", "do"))
    t = params_dev(prm)
    o, lse = ba.attention_forward(q, k, v, t["alpha"], t["beta"], t["mu"], t["s"],
                                  causal=True, ssmax=ssmax)
    dq, dk, dv = (torch.empty_like(q) for _ in range(3))
    outs = [torch.full((H,), float("nan"), dtype=torch.float32, device=q.device)
            for _ in range(4)]
    ws = ba.workspace(ba.BAM_OP_BWD, B, H, T, q.device)
    p = ba.make_params(t["alpha"], t["beta"], t["mu"], t["s"], 1e-5, True, ssmax,
                       ba.BAM_PRIOR_ALPHA)
    ref = _ref(bits, prm, True, ssmax)
    got = []
    for _ in range(2):
        ba.bam_attn_bwd(q, k, v, o, lse, g, dq, dk, dv, *outs, p, ws)
        torch.cuda.synchronize()
        got.append([x.cpu().numpy().copy() for x in outs])
        res = {n: x.float().cpu().numpy() for n, x in zip(("dq", "dk", "dv"), (dq, dk, dv))}
        res.update(zip(("dalpha", "dbeta", "dmu", "ds"), got[-1]))
        _compare(res, ref, ssmax)
    for a, b in zip(*got):
        np.testing.assert_allclose(a, b, rtol=1e-4, atol=1e-6)


@pytest.mark.parametrize("causal", [True, False])
def test_long_sequence_full(causal):
    """T = 2048 (16 key tiles, so each dQ tile is summed from up to 16
    items): every output against the oracle, causal and not."""
    rng = np.random.default_rng(2048 + causal)
    B, H, T = 1, 2, 2048
    bits = {n: normal_bits(rng, (B, H, T, 64)) for n in ("q", "k", "v", "do")}
    prm = random_params(H, rng, mu_hi=16.0)
    prm["beta"][0] = -0.4
    got = _gpu(bits, prm, causal, True)
    _compare(got, _ref(bits, prm, causal, True), True)
