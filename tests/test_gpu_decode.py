"""GPU decode parity: split-KV decode through the C ABI against the oracle."""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
from transformer_attention_ggd_gb300 import bam_attn as ba
from transformer_attention_ggd_gb300.inputs import make_inputs, random_params

from _gpu_helpers import LSE_ATOL, LSE_RTOL, O_ATOL, dev_bf16, f64, normal_bits, params_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    ba.load_library()


def _run(q, kc, vc, prm, ssmax, o_dtype=torch.float32):
    t = params_dev(prm)
    o, lse = ba.attention_decode(dev_bf16(q), dev_bf16(kc), dev_bf16(vc), t["alpha"], t["beta"],
                                 t["mu"], t["s"], ssmax=ssmax, o_dtype=o_dtype)
    torch.cuda.synchronize()
    return o.float().cpu().numpy(), lse.cpu().numpy()


@pytest.mark.parametrize("Tkv", [1, 2, 5, 63, 64, 65, 1000, 4097, 20000])
@pytest.mark.parametrize("ssmax", [True, False])
def test_small_ragged(Tkv, ssmax):
    rng = np.random.default_rng(Tkv + 11 * ssmax)
    B, H = 3, 4
    q = normal_bits(rng, (B, H, 64))
    kc = normal_bits(rng, (B, H, Tkv, 64))
    vc = normal_bits(rng, (B, H, Tkv, 64))
    prm = random_params(H, rng, mu_hi=10.0)
    prm["beta"][1] = -0.5
    o, lse = _run(q, kc, vc, prm, ssmax)
    oref, lref = oracle.decode(f64(q), f64(kc), f64(vc), prm["alpha"], prm["beta"], prm["mu"],
                               prm["s"], ssmax=ssmax)
    np.testing.assert_allclose(o, oref, rtol=0, atol=O_ATOL)
    np.testing.assert_allclose(lse, lref, rtol=LSE_RTOL, atol=LSE_ATOL)


def test_decode_matches_last_prefill_row_on_gpu():
    rng = np.random.default_rng(21)
    B, H, T = 2, 3, 777
    bits = {n: normal_bits(rng, (B, H, T, 64)) for n in "qkv"}
    prm = random_params(H, rng, mu_hi=5.0)
    t = params_dev(prm)
    q, k, v = (dev_bf16(bits[n]) for n in "qkv")
    o, lse = ba.attention_forward(q, k, v, t["alpha"], t["beta"], t["mu"], t["s"], causal=True,
                                  ssmax=True)
    od, lsed = ba.attention_decode(q[:, :, -1].contiguous(), k, v, t["alpha"], t["beta"],
                                   t["mu"], t["s"], ssmax=True)
    torch.cuda.synchronize()
    np.testing.assert_allclose(od.cpu().numpy(), o[:, :, -1].cpu().numpy(), rtol=0, atol=O_ATOL)
    np.testing.assert_allclose(lsed.cpu().numpy(), lse[:, :, -1].cpu().numpy(),
                               rtol=LSE_RTOL, atol=LSE_ATOL)


def test_config5_full():
    d = make_inputs(5)
    o, lse = _run(d["q"], d["k"], d["v"], d, True)
    oref, lref = oracle.decode(f64(d["q"]), f64(d["k"]), f64(d["v"]), d["alpha"], d["beta"],
                               d["mu"], d["s"], ssmax=True)
    np.testing.assert_allclose(o, oref, rtol=0, atol=O_ATOL)
    np.testing.assert_allclose(lse, lref, rtol=LSE_RTOL, atol=LSE_ATOL)
