"""Failure detection on the GPU without a fault: a bounded wait that runs out
(a barrier nothing arrives at) records BAM_ERR_TIMEOUT in the workspace
status word, the kernel returns, the host reads and clears the status, and
the context stays usable for the next call."""

import time

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
from transformer_attention_ggd_gb300 import bam_attn as ba
from transformer_attention_ggd_gb300.inputs import random_params

from _gpu_helpers import O_ATOL, dev_bf16, f64, normal_bits, params_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    ba.load_library()


def test_bounded_wait_gives_up_and_the_context_stays_usable():
    B, H, T = 1, 2, 200
    ws = ba.workspace(ba.BAM_OP_FWD, B, H, T)
    assert ba.bam_attn_check_status(ws) == ba.BAM_OK
    t0 = time.monotonic()
    ba.bam_attn_selftest_wait(ws)
    torch.cuda.synchronize()
    waited = time.monotonic() - t0
    # status word: abort, code, site, block (int32 each)
    words = ws[:16].cpu().numpy().view(np.int32)
    assert words[0] == 1 and words[1] == 1 and words[2] == 90 and words[3] == 0, words
    assert 1.0 < waited < 60.0, waited
    assert ba.bam_attn_check_status(ws) == ba.BAM_ERR_TIMEOUT
    assert ba.bam_attn_check_status(ws) == ba.BAM_OK  # read and cleared
    # the same context and workspace serve a normal call afterwards
    rng = np.random.default_rng(9)
    bits = {n: normal_bits(rng, (B, H, T, 64)) for n in "qkv"}
    prm = random_params(H, rng, mu_hi=2.0)
    t = params_dev(prm)
    o, lse = ba.attention_forward(*(dev_bf16(bits[n]) for n in "qkv"), t["alpha"], t["beta"],
                                  t["mu"], t["s"], causal=True, ssmax=True, ws=ws)
    assert ba.bam_attn_check_status(ws) == ba.BAM_OK
    oref, _ = oracle.fwd(f64(bits["q"]), f64(bits["k"]), f64(bits["v"]), prm["alpha"],
                         prm["beta"], prm["mu"], prm["s"], causal=True, ssmax=True)
    np.testing.assert_allclose(o.cpu().numpy(), oref, rtol=0, atol=O_ATOL)


def test_unread_error_survives_the_next_call():
    """A call that gives up leaves its error in the workspace status; a later
    call on the same workspace runs normally and neither erases nor
    overwrites it: bam_attn_check_status reports the first error since the
    previous check, then the status is clear."""
    B, H, T = 1, 2, 200
    ws = ba.workspace(ba.BAM_OP_FWD, B, H, T)
    ba.bam_attn_selftest_wait(ws)
    rng = np.random.default_rng(10)
    bits = {n: normal_bits(rng, (B, H, T, 64)) for n in "qkv"}
    prm = random_params(H, rng, mu_hi=2.0)
    t = params_dev(prm)
    o, _ = ba.attention_forward(*(dev_bf16(bits[n]) for n in "qkv"), t["alpha"], t["beta"],
                                t["mu"], t["s"], causal=True, ssmax=True, ws=ws)
    torch.cuda.synchronize()
    words = ws[:16].cpu().numpy().view(np.int32)
    assert words[0] == 0 and words[1] == 1 and words[2] == 90, words  # abort cleared, code kept
    assert ba.bam_attn_check_status(ws) == ba.BAM_ERR_TIMEOUT
    assert ba.bam_attn_check_status(ws) == ba.BAM_OK
    oref, _ = oracle.fwd(f64(bits["q"]), f64(bits["k"]), f64(bits["v"]), prm["alpha"],
                         prm["beta"], prm["mu"], prm["s"], causal=True, ssmax=True)
    np.testing.assert_allclose(o.cpu().numpy(), oref, rtol=0, atol=O_ATOL)


def test_noalloc_status_reads_clean_after_a_normal_call():
    B, H, Tkv = 2, 3, 1000
    rng = np.random.default_rng(11)
    q = dev_bf16(normal_bits(rng, (B, H, 64)))
    kc = dev_bf16(normal_bits(rng, (B, H, Tkv, 64)))
    vc = dev_bf16(normal_bits(rng, (B, H, Tkv, 64)))
    t = params_dev(random_params(H, rng, mu_hi=2.0))
    p = ba.make_params(t["alpha"], t["beta"], t["mu"], t["s"], 1e-5, True, True)
    o = torch.empty((B, H, 64), dtype=torch.float32, device="cuda")
    ba.bam_attn_decode_noalloc(q, kc, vc, o, None, p)
    assert ba.bam_attn_decode_noalloc_check_status() == ba.BAM_OK
    assert torch.isfinite(o).all()
