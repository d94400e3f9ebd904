"""The real kernels' give-up paths, driven without a fault or a hang.

Every device wait of the library is bounded; when one gives up, the kernel
records BAM_ERR_TIMEOUT, drains the copies and tensor-core work it has in
flight, frees its Tensor Memory and returns, and the rest of the call
follows the abort.  In the debug build (BAM_DEBUG) a test can arm a give-up
count on a workspace (bam_attn_debug_arm_giveup): the n-th bounded wait of
the next call gives up as if its time limit had passed.  For the forward,
the backward, the decode and the no-alloc decode, and for several n (so the
give-up lands at different points of the pipelines), the call must report
BAM_ERR_TIMEOUT, the context must stay usable, and the next normal call on
the same workspace must match the oracle.  The decode forms must also mark
their outputs invalid (NaN) on a give-up.  A recorded error must survive a
later call until it is read.

As in test_gpu_debug, the debug library is a separate build and the binding
loads one library per process, so `test_giveup_paths_in_debug_build` runs
this module again in a child process with BAM_ATTN_DEBUG=1.
"""

import os
import re
import subprocess
import sys

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
from transformer_attention_ggd_gb300 import bam_attn as ba
from transformer_attention_ggd_gb300.inputs import random_params

from _gpu_helpers import (GRAD_RTOL, LSE_ATOL, LSE_RTOL, O_ATOL, dev_bf16, f64, normal_bits,
                          params_dev, tensor_rel_err)

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
IN_DEBUG = ba.DEBUG
debug_only = pytest.mark.skipif(not IN_DEBUG, reason="runs in the debug-library child process")
GIVEUP_AT = [1, 9, 120, 1500]


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")


@pytest.mark.skipif(IN_DEBUG, reason="this is the child process")
def test_giveup_paths_in_debug_build():
    from transformer_attention_ggd_gb300 import build
    build.build(debug=True)
    env = dict(os.environ, BAM_ATTN_DEBUG="1")
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-m", "gpu", "-p",
                        "no:cacheprovider", os.path.abspath(__file__)],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=1200)
    tail = r.stdout[-6000:] + r.stderr[-3000:]
    assert r.returncode == 0, tail
    m = re.search(r"(\d+) passed", r.stdout)
    assert m and int(m.group(1)) >= 6 * len(GIVEUP_AT) + 2, tail


@pytest.mark.skipif(IN_DEBUG, reason="the release build")
def test_release_build_refuses_the_giveup_knob():
    ws = ba.workspace(ba.BAM_OP_FWD, 1, 1, 16)
    assert ba.bam_attn_debug_arm_giveup(ws, 3) == ba.BAM_ERR_UNSUPPORTED
    assert ba.bam_attn_debug_arm_giveup_noalloc(3) == ba.BAM_ERR_UNSUPPORTED


def _fwd_case(seed, B=1, H=2, T=300):
    rng = np.random.default_rng(seed)
    bits = {n: normal_bits(rng, (B, H, T, 64)) for n in "qkvg"}
    prm = random_params(H, rng, mu_hi=4.0)
    prm["beta"][0] = -0.5
    return bits, prm


def _fwd(bits, prm, ws, o, lse):
    t = params_dev(prm)
    p = ba.make_params(t["alpha"], t["beta"], t["mu"], t["s"], 1e-5, True, True)
    ba.bam_attn_fwd(*(dev_bf16(bits[n]) for n in "qkv"), o, lse, p, ws)
    torch.cuda.synchronize()


@debug_only
@pytest.mark.parametrize("n", GIVEUP_AT)
def test_forward_gives_up_then_recovers(n):
    B, H, T = 1, 2, 300
    bits, prm = _fwd_case(100 + n, B, H, T)
    ws = ba.workspace(ba.BAM_OP_FWD, B, H, T)
    o = torch.empty((B, H, T, 64), dtype=torch.float32, device="cuda")
    lse = torch.empty((B, H, T), dtype=torch.float32, device="cuda")
    assert ba.bam_attn_debug_arm_giveup(ws, n) == ba.BAM_OK
    _fwd(bits, prm, ws, o, lse)
    assert ba.bam_attn_check_status(ws) == ba.BAM_ERR_TIMEOUT
    _fwd(bits, prm, ws, o, lse)
    assert ba.bam_attn_check_status(ws) == ba.BAM_OK
    oref, lref = oracle.fwd(f64(bits["q"]), f64(bits["k"]), f64(bits["v"]), prm["alpha"],
                            prm["beta"], prm["mu"], prm["s"], causal=True, ssmax=True)
    np.testing.assert_allclose(o.cpu().numpy(), oref, rtol=0, atol=O_ATOL)
    np.testing.assert_allclose(lse.cpu().numpy(), lref, rtol=LSE_RTOL, atol=LSE_ATOL)


@debug_only
@pytest.mark.parametrize("n", GIVEUP_AT)
def test_paired_forward_gives_up_then_recovers(n):
    # 4 x 76 heads of 256 rows: 304 paired CTAs (two waves of 152 SMs), so the
    # long-sequence kernel runs rather than the single-tile one.
    B, H, T = 4, 76, 256
    bits, prm = _fwd_case(600 + n, B, H, T)
    ws = ba.workspace(ba.BAM_OP_FWD, B, H, T)
    o = torch.empty((B, H, T, 64), dtype=torch.float32, device="cuda")
    lse = torch.empty((B, H, T), dtype=torch.float32, device="cuda")
    assert ba.bam_attn_debug_arm_giveup(ws, n) == ba.BAM_OK
    _fwd(bits, prm, ws, o, lse)
    assert ba.bam_attn_check_status(ws) == ba.BAM_ERR_TIMEOUT
    _fwd(bits, prm, ws, o, lse)
    assert ba.bam_attn_check_status(ws) == ba.BAM_OK
    # The oracle on the first batch row (76 heads).
    oref, lref = oracle.fwd(f64(bits["q"][:1]), f64(bits["k"][:1]), f64(bits["v"][:1]),
                            prm["alpha"], prm["beta"], prm["mu"], prm["s"], causal=True,
                            ssmax=True)
    np.testing.assert_allclose(o[:1].cpu().numpy(), oref, rtol=0, atol=O_ATOL)
    np.testing.assert_allclose(lse[:1].cpu().numpy(), lref, rtol=LSE_RTOL, atol=LSE_ATOL)


@debug_only
@pytest.mark.parametrize("n", GIVEUP_AT)
def test_scheduled_backward_gives_up_then_recovers(n):
    # The training shape, whose work items run in host-packed per-CTA lists.
    B, H, T = 8, 12, 512
    assert ba.bam_attn_bwd_schedule(B, H, T, True, 152) is not None
    bits, prm = _fwd_case(700 + n, B, H, T)
    t = params_dev(prm)
    q, k, v, g = (dev_bf16(bits[c]) for c in "qkvg")
    o, lse = ba.attention_forward(q, k, v, t["alpha"], t["beta"], t["mu"], t["s"], causal=True,
                                  ssmax=True)
    p = ba.make_params(t["alpha"], t["beta"], t["mu"], t["s"], 1e-5, True, True)
    ws = ba.workspace(ba.BAM_OP_BWD, B, H, T)
    dq, dk, dv = (torch.empty_like(q) for _ in range(3))
    gr = [torch.empty(H, dtype=torch.float32, device="cuda") for _ in range(4)]
    assert ba.bam_attn_debug_arm_giveup(ws, n) == ba.BAM_OK
    ba.bam_attn_bwd(q, k, v, o, lse, g, dq, dk, dv, *gr, p, ws)
    torch.cuda.synchronize()
    assert ba.bam_attn_check_status(ws) == ba.BAM_ERR_TIMEOUT
    ba.bam_attn_bwd(q, k, v, o, lse, g, dq, dk, dv, *gr, p, ws)
    torch.cuda.synchronize()
    assert ba.bam_attn_check_status(ws) == ba.BAM_OK
    # The oracle on the first batch row (its dq, dk, dv do not depend on the
    # other rows).
    ref = oracle.bwd(f64(bits["q"][:1]), f64(bits["k"][:1]), f64(bits["v"][:1]),
                     f64(bits["g"][:1]), prm["alpha"], prm["beta"], prm["mu"], prm["s"],
                     causal=True, ssmax=True)
    for name, got in (("dq", dq), ("dk", dk), ("dv", dv)):
        assert tensor_rel_err(got[:1].float().cpu().numpy(), ref[name]) < GRAD_RTOL, name


@debug_only
@pytest.mark.parametrize("n", GIVEUP_AT)
def test_backward_gives_up_then_recovers(n):
    B, H, T = 1, 2, 300
    bits, prm = _fwd_case(200 + n, B, H, T)
    t = params_dev(prm)
    q, k, v, g = (dev_bf16(bits[c]) for c in "qkvg")
    o, lse = ba.attention_forward(q, k, v, t["alpha"], t["beta"], t["mu"], t["s"], causal=True,
                                  ssmax=True)
    p = ba.make_params(t["alpha"], t["beta"], t["mu"], t["s"], 1e-5, True, True)
    ws = ba.workspace(ba.BAM_OP_BWD, B, H, T)
    dq, dk, dv = (torch.empty_like(q) for _ in range(3))
    gr = [torch.empty(H, dtype=torch.float32, device="cuda") for _ in range(4)]
    assert ba.bam_attn_debug_arm_giveup(ws, n) == ba.BAM_OK
    ba.bam_attn_bwd(q, k, v, o, lse, g, dq, dk, dv, *gr, p, ws)
    torch.cuda.synchronize()
    assert ba.bam_attn_check_status(ws) == ba.BAM_ERR_TIMEOUT
    ba.bam_attn_bwd(q, k, v, o, lse, g, dq, dk, dv, *gr, p, ws)
    torch.cuda.synchronize()
    assert ba.bam_attn_check_status(ws) == ba.BAM_OK
    ref = oracle.bwd(f64(bits["q"]), f64(bits["k"]), f64(bits["v"]), f64(bits["g"]),
                     prm["alpha"], prm["beta"], prm["mu"], prm["s"], causal=True, ssmax=True)
    for name, got in (("dq", dq), ("dk", dk), ("dv", dv)):
        assert tensor_rel_err(got.float().cpu().numpy(), ref[name]) < GRAD_RTOL, name


def _decode_case(seed, B=4, H=3, Tkv=3000):
    rng = np.random.default_rng(seed)
    q = dev_bf16(normal_bits(rng, (B, H, 64)))
    kc = dev_bf16(normal_bits(rng, (B, H, Tkv, 64)))
    vc = dev_bf16(normal_bits(rng, (B, H, Tkv, 64)))
    prm = random_params(H, rng, mu_hi=4.0)
    return q, kc, vc, prm


def _decode_ref(q, kc, vc, prm):
    def back(x):
        return f64(x.view(torch.int16).cpu().numpy().view(np.uint16))
    return oracle.decode(back(q), back(kc), back(vc), prm["alpha"], prm["beta"], prm["mu"],
                         prm["s"], ssmax=True)


@debug_only
@pytest.mark.parametrize("n", GIVEUP_AT)
def test_decode_gives_up_marks_outputs_then_recovers(n):
    q, kc, vc, prm = _decode_case(300 + n)
    B, H, Tkv = kc.shape[:3]
    t = params_dev(prm)
    p = ba.make_params(t["alpha"], t["beta"], t["mu"], t["s"], 1e-5, True, True)
    ws = ba.workspace(ba.BAM_OP_DECODE, B, H, Tkv)
    o = torch.zeros((B, H, 64), dtype=torch.float32, device="cuda")
    lse = torch.zeros((B, H), dtype=torch.float32, device="cuda")
    assert ba.bam_attn_debug_arm_giveup(ws, n) == ba.BAM_OK
    ba.bam_attn_decode(q, kc, vc, o, lse, p, ws)
    torch.cuda.synchronize()
    assert ba.bam_attn_check_status(ws) == ba.BAM_ERR_TIMEOUT
    assert torch.isnan(o).all() and torch.isnan(lse).all()
    ba.bam_attn_decode(q, kc, vc, o, lse, p, ws)
    torch.cuda.synchronize()
    assert ba.bam_attn_check_status(ws) == ba.BAM_OK
    oref, lref = _decode_ref(q, kc, vc, prm)
    np.testing.assert_allclose(o.cpu().numpy(), oref, rtol=0, atol=O_ATOL)
    np.testing.assert_allclose(lse.cpu().numpy(), lref, rtol=LSE_RTOL, atol=LSE_ATOL)


@debug_only
@pytest.mark.parametrize("n", GIVEUP_AT)
def test_noalloc_decode_reports_its_giveup_then_recovers(n):
    q, kc, vc, prm = _decode_case(400 + n)
    B, H = kc.shape[:2]
    t = params_dev(prm)
    p = ba.make_params(t["alpha"], t["beta"], t["mu"], t["s"], 1e-5, True, True)
    o = torch.zeros((B, H, 64), dtype=torch.float32, device="cuda")
    lse = torch.zeros((B, H), dtype=torch.float32, device="cuda")
    ba.bam_attn_decode_noalloc(q, kc, vc, o, lse, p)  # first call: the scratch set-up
    assert ba.bam_attn_decode_noalloc_check_status() == ba.BAM_OK
    assert ba.bam_attn_debug_arm_giveup_noalloc(n) == ba.BAM_OK
    ba.bam_attn_decode_noalloc(q, kc, vc, o, lse, p)
    assert ba.bam_attn_decode_noalloc_check_status() == ba.BAM_ERR_TIMEOUT
    assert torch.isnan(o).all() and torch.isnan(lse).all()
    ba.bam_attn_decode_noalloc(q, kc, vc, o, lse, p)
    assert ba.bam_attn_decode_noalloc_check_status() == ba.BAM_OK
    oref, lref = _decode_ref(q, kc, vc, prm)
    np.testing.assert_allclose(o.cpu().numpy(), oref, rtol=0, atol=O_ATOL)
    np.testing.assert_allclose(lse.cpu().numpy(), lref, rtol=LSE_RTOL, atol=LSE_ATOL)


@debug_only
def test_unread_giveup_survives_a_later_call():
    B, H, T = 1, 2, 300
    bits, prm = _fwd_case(500, B, H, T)
    ws = ba.workspace(ba.BAM_OP_FWD, B, H, T)
    o = torch.empty((B, H, T, 64), dtype=torch.float32, device="cuda")
    lse = torch.empty((B, H, T), dtype=torch.float32, device="cuda")
    assert ba.bam_attn_debug_arm_giveup(ws, 5) == ba.BAM_OK
    _fwd(bits, prm, ws, o, lse)  # gives up
    _fwd(bits, prm, ws, o, lse)  # runs normally, leaves the first error in place
    oref, _ = oracle.fwd(f64(bits["q"]), f64(bits["k"]), f64(bits["v"]), prm["alpha"],
                         prm["beta"], prm["mu"], prm["s"], causal=True, ssmax=True)
    np.testing.assert_allclose(o.cpu().numpy(), oref, rtol=0, atol=O_ATOL)
    assert ba.bam_attn_check_status(ws) == ba.BAM_ERR_TIMEOUT
    assert ba.bam_attn_check_status(ws) == ba.BAM_OK


@debug_only
def test_disarmed_knob_leaves_calls_alone():
    B, H, T = 1, 2, 300
    bits, prm = _fwd_case(600, B, H, T)
    ws = ba.workspace(ba.BAM_OP_FWD, B, H, T)
    o = torch.empty((B, H, T, 64), dtype=torch.float32, device="cuda")
    lse = torch.empty((B, H, T), dtype=torch.float32, device="cuda")
    assert ba.bam_attn_debug_arm_giveup(ws, 0) == ba.BAM_OK
    _fwd(bits, prm, ws, o, lse)
    assert ba.bam_attn_check_status(ws) == ba.BAM_OK
