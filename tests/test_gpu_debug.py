"""The bounds-checked debug build (libbam_attn_debug.so, BAM_DEBUG) on the
edge cases of every entry point.

compute-sanitizer is not available to these tests, so the library carries its
own checks: in the debug build every plain bulk copy (distance-table windows
of the forward and backward, K/V/table stages of the decode) is checked
against its own row, page or buffer and the 16-byte rule before it is
issued, and every tiled store's row coordinate against [0, T).  A failed
check skips the copy and reports BAM_ERR_BOUNDS; nothing traps.  The cases
here are shapes where off-by-one address arithmetic would show: one key, a
tile plus or minus one, ragged tails, the last row of the last head, cache
lengths on page boundaries.  Each call's status must be BAM_OK and its
results must match the oracle.

The debug library is a separate build of the same ABI, and the binding loads
one library per process, so `test_debug_build_edge_cases` builds it and runs
this module again in a child process with BAM_ATTN_DEBUG=1; the other tests
run only there.
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
from transformer_attention_ggd_gb300.inputs import random_params, random_theta_params

from _gpu_helpers import (GRAD_RTOL, LSE_ATOL, LSE_RTOL, O_ATOL, dev_bf16, f64, normal_bits,
                          params_dev, scalar_rel_err, tensor_rel_err)

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
IN_DEBUG = ba.DEBUG
debug_only = pytest.mark.skipif(not IN_DEBUG, reason="runs in the debug-library child process")


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")


@pytest.mark.skipif(IN_DEBUG, reason="this is the child process")
def test_debug_build_edge_cases():
    from transformer_attention_ggd_gb300 import build
    build.build(debug=True)
    env = dict(os.environ, BAM_ATTN_DEBUG="1")
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-m", "gpu", "-p",
                        "no:cacheprovider", os.path.abspath(__file__)],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=1200)
    tail = r.stdout[-6000:] + r.stderr[-3000:]
    assert r.returncode == 0, tail
    m = re.search(r"(\d+) passed", r.stdout)
    assert m and int(m.group(1)) >= 29, tail


def _status_ok(ws, what):
    st = ba.bam_attn_check_status(ws)
    assert st == ba.BAM_OK, f"{what}: status {st} ({ba.bam_status_string(st)})"


@debug_only
def test_loaded_library_is_the_debug_build():
    assert ba.bam_attn_debug_build()
    assert os.path.basename(ba.LIB_PATH) == "libbam_attn_debug.so"


# ---------------------------------------------------------------- forward + backward

@pytest.mark.parametrize("T", [1, 127, 128, 129, 255, 256, 257, 640])
@pytest.mark.parametrize("causal", [True, False])
@debug_only
def test_fwd_bwd(T, causal):
    rng = np.random.default_rng(900 + 3 * T + causal)
    B, H = 2, 3
    bits = {n: normal_bits(rng, (B, H, T, 64)) for n in ("q", "k", "v", "do")}
    prm = random_params(H, rng, mu_hi=6.0)
    prm["beta"][0] = -0.7
    _fwd_bwd(bits, prm, causal, ba.BAM_PRIOR_ALPHA)


@pytest.mark.parametrize("T,causal", [(129, True), (300, False)])
@debug_only
def test_fwd_bwd_theta(T, causal):
    rng = np.random.default_rng(950 + T)
    B, H = 1, 4
    bits = {n: normal_bits(rng, (B, H, T, 64)) for n in ("q", "k", "v", "do")}
    _fwd_bwd(bits, random_theta_params(H, rng), causal, ba.BAM_PRIOR_THETA)


def _fwd_bwd(bits, prm, causal, prior):
    B, H, T = bits["q"].shape[:3]
    q, k, v, g = (dev_bf16(bits[n]) for n in ("q", "k", "v", "do"))
    t = params_dev(prm)
    ws_f = ba.workspace(ba.BAM_OP_FWD, B, H, T)
    o, lse = ba.attention_forward(q, k, v, t["alpha"], t["beta"], t["mu"], t["s"],
                                  causal=causal, ssmax=True, o_dtype=torch.float32, ws=ws_f,
                                  prior=prior)
    _status_ok(ws_f, "forward")
    ws_b = ba.workspace(ba.BAM_OP_BWD, B, H, T)
    out = ba.attention_backward(q, k, v, o, lse, g, t["alpha"], t["beta"], t["mu"], t["s"],
                                causal=causal, ssmax=True, ws=ws_b, prior=prior)
    _status_ok(ws_b, "backward")
    oref, lref = oracle.fwd(f64(bits["q"]), f64(bits["k"]), f64(bits["v"]), prm["alpha"],
                            prm["beta"], prm["mu"], prm["s"], causal=causal, ssmax=True,
                            prior=prior)
    np.testing.assert_allclose(o.cpu().numpy(), oref, rtol=0, atol=O_ATOL)
    np.testing.assert_allclose(lse.cpu().numpy(), lref, rtol=LSE_RTOL, atol=LSE_ATOL)
    ref = oracle.bwd(f64(bits["q"]), f64(bits["k"]), f64(bits["v"]), f64(bits["do"]),
                     prm["alpha"], prm["beta"], prm["mu"], prm["s"], causal=causal, ssmax=True,
                     prior=prior)
    got = {n: x.float().cpu().numpy()
           for n, x in zip(("dq", "dk", "dv", "dalpha", "dbeta", "dmu", "ds"), out)}
    for n in ("dq", "dk", "dv"):
        rel = tensor_rel_err(got[n], ref[n])
        assert rel <= GRAD_RTOL, f"{n}: relative error {rel:.3e}"
    for w, n in enumerate(("dalpha", "dbeta", "dmu", "ds")):
        err = scalar_rel_err(got[n], ref[n], ref["absg"][w], ref["absp"][w])
        assert err.max() <= GRAD_RTOL, f"{n}: {got[n]} vs {ref[n]}"


# ---------------------------------------------------------------- decode

def _decode_ref(q, kc, vc, lens, prm):
    B, H = q.shape[:2]
    o = np.zeros((B, H, 64))
    lse = np.zeros((B, H))
    for b, n in enumerate(lens):
        ob, lb = oracle.decode(f64(q[b:b + 1]), f64(kc[b:b + 1, :, :n]), f64(vc[b:b + 1, :, :n]),
                               prm["alpha"], prm["beta"], prm["mu"], prm["s"], ssmax=True)
        o[b], lse[b] = ob[0], lb[0]
    return o, lse


def _check_decode(o, lse, q, kc, vc, lens, prm):
    oref, lref = _decode_ref(q, kc, vc, lens, prm)
    np.testing.assert_allclose(o.float().cpu().numpy(), oref, rtol=0, atol=O_ATOL)
    np.testing.assert_allclose(lse.cpu().numpy(), lref, rtol=LSE_RTOL, atol=LSE_ATOL)


@pytest.mark.parametrize("Tkv", [1, 63, 64, 65, 257, 1000, 4097])
@debug_only
def test_decode(Tkv):
    rng = np.random.default_rng(970 + Tkv)
    B, H = 3, 2
    q = normal_bits(rng, (B, H, 64))
    kc, vc = normal_bits(rng, (B, H, Tkv, 64)), normal_bits(rng, (B, H, Tkv, 64))
    prm = random_params(H, rng, mu_hi=8.0)
    t = params_dev(prm)
    ws = ba.workspace(ba.BAM_OP_DECODE, B, H, Tkv)
    o, lse = ba.attention_decode(dev_bf16(q), dev_bf16(kc), dev_bf16(vc), t["alpha"], t["beta"],
                                 t["mu"], t["s"], ssmax=True, o_dtype=torch.float32, ws=ws)
    _status_ok(ws, "decode")
    _check_decode(o, lse, q, kc, vc, [Tkv] * B, prm)


@debug_only
def test_decode_varlen():
    rng = np.random.default_rng(990)
    B, H, Tmax = 6, 2, 1000
    lens = [1, 3, 64, 65, 999, 1000]
    q = normal_bits(rng, (B, H, 64))
    kc, vc = normal_bits(rng, (B, H, Tmax, 64)), normal_bits(rng, (B, H, Tmax, 64))
    prm = random_params(H, rng, mu_hi=8.0)
    t = params_dev(prm)
    ws = ba.workspace(ba.BAM_OP_DECODE, B, H, Tmax)
    o, lse = ba.attention_decode_varlen(
        dev_bf16(q), dev_bf16(kc), dev_bf16(vc), torch.tensor(lens, dtype=torch.int32,
                                                               device="cuda"),
        t["alpha"], t["beta"], t["mu"], t["s"], ssmax=True, o_dtype=torch.float32, ws=ws)
    _status_ok(ws, "varlen decode")
    _check_decode(o, lse, q, kc, vc, lens, prm)


@pytest.mark.parametrize("page", [64, 128])
@debug_only
def test_decode_paged(page):
    """Permuted pages; lengths of one key, a page minus or plus one, and the
    whole table; the last page of the pool is in use."""
    rng = np.random.default_rng(995 + page)
    B, H, max_blocks = 5, 2, 4
    Tmax = page * max_blocks
    lens = [1, page - 1, page + 1, 2 * page, Tmax]
    q = normal_bits(rng, (B, H, 64))
    kc, vc = normal_bits(rng, (B, H, Tmax, 64)), normal_bits(rng, (B, H, Tmax, 64))
    prm = random_params(H, rng, mu_hi=8.0)
    used = [(b, i) for b in range(B) for i in range((lens[b] + page - 1) // page)]
    num_pages = len(used)
    perm = rng.permutation(num_pages)
    kp = np.zeros((num_pages, H, page, 64), np.uint16)
    vp = np.zeros_like(kp)
    table = np.full((B, max_blocks), -1, np.int32)
    for (b, i), pg in zip(used, perm):
        table[b, i] = pg
        kp[pg] = kc[b, :, i * page:(i + 1) * page]
        vp[pg] = vc[b, :, i * page:(i + 1) * page]
    t = params_dev(prm)
    ws = ba.workspace(ba.BAM_OP_DECODE, B, H, Tmax)
    o, lse = ba.attention_decode_paged(
        dev_bf16(q), dev_bf16(kp), dev_bf16(vp), torch.from_numpy(table).cuda(),
        torch.tensor(lens, dtype=torch.int32, device="cuda"), t["alpha"], t["beta"], t["mu"],
        t["s"], ssmax=True, o_dtype=torch.float32, ws=ws)
    _status_ok(ws, "paged decode")
    _check_decode(o, lse, q, kc, vc, lens, prm)
