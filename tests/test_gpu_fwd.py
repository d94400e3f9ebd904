"""GPU forward parity: the CUDA path through the C ABI against the fp64 oracle.

Small ragged shapes and the configurations of the method's workloads, with
full comparison where the oracle finishes in seconds and sampled rows (the
oracle computes them one by one) at the long-context sizes.
"""

import math

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
from transformer_attention_ggd_gb300 import bam_attn as ba
from transformer_attention_ggd_gb300.inputs import make_inputs, random_params, workload

from _gpu_helpers import (LSE_ATOL, LSE_RTOL, O_ATOL, dev_bf16, dev_f32, f64, normal_bits, params_dev)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    ba.load_library()


def _run(bits, prm, causal, ssmax, o_dtype=torch.float32):
    q, k, v = (dev_bf16(bits[n]) for n in "qkv")
    t = params_dev(prm)
    o, lse = ba.attention_forward(q, k, v, t["alpha"], t["beta"], t["mu"], t["s"],
                                  causal=causal, ssmax=ssmax, o_dtype=o_dtype)
    torch.cuda.synchronize()
    return o.float().cpu().numpy(), lse.cpu().numpy()


def _oracle(bits, prm, causal, ssmax):
    return oracle.fwd(f64(bits["q"]), f64(bits["k"]), f64(bits["v"]), prm["alpha"], prm["beta"],
                      prm["mu"], prm["s"], causal=causal, ssmax=ssmax)


@pytest.mark.parametrize("T", [1, 2, 3, 17, 128, 129, 255, 256, 300, 513])
@pytest.mark.parametrize("causal,ssmax", [(True, True), (True, False), (False, True)])
def test_small_ragged(T, causal, ssmax):
    rng = np.random.default_rng(T * 7 + causal * 3 + ssmax)
    B, H = 2, 3
    bits = {n: normal_bits(rng, (B, H, T, 64)) for n in "qkv"}
    prm = random_params(H, rng, mu_hi=6.0)
    prm["beta"][0] = -0.7  # an inverted-prior head
    o, lse = _run(bits, prm, causal, ssmax)
    oref, lref = _oracle(bits, prm, causal, ssmax)
    np.testing.assert_allclose(o, oref, rtol=0, atol=O_ATOL)
    np.testing.assert_allclose(lse, lref, rtol=LSE_RTOL, atol=LSE_ATOL)


@pytest.mark.parametrize("T", [129, 300, 513, 2048])
@pytest.mark.parametrize("causal", [True, False])
def test_paired_and_single_tile_schedules(T, causal):
    """The forward runs 256-row CTAs (two query tiles sharing each K/V tile)
    when they fill at least two waves of the SMs, else single-tile CTAs (128
    rows, two per SM).  One (b, h) pair of heads runs the single-tile kernel;
    the same heads repeated over 160 batch rows run paired; both match the
    oracle, every repeat alike."""
    rng = np.random.default_rng(T + 11 * causal)
    H = 2
    bits = {n: normal_bits(rng, (1, H, T, 64)) for n in "qkv"}
    prm = random_params(H, rng, mu_hi=6.0)
    prm["beta"][0] = -0.6
    oref, lref = _oracle(bits, prm, causal, True)
    o1, l1 = _run(bits, prm, causal, True)
    np.testing.assert_allclose(o1, oref, rtol=0, atol=O_ATOL)
    np.testing.assert_allclose(l1, lref, rtol=LSE_RTOL, atol=LSE_ATOL)
    rep = {n: np.ascontiguousarray(np.repeat(b, 160, axis=0)) for n, b in bits.items()}
    o2, l2 = _run(rep, prm, causal, True)
    np.testing.assert_allclose(o2, np.repeat(oref, 160, axis=0), rtol=0, atol=O_ATOL)
    np.testing.assert_allclose(l2, np.repeat(lref, 160, axis=0), rtol=LSE_RTOL, atol=LSE_ATOL)
    assert (o2 == o2[:1]).all() and (l2 == l2[:1]).all()


def test_worked_example_on_gpu():
    """Non-causal T=2, four heads, zero content, values 0 and 1 in column 0:
    head 0 gives 0.4378235, 0.5621765 (the ALiBi-style exercise's printed
    numbers); every head's position 0 gives 1/(1+exp(slope))."""
    H, T = 4, 2
    slopes = np.array([2.0 ** (-8.0 * (h + 1) / H) for h in range(H)])
    zeros = np.zeros((1, H, T, 64), np.uint16)
    vbits = np.zeros((1, H, T, 64), np.uint16)
    vbits[..., 1, 0] = 0x3F80  # 1.0 in bf16
    prm = {"alpha": (1 / slopes).astype(np.float32), "beta": np.ones(H, np.float32),
           "mu": np.zeros(H, np.float32), "s": np.ones(H, np.float32)}
    o, _ = _run({"q": zeros, "k": zeros, "v": vbits}, prm, causal=False, ssmax=False)
    np.testing.assert_allclose(o[0, 0, :, 0], [0.4378235, 0.5621765], rtol=0, atol=O_ATOL)
    np.testing.assert_allclose(o[0, :, 0, 0], 1 / (1 + np.exp(slopes)), rtol=0, atol=O_ATOL)


def test_alibi_and_nope_special_cases_on_gpu():
    rng = np.random.default_rng(5)
    B, H, T = 1, 8, 333
    bits = {n: normal_bits(rng, (B, H, T, 64)) for n in "qkv"}
    slopes = np.array([2.0 ** (-8.0 * (h + 1) / H) for h in range(H)])
    for beta in (1.0, 0.0):
        prm = {"alpha": (1 / slopes).astype(np.float32), "beta": np.full(H, beta, np.float32),
               "mu": np.zeros(H, np.float32), "s": np.ones(H, np.float32)}
        o, _ = _run(bits, prm, causal=True, ssmax=False)
        q, k, v = (f64(bits[n]) for n in "qkv")
        s = np.einsum("bhid,bhjd->bhij", q, k) / 8.0
        pos = np.arange(T)
        if beta == 1.0:
            s = s - slopes[None, :, None, None] * np.abs(pos[:, None] - pos[None, :])
        s = np.where(np.tril(np.ones((T, T), bool)), s, -np.inf)
        w = np.exp(s - s.max(-1, keepdims=True))
        ref = np.einsum("bhij,bhjd->bhid", w / w.sum(-1, keepdims=True), v)
        np.testing.assert_allclose(o, ref, rtol=0, atol=O_ATOL)


@pytest.mark.parametrize("rows", [1, 160])
def test_bf16_output_mode(rows):
    """bf16 O against fp32 O; 160 batch rows of the same two heads run the
    long-sequence kernel (its own bf16 staging and stores), one row the
    short-sequence one."""
    rng = np.random.default_rng(9)
    B, H, T = 1, 2, 384
    bits = {n: normal_bits(rng, (B, H, T, 64)) for n in "qkv"}
    bits = {n: np.ascontiguousarray(np.repeat(b, rows, axis=0)) for n, b in bits.items()}
    prm = random_params(H, rng)
    o16, lse16 = _run(bits, prm, True, True, o_dtype=torch.bfloat16)
    o32, lse32 = _run(bits, prm, True, True)
    # bf16 output = fp32 output rounded (half an ulp at |O| <= 8 is 2^-6)
    np.testing.assert_allclose(o16, o32, rtol=2 ** -8, atol=1e-6)
    np.testing.assert_array_equal(lse16, lse32)


def test_config1_full():
    d = make_inputs(1)
    o, lse = _run(d, d, d["causal"], d["ssmax"])
    oref, lref = _oracle(d, d, d["causal"], d["ssmax"])
    np.testing.assert_allclose(o, oref, rtol=0, atol=O_ATOL)
    np.testing.assert_allclose(lse, lref, rtol=LSE_RTOL, atol=LSE_ATOL)


def test_config2_forward_full():
    d = make_inputs(2)
    o, lse = _run(d, d, True, True)
    oref, lref = _oracle(d, d, True, True)
    np.testing.assert_allclose(o, oref, rtol=0, atol=O_ATOL)
    np.testing.assert_allclose(lse, lref, rtol=LSE_RTOL, atol=LSE_ATOL)


def _sampled_rows(T, per_head, rng):
    rows = {0, T - 1, T // 2, 127, 128, 255, 256}
    rows |= set(rng.integers(0, T, per_head).tolist())
    return sorted(r for r in rows if r < T)


@pytest.mark.parametrize("cfg,per_head", [(3, 40), (4, 12)])
def test_long_context_sampled_rows(cfg, per_head):
    d = make_inputs(cfg)
    w = workload(cfg)
    o, lse = _run(d, d, True, True)
    rng = np.random.default_rng(77)
    B, H, T = d["B"], d["H"], d["T"]
    for h in range(H):
        rows = _sampled_rows(T, per_head, rng)
        n = max(rows) + 1
        sl = (slice(0, 1), slice(h, h + 1), slice(0, n))
        sub = {x: d[x][sl] for x in "qkv"}
        ph = {x: d[x][h:h + 1] for x in ("alpha", "beta", "mu", "s")}
        oref, lref = oracle.fwd_rows(f64(sub["q"]), f64(sub["k"]), f64(sub["v"]), rows,
                                     ph["alpha"], ph["beta"], ph["mu"], ph["s"], causal=True,
                                     ssmax=True)
        np.testing.assert_allclose(o[0, h, rows], oref, rtol=0, atol=O_ATOL,
                                   err_msg=f"{w.name} head {h}")
        np.testing.assert_allclose(lse[0, h, rows], lref, rtol=LSE_RTOL, atol=LSE_ATOL)


def test_long_context_noncausal_sampled_rows():
    """The 32k prefill with every key visible (the bench's non-causal line):
    n = T for every row, distances of both signs."""
    d = make_inputs(3)
    o, lse = _run(d, d, False, True)
    rng = np.random.default_rng(78)
    B, H, T = d["B"], d["H"], d["T"]
    for h in range(H):
        rows = _sampled_rows(T, 12, rng)
        sub = {x: d[x][0:1, h:h + 1] for x in "qkv"}
        ph = {x: d[x][h:h + 1] for x in ("alpha", "beta", "mu", "s")}
        oref, lref = oracle.fwd_rows(f64(sub["q"]), f64(sub["k"]), f64(sub["v"]), rows,
                                     ph["alpha"], ph["beta"], ph["mu"], ph["s"], causal=False,
                                     ssmax=True)
        np.testing.assert_allclose(o[0, h, rows], oref, rtol=0, atol=O_ATOL,
                                   err_msg=f"non-causal head {h}")
        np.testing.assert_allclose(lse[0, h, rows], lref, rtol=LSE_RTOL, atol=LSE_ATOL)


def test_repeat_calls_identical():
    rng = np.random.default_rng(3)
    bits = {n: normal_bits(rng, (2, 2, 700, 64)) for n in "qkv"}
    prm = random_params(2, rng, mu_hi=3.0)
    o1, l1 = _run(bits, prm, True, True)
    o2, l2 = _run(bits, prm, True, True)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)


def test_binding_refuses_bad_tensors_then_runs():
    """A tensor of the wrong shape, dtype or layout is refused before any
    launch; the next good call on the same workspace is correct."""
    rng = np.random.default_rng(31)
    B, H, T = 1, 2, 130
    bits = {n: normal_bits(rng, (B, H, T, 64)) for n in "qkv"}
    prm_np = random_params(H, rng, mu_hi=3.0)
    q, k, v = (dev_bf16(bits[n]) for n in "qkv")
    t = params_dev(prm_np)
    prm = ba.make_params(t["alpha"], t["beta"], t["mu"], t["s"], 1e-5, True, True)
    o = torch.empty((B, H, T, 64), dtype=torch.float32, device="cuda")
    lse = torch.empty((B, H, T), dtype=torch.float32, device="cuda")
    ws = ba.workspace(ba.BAM_OP_FWD, B, H, T)
    k_strided = torch.empty((B, H, 64, T), dtype=torch.bfloat16, device="cuda").transpose(2, 3)
    n0 = ba.bam_attn_launch_count()
    with pytest.raises(ValueError, match="contiguous"):
        ba.bam_attn_fwd(q, k_strided, v, o, lse, prm, ws)
    with pytest.raises(ValueError, match="shape"):
        ba.bam_attn_fwd(q, k[:, :, :-1], v, o, lse, prm, ws)
    with pytest.raises(ValueError, match="dtype"):
        ba.bam_attn_fwd(q, k, v.float(), o, lse, prm, ws)
    with pytest.raises(ValueError, match="ws"):
        ba.bam_attn_fwd(q, k, v, o, lse, prm, ws.view(torch.int32))
    with pytest.raises(ValueError, match="shape"):
        ba.bam_attn_fwd(q[:, :1].contiguous(), k[:, :1].contiguous(), v[:, :1].contiguous(),
                        o[:, :1].contiguous(), lse[:, :1].contiguous(), prm, ws)
    assert ba.bam_attn_launch_count() == n0
    ba.bam_attn_fwd(q, k, v, o, lse, prm, ws)
    assert ba.bam_attn_check_status(ws) == ba.BAM_OK
    oref, _ = _oracle(bits, prm_np, True, True)
    np.testing.assert_allclose(o.cpu().numpy(), oref, rtol=0, atol=O_ATOL)
