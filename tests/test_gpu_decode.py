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


# ---------------------------------------------------------------- ragged decode

def _varlen(q, kc, vc, lens, prm, ssmax, o_dtype=torch.float32):
    t = params_dev(prm)
    ln = torch.from_numpy(np.asarray(lens, np.int32)).cuda()
    ws = ba.workspace(ba.BAM_OP_DECODE, kc.shape[0], kc.shape[1], kc.shape[2])
    o, lse = ba.attention_decode_varlen(dev_bf16(q), dev_bf16(kc), dev_bf16(vc), ln, t["alpha"],
                                        t["beta"], t["mu"], t["s"], ssmax=ssmax, o_dtype=o_dtype,
                                        ws=ws)
    status = ba.bam_attn_check_status(ws)
    return o.float().cpu().numpy(), lse.cpu().numpy(), status


def _varlen_ref(q, kc, vc, lens, prm, ssmax):
    """Each sequence is a plain decode over its own cache prefix."""
    B, H = q.shape[:2]
    o = np.zeros((B, H, 64))
    lse = np.zeros((B, H))
    for b, n in enumerate(lens):
        ob, lb = oracle.decode(f64(q[b:b + 1]), f64(kc[b:b + 1, :, :n]), f64(vc[b:b + 1, :, :n]),
                               prm["alpha"], prm["beta"], prm["mu"], prm["s"], ssmax=ssmax)
        o[b], lse[b] = ob[0], lb[0]
    return o, lse


@pytest.mark.parametrize("ssmax", [True, False])
def test_varlen_matches_per_sequence_decode(ssmax):
    rng = np.random.default_rng(61 + ssmax)
    B, H, Tmax = 7, 3, 700
    lens = [1, 2, 63, 64, 65, 333, 700]
    q = normal_bits(rng, (B, H, 64))
    kc, vc = normal_bits(rng, (B, H, Tmax, 64)), normal_bits(rng, (B, H, Tmax, 64))
    prm = random_params(H, rng, mu_hi=6.0)
    prm["beta"][2] = -0.4
    o, lse, st = _varlen(q, kc, vc, lens, prm, ssmax)
    assert st == ba.BAM_OK
    oref, lref = _varlen_ref(q, kc, vc, lens, prm, ssmax)
    np.testing.assert_allclose(o, oref, rtol=0, atol=O_ATOL)
    np.testing.assert_allclose(lse, lref, rtol=LSE_RTOL, atol=LSE_ATOL)


def test_varlen_at_full_length_is_the_plain_decode():
    rng = np.random.default_rng(62)
    B, H, Tmax = 3, 4, 1000
    q = normal_bits(rng, (B, H, 64))
    kc, vc = normal_bits(rng, (B, H, Tmax, 64)), normal_bits(rng, (B, H, Tmax, 64))
    prm = random_params(H, rng, mu_hi=4.0)
    o1, l1, st = _varlen(q, kc, vc, [Tmax] * B, prm, True)
    o2, l2 = _run(q, kc, vc, prm, True)
    assert st == ba.BAM_OK
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)


def test_varlen_out_of_range_length_is_reported():
    """A cache length outside [1, Tmax] is clamped on the device (no access
    beyond the cache) and reported by check_status; the other sequences are
    unaffected."""
    rng = np.random.default_rng(63)
    B, H, Tmax = 3, 2, 200
    q = normal_bits(rng, (B, H, 64))
    kc, vc = normal_bits(rng, (B, H, Tmax, 64)), normal_bits(rng, (B, H, Tmax, 64))
    prm = random_params(H, rng)
    o, lse, st = _varlen(q, kc, vc, [0, 50, Tmax + 7], prm, True)
    assert st == ba.BAM_ERR_INVALID_ARG
    oref, lref = _varlen_ref(q, kc, vc, [1, 50, Tmax], prm, True)
    np.testing.assert_allclose(o, oref, rtol=0, atol=O_ATOL)
    # the status word is cleared by the read: a good call afterwards is clean
    o, lse, st = _varlen(q, kc, vc, [1, 50, Tmax], prm, True)
    assert st == ba.BAM_OK


def test_varlen_full_size():
    """B=64 H=12 Tmax=32768 with seeded lengths U[1, Tmax] (the bench's ragged
    decode line), every sequence against the oracle."""
    d = make_inputs(5)
    B, H, Tmax = d["B"], d["H"], d["T"]
    lens = np.random.default_rng(5005).integers(1, Tmax + 1, B)
    lens[:3] = [1, Tmax, 64]
    o, lse, st = _varlen(d["q"], d["k"], d["v"], lens, d, True)
    assert st == ba.BAM_OK
    oref, lref = _varlen_ref(d["q"], d["k"], d["v"], lens, d, True)
    np.testing.assert_allclose(o, oref, rtol=0, atol=O_ATOL)
    np.testing.assert_allclose(lse, lref, rtol=LSE_RTOL, atol=LSE_ATOL)


# ---------------------------------------------------------------- paged decode

def _to_pages(kc, lens, page, rng, extra_pages=3, junk=True):
    """Scatter a contiguous [B,H,Tmax,64] cache into randomly permuted pages
    [num_pages,H,page,64] (unused pages and the tails of partly used ones hold
    junk, or zeros); block-table entries past a sequence's length are -1
    (never read)."""
    B, H, Tmax, D = kc.shape
    max_blocks = Tmax // page
    used = [(b, i) for b in range(B) for i in range((lens[b] + page - 1) // page)]
    num_pages = len(used) + extra_pages
    perm = rng.permutation(num_pages)[:len(used)]
    shape = (num_pages, H, page, D)
    pages = rng.integers(0, 1 << 16, shape).astype(np.uint16) if junk else np.zeros(shape,
                                                                                      np.uint16)
    table = np.full((B, max_blocks), -1, np.int32)
    for (b, i), pg in zip(used, perm):
        table[b, i] = pg
        pages[pg] = kc[b, :, i * page:(i + 1) * page]
    return pages, table


def _paged(q, kp, vp, table, lens, prm, ssmax):
    t = params_dev(prm)
    B, H = q.shape[:2]
    ws = ba.workspace(ba.BAM_OP_DECODE, B, H, kp.shape[2] * table.shape[1])
    o, lse = ba.attention_decode_paged(
        dev_bf16(q), dev_bf16(kp), dev_bf16(vp), torch.from_numpy(table).cuda(),
        torch.from_numpy(np.asarray(lens, np.int32)).cuda(), t["alpha"], t["beta"], t["mu"],
        t["s"], ssmax=ssmax, ws=ws)
    status = ba.bam_attn_check_status(ws)
    return o.float().cpu().numpy(), lse.cpu().numpy(), status


@pytest.mark.parametrize("page", [64, 256])
def test_paged_equals_contiguous_ragged(page):
    """Same kernels, same order of arithmetic: only the source addresses of the
    K/V stages differ, so the results are bit-identical."""
    rng = np.random.default_rng(70 + page)
    B, H, Tmax = 6, 3, 1024
    lens = [1, 63, 64, 65, 700, 1024]
    q = normal_bits(rng, (B, H, 64))
    kc, vc = normal_bits(rng, (B, H, Tmax, 64)), normal_bits(rng, (B, H, Tmax, 64))
    prm = random_params(H, rng, mu_hi=5.0)
    kp, table = _to_pages(kc, lens, page, np.random.default_rng(1))
    vp, _ = _to_pages(vc, lens, page, np.random.default_rng(1))
    o1, l1, st1 = _paged(q, kp, vp, table, lens, prm, True)
    o2, l2, st2 = _varlen(q, kc, vc, lens, prm, True)
    assert st1 == ba.BAM_OK and st2 == ba.BAM_OK
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)
    oref, lref = _varlen_ref(q, kc, vc, lens, prm, True)
    np.testing.assert_allclose(o1, oref, rtol=0, atol=O_ATOL)


def test_paged_bad_page_is_reported():
    rng = np.random.default_rng(72)
    B, H, Tmax, page = 2, 2, 256, 64
    lens = [200, 256]
    q = normal_bits(rng, (B, H, 64))
    kc, vc = normal_bits(rng, (B, H, Tmax, 64)), normal_bits(rng, (B, H, Tmax, 64))
    prm = random_params(H, rng)
    kp, table = _to_pages(kc, lens, page, np.random.default_rng(2))
    vp, _ = _to_pages(vc, lens, page, np.random.default_rng(2))
    table[1, 2] = kp.shape[0] + 5   # a used block pointing past the pool
    o, lse, st = _paged(q, kp, vp, table, lens, prm, True)
    assert st == ba.BAM_ERR_INVALID_ARG
    assert np.all(np.isfinite(o))


def test_paged_full_size():
    """B=64 H=12 with lengths U[1, 32768] in 256-key pages, permuted: equal to
    the contiguous ragged decode (the bench's paged line)."""
    d = make_inputs(5)
    B, H, Tmax = d["B"], d["H"], d["T"]
    lens = np.random.default_rng(5005).integers(1, Tmax + 1, B)
    lens[:3] = [1, Tmax, 64]
    kp, table = _to_pages(d["k"], lens, 256, np.random.default_rng(6), extra_pages=0, junk=False)
    vp, _ = _to_pages(d["v"], lens, 256, np.random.default_rng(6), extra_pages=0, junk=False)
    o1, l1, st1 = _paged(d["q"], kp, vp, table, lens, d, True)
    o2, l2, st2 = _varlen(d["q"], d["k"], d["v"], lens, d, True)
    assert st1 == ba.BAM_OK and st2 == ba.BAM_OK
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)
