"""bam_attn_decode_noalloc: decode for callers that cannot allocate.

Plugin-style hosts hand a library only input and output pointers and own
all other device memory, and a per-token decode loop cannot afford
cudaMalloc's possible device-wide synchronisation; this entry point takes
its scratch from a fixed array in the library instead of a workspace.  The
test calls it through the C ABI and checks it against bam_attn_decode (the
workspace entry point) on two calls in a row, with the parity tolerances of
the other tests.  The file name makes pytest collect it last.
"""

import ctypes

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from transformer_attention_ggd_gb300 import bam_attn as ba
from transformer_attention_ggd_gb300 import build as lib_build
from transformer_attention_ggd_gb300.inputs import random_params

from _gpu_helpers import LSE_ATOL, LSE_RTOL, O_ATOL, dev_bf16, normal_bits, params_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    lib_build.build()
    return ba.load_library()


def _case(seed, B, H, Tkv):
    rng = np.random.default_rng(seed)
    q = dev_bf16(normal_bits(rng, (B, H, 64)))
    kc = dev_bf16(normal_bits(rng, (B, H, Tkv, 64)))
    vc = dev_bf16(normal_bits(rng, (B, H, Tkv, 64)))
    prm = random_params(H, rng, mu_hi=6.0)
    prm["beta"][0] = -0.4
    return q, kc, vc, params_dev(prm)


def test_noalloc_matches_workspace_decode_twice(lib):
    # Two calls in a row with different sizes: the second must not depend on
    # what the first left in the shared scratch.
    for seed, (B, H, Tkv) in ((1, (4, 12, 5000)), (2, (64, 12, 2048))):
        q, kc, vc, t = _case(seed, B, H, Tkv)
        prm = ba.make_params(t["alpha"], t["beta"], t["mu"], t["s"], 1e-5, True, True)
        o_ref = torch.empty((B, H, 64), dtype=torch.float32, device="cuda")
        l_ref = torch.empty((B, H), dtype=torch.float32, device="cuda")
        ws = ba.workspace(ba.BAM_OP_DECODE, B, H, Tkv)
        ba.bam_attn_decode(q, kc, vc, o_ref, l_ref, prm, ws)
        o = torch.full((B, H, 64), float("nan"), dtype=torch.float32, device="cuda")
        lse = torch.full((B, H), float("nan"), dtype=torch.float32, device="cuda")
        ba.bam_attn_decode_noalloc(q, kc, vc, o, lse, prm)
        torch.cuda.synchronize()
        np.testing.assert_allclose(o.cpu().numpy(), o_ref.cpu().numpy(), rtol=0, atol=O_ATOL)
        np.testing.assert_allclose(lse.cpu().numpy(), l_ref.cpu().numpy(), rtol=LSE_RTOL,
                                   atol=LSE_ATOL)


def test_noalloc_rejects_sizes_beyond_its_scratch(lib):
    B, H, Tkv = 64, 64, 1 << 20
    assert ba.bam_attn_workspace_size(ba.BAM_OP_DECODE, B, H, Tkv) > \
        ba.BAM_DECODE_NOALLOC_SCRATCH_BYTES
    fake = ctypes.c_void_p(0x7F0000000000)
    p = ba.BamParams(0x7F0000000000, 0x7F0000000000, 0x7F0000000000, 0x7F0000000000, 1e-5, 1, 1)
    st = lib.bam_attn_decode_noalloc(fake, fake, fake, fake, 1, None, B, H, Tkv, 64,
                                     ctypes.byref(p), None)
    assert st == ba.BAM_ERR_WORKSPACE
