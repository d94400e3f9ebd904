"""The per-head distance table against the oracle's bias, entry by entry.

The forward writes b_h(d) * log2(e) for every distance its tiles can touch
into the workspace right after the 256 status bytes.  Rows are stored
reversed, in four copies each shifted by one more entry: copy k holds H rows
of `len` entries, entry y of a row holding table index x = len - 1 - y + k,
i.e. d = x - off (0 where x >= len), with off = 256 causal,
round_up(T,256) + 256 otherwise and len = off + round_up(T,256) + 256.
fp32 storage of an fp32-evaluated value with a compensated exponent:
relative error <= 1e-6 against the fp64 oracle.
"""

import math

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
from transformer_attention_ggd_gb300 import bam_attn as ba

from _gpu_helpers import dev_bf16, params_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    ba.load_library()


@pytest.mark.parametrize("causal", [True, False])
def test_distance_table_matches_oracle_bias(causal):
    T, H = 700, 6
    prm = {"alpha": np.array([1.0, 7.5, 300.0, 1e4, 0.3, 40.0], np.float32),
           "beta": np.array([2.0, 0.5, -0.7, -1.0, 1.0, 0.0], np.float32),
           "mu": np.array([0.0, 3.25, 60.0, 0.0, 2.0, 5.0], np.float32),
           "s": np.ones(H, np.float32)}
    z = np.zeros((1, H, T, 64), np.uint16)
    q = dev_bf16(z)
    ws = ba.workspace(ba.BAM_OP_FWD, 1, H, T)
    t = params_dev(prm)
    ba.attention_forward(q, q, q, t["alpha"], t["beta"], t["mu"], t["s"], causal=causal,
                         ws=ws)
    torch.cuda.synchronize()
    t256 = (T + 255) // 256 * 256
    off = 256 if causal else t256 + 256
    length = off + t256 + 256
    copies = ws[256:256 + 4 * H * length * 4].cpu().numpy().view(np.float32)
    copies = copies.reshape(4, H, length)
    log2e = 1.0 / math.log(2.0)
    worst = 0.0
    for h in range(H):
        ref = np.array([oracle.bias(x - off, prm["alpha"][h], prm["beta"][h], prm["mu"][h])
                        for x in range(length)]) * log2e
        ref = np.maximum(ref, -3.0e38)
        tab = copies[0, h, ::-1]  # copy 0 reversed back: entry x
        err = np.abs(tab - ref) / np.maximum(np.abs(ref), 1e-30)
        worst = max(worst, float(err.max()))
        assert err.max() <= 1e-6, (h, int(err.argmax()), tab[err.argmax()], ref[err.argmax()])
        for k in range(1, 4):
            # copy k is copy 0 shifted by k entries, zero-filled at the front
            assert np.array_equal(copies[k, h, k:], copies[0, h, :length - k]), (h, k)
            assert np.all(copies[k, h, :k] == 0.0), (h, k)


@pytest.mark.parametrize("causal", [True, False])
def test_backward_tables_match_oracle_bias_grad(causal):
    """The backward preprocess's three planes, copy 0 each: b log2 e,
    db/dbeta = b ln(u/alpha) and db/dmu = -beta b sgn(d - mu) / u (0 inside
    the eps clamp and at u = 0), against the oracle's partial derivatives."""
    T, H = 700, 6
    prm = {"alpha": np.array([1.0, 7.5, 300.0, 1e4, 0.3, 40.0], np.float32),
           "beta": np.array([2.0, 0.5, -0.7, -1.0, 1.0, 0.0], np.float32),
           "mu": np.array([0.0, 3.25, 60.0, 0.0, 2.0, 5.0], np.float32),
           "s": np.ones(H, np.float32)}
    z = dev_bf16(np.zeros((1, H, T, 64), np.uint16))
    t = params_dev(prm)
    o, lse = ba.attention_forward(z, z, z, t["alpha"], t["beta"], t["mu"], t["s"],
                                  causal=causal)
    ws = ba.workspace(ba.BAM_OP_BWD, 1, H, T)
    ba.attention_backward(z, z, z, o, lse, z, t["alpha"], t["beta"], t["mu"], t["s"],
                          causal=causal, ws=ws)
    torch.cuda.synchronize()
    t256 = (T + 255) // 256 * 256
    off = 256 if causal else t256 + 256
    length = off + t256 + 256
    planes = ws[256:256 + 3 * 4 * H * length * 4].cpu().numpy().view(np.float32)
    planes = planes.reshape(3, 4, H, length)
    log2e = 1.0 / math.log(2.0)
    for h in range(H):
        a, b, m = prm["alpha"][h], prm["beta"][h], prm["mu"][h]
        refs = [np.array([oracle.bias(x - off, a, b, m) for x in range(length)]) * log2e]
        g = np.array([oracle.bias_grad(x - off, a, b, m) for x in range(length)])
        refs += [g[:, 1], g[:, 2]]
        for p, name in enumerate(("b", "db/dbeta", "db/dmu")):
            ref = np.clip(refs[p], -3.0e38, 3.0e38)
            got = planes[p, 0, h, ::-1]
            err = np.abs(got - ref) / np.maximum(np.abs(ref), 1e-30)
            bad = (err > 1e-6) & ~((ref == 0.0) & (got == 0.0))
            assert not bad.any(), (name, h, int(bad.argmax()) - off, got[bad.argmax()],
                                   ref[bad.argmax()])
