"""The per-head distance table against the oracle's bias, entry by entry.

The forward writes b_h(d) * log2(e) for every distance its tiles can touch
into the workspace right after the 256 status bytes: H rows of `len`
entries, entry x holding d = x - off (len, off as laid out by the library:
off = 256 causal, round_up(T,256) + 256 otherwise; len = off +
round_up(T,256) + 256).  fp32 storage of an fp32-evaluated value with a
compensated exponent: relative error <= 1e-6 against the fp64 oracle.
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
    tab = ws[256:256 + H * length * 4].cpu().numpy().view(np.float32).reshape(H, length)
    log2e = 1.0 / math.log(2.0)
    worst = 0.0
    for h in range(H):
        ref = np.array([oracle.bias(x - off, prm["alpha"][h], prm["beta"][h], prm["mu"][h])
                        for x in range(length)]) * log2e
        ref = np.maximum(ref, -3.0e38)
        err = np.abs(tab[h] - ref) / np.maximum(np.abs(ref), 1e-30)
        worst = max(worst, float(err.max()))
        assert err.max() <= 1e-6, (h, int(err.argmax()), tab[h][err.argmax()], ref[err.argmax()])
