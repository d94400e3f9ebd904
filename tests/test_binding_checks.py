"""Argument checks of the Python binding, on the host: the C ABI receives raw
pointers only, so the binding refuses a tensor of the wrong shape, dtype,
device or layout before anything reaches a kernel.  No GPU needed: every
call here is refused before the library is called."""

import pytest

torch = pytest.importorskip("torch")

from transformer_attention_ggd_gb300 import bam_attn as ba

CPU = torch.device("cpu")


def test_require_accepts_a_matching_tensor():
    ba._require(torch.zeros(2, 3, dtype=torch.float32), "x", (2, 3), (torch.float32,), CPU)
    ba._require(None, "x", (2, 3), (torch.float32,), CPU, optional=True)


@pytest.mark.parametrize("t,msg", [
    (torch.zeros(2, 3, dtype=torch.float64), "dtype"),
    (torch.zeros(3, 2, dtype=torch.float32), "shape"),
    (torch.zeros(3, 2, dtype=torch.float32).t(), "contiguous"),
    (None, "required"),
])
def test_require_rejects(t, msg):
    with pytest.raises(ValueError, match=msg):
        ba._require(t, "x", (2, 3), (torch.float32,), CPU)


def test_require_rejects_another_device():
    with pytest.raises(ValueError, match="expected meta"):
        ba._require(torch.zeros(2, 3), "x", (2, 3), (torch.float32,), torch.device("meta"))
    with pytest.raises(TypeError):
        ba._require([0.0] * 6, "x", (2, 3), (torch.float32,), CPU)


def _params(H=3, dtype=torch.float32):
    return [torch.ones(H, dtype=dtype) for _ in range(4)]


def test_make_params_checks_the_per_head_tensors():
    a, b, m, s = _params()
    prm = ba.make_params(a, b, m, s, 1e-5, True, True)
    assert prm.tensors[0] is a and prm.alpha == a.data_ptr()
    with pytest.raises(ValueError, match="dtype"):
        ba.make_params(*_params(dtype=torch.float64))
    with pytest.raises(ValueError, match="shape"):
        ba.make_params(a, b, torch.ones(4), s)
    with pytest.raises(ValueError, match="ssmax needs"):
        ba.make_params(a, b, m, None, ssmax=True)
    with pytest.raises(ValueError, match="1-D"):
        ba.make_params(torch.ones(2, 2), b, m, s)


def test_entry_points_refuse_host_tensors_before_the_library():
    B, H, T, D = 1, 2, 8, 64
    x = torch.zeros(B, H, T, D, dtype=torch.bfloat16)
    lse = torch.zeros(B, H, T)
    prm = ba.make_params(*_params(H))
    ws = torch.zeros(256, dtype=torch.uint8)
    g = torch.zeros(H)
    calls = [
        lambda: ba.bam_attn_fwd(x, x, x, x, lse, prm, ws),
        lambda: ba.bam_attn_bwd(x, x, x, x, lse, x, x, x, x, g, g, g, g, prm, ws),
        lambda: ba.bam_attn_decode(x[:, :, 0], x, x, x[:, :, 0], None, prm, ws),
        lambda: ba.bam_attn_decode_noalloc(x[:, :, 0], x, x, x[:, :, 0], None, prm),
        lambda: ba.bam_attn_decode_varlen(x[:, :, 0], x, x, torch.ones(B, dtype=torch.int32),
                                          x[:, :, 0], None, prm, ws),
        lambda: ba.bam_attn_decode_paged(x[:, :, 0], x, x, torch.zeros(B, 1, dtype=torch.int32),
                                         torch.ones(B, dtype=torch.int32), x[:, :, 0], None,
                                         prm, ws),
    ]
    for call in calls:
        with pytest.raises(ValueError, match="CUDA tensor"):
            call()
