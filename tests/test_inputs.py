"""The seeded input module shared by the oracle and the CUDA path: its bf16
rounding against PyTorch's float32 -> bfloat16 conversion (round to nearest
even), its exact widening, and the seeding of the workloads."""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from transformer_attention_ggd_gb300.inputs import bf16_bits, bf16_to_f32, make_inputs


def _torch_bits(x):
    return torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_rounding_matches_torch():
    rng = np.random.default_rng(0)
    parts = [rng.standard_normal(200_000).astype(np.float32) * s
             for s in (1e-40, 1e-30, 1e-3, 1.0, 1e3, 1e30)]
    special = np.array([0.0, -0.0, 1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, 1.0 - 2.0 ** -9,
                        np.finfo(np.float32).max, np.finfo(np.float32).tiny, 1e-45,
                        np.inf, -np.inf], np.float32)
    x = np.concatenate(parts + [special])
    np.testing.assert_array_equal(bf16_bits(x), _torch_bits(x))


def test_ties_go_to_even():
    # 1 + 2^-8 lies halfway between bf16 1 and 1 + 2^-7: even mantissa (1) wins;
    # 1 + 3 * 2^-8 lies halfway between 1 + 2^-7 and 1 + 2^-6: 1 + 2^-6 wins.
    x = np.array([1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8], np.float32)
    np.testing.assert_array_equal(bf16_to_f32(bf16_bits(x)), [1.0, 1.0 + 2.0 ** -6])


def test_every_bf16_pattern_round_trips():
    b = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    f = bf16_to_f32(b)
    ok = ~np.isnan(f)
    np.testing.assert_array_equal(bf16_bits(f)[ok], b[ok])
    assert np.all(np.isnan(bf16_to_f32(bf16_bits(f[~ok]))))


def test_nan_stays_nan():
    x = np.array([0x7F800001, 0xFF800001, 0x7FC00000], np.uint32).view(np.float32)
    assert np.all(np.isnan(bf16_to_f32(bf16_bits(x))))


def test_workloads_are_seeded_and_shaped():
    a, b = make_inputs(1), make_inputs(1)
    for n in ("q", "k", "v", "alpha", "beta", "mu", "s"):
        np.testing.assert_array_equal(a[n], b[n])
    assert a["q"].shape == (a["B"], a["H"], a["T"], 64) and a["q"].dtype == np.uint16
    c = make_inputs(1, seed=7)
    assert not np.array_equal(a["q"], c["q"])
    d = make_inputs(2, B=1, H=2, T=16)
    assert d["do"].shape == (1, 2, 16, 64)
    e = make_inputs(5, B=2, H=3, T=100)
    assert e["q"].shape == (2, 3, 64) and e["k"].shape == (2, 3, 100, 64)
