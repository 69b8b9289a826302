"""Pins for the oracle's bf16 conversions (CPU only).

The oracle rounds float64 results to bf16 once, round-to-nearest-even; these
tests fix that against IEEE 754 facts and against torch's float32 -> bf16
cast (a library routine) on float32-representable inputs.
"""

import numpy as np
import torch

from oracle import bf16_bits_to_f64, f64_to_bf16_bits


def test_widen_known_patterns():
    bits = np.array([0x3F80, 0xC000, 0x7F80, 0xFF80, 0x0001, 0x3F81, 0x0000, 0x8000], np.uint16)
    want = [1.0, -2.0, np.inf, -np.inf, 2.0 ** -133, 1.0 + 2.0 ** -7, 0.0, -0.0]
    got = bf16_bits_to_f64(bits)
    assert np.array_equal(got, np.array(want))
    assert np.signbit(got[-1])


def test_roundtrip_every_finite_pattern():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    x = bf16_bits_to_f64(bits)
    keep = ~np.isnan(x)
    back = f64_to_bf16_bits(x[keep])
    assert np.array_equal(back, bits[keep])


def test_ties_go_to_even():
    # 1 + 2^-8 is halfway between 1.0 (mantissa even) and 1 + 2^-7 (odd).
    assert f64_to_bf16_bits(1.0 + 2.0 ** -8) == 0x3F80
    # 1 + 3*2^-8 is halfway between 1 + 2^-7 (odd) and 1 + 2^-6 (even).
    assert f64_to_bf16_bits(1.0 + 3 * 2.0 ** -8) == 0x3F82
    assert f64_to_bf16_bits(-(1.0 + 2.0 ** -8)) == 0xBF80


def test_single_rounding_no_double_rounding():
    # Just above the tie: correct single rounding goes up.  Rounding to
    # float32 first would land exactly on the tie and then go down to 1.0.
    x = 1.0 + 2.0 ** -8 + 2.0 ** -40
    assert f64_to_bf16_bits(x) == 0x3F81
    x = 1.0 + 2.0 ** -8 - 2.0 ** -40
    assert f64_to_bf16_bits(x) == 0x3F80


def test_subnormals_and_overflow():
    assert f64_to_bf16_bits(2.0 ** -133) == 0x0001
    assert f64_to_bf16_bits(2.0 ** -134) == 0x0000          # tie -> even (0)
    assert f64_to_bf16_bits(1.5 * 2.0 ** -134) == 0x0001
    assert f64_to_bf16_bits(3.0 * 2.0 ** -134) == 0x0002    # tie 1.5 ulp -> even 2
    big = (2.0 - 2.0 ** -7) * 2.0 ** 127                     # largest finite bf16
    assert f64_to_bf16_bits(big) == 0x7F7F
    assert f64_to_bf16_bits((2.0 - 2.0 ** -8) * 2.0 ** 127) == 0x7F80   # tie -> inf (even)
    assert f64_to_bf16_bits(-1e300) == 0xFF80
    assert f64_to_bf16_bits(np.nan) & 0x7F80 == 0x7F80


def test_matches_torch_cast_on_float32_inputs():
    g = torch.Generator().manual_seed(0)
    x32 = torch.randn(200000, generator=g) * torch.exp(4 * torch.randn(200000, generator=g))
    want = x32.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = f64_to_bf16_bits(x32.numpy().astype(np.float64))
    assert np.array_equal(got, want)
