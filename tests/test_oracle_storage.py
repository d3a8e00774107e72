"""Pins for the oracle's storage rounding (fp64 -> bf16 / fp32, round-to-nearest-even)."""

from fractions import Fraction

import numpy as np
import torch

from oracle.storage import round_to_storage


def _nearest_even(x, mant_bits):
    """Brute force: the nearest value with ``mant_bits`` stored mantissa bits, ties to even."""
    f = Fraction(x)
    if f == 0:
        return 0.0
    sign = -1 if f < 0 else 1
    a = abs(f)
    e = 0
    while a >= 2:
        a /= 2
        e += 1
    while a < 1:
        a *= 2
        e -= 1
    scaled = a * (1 << mant_bits)
    lo = scaled.numerator // scaled.denominator
    rem = scaled - lo
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and lo % 2 == 1):
        lo += 1
    return sign * float(Fraction(lo, 1 << mant_bits) * (Fraction(2) ** e))


def test_bf16_matches_torch_on_fp32_values():
    rng = np.random.default_rng(1)
    x32 = (rng.standard_normal(20000) * np.exp(rng.uniform(-20, 20, 20000))).astype(np.float32)
    # exact ties: fp32 values whose low 16 bits are 0x8000
    ties = (rng.integers(0x3F800000, 0x40800000, 2000, dtype=np.int64) & ~0xFFFF) | 0x8000
    x32 = np.concatenate([x32, ties.astype(np.uint32).view(np.float32)])
    ref = torch.from_numpy(x32).to(torch.bfloat16).to(torch.float64).numpy()
    got = round_to_storage(x32.astype(np.float64), "bf16")
    assert np.array_equal(got, ref)


def test_bf16_matches_exact_rational_on_fp64_values():
    rng = np.random.default_rng(2)
    xs = rng.standard_normal(400) * np.exp(rng.uniform(-30, 30, 400))
    got = round_to_storage(xs, "bf16")
    for x, y in zip(xs, got):
        assert y == _nearest_even(float(x), 7)


def test_f32_matches_exact_rational():
    rng = np.random.default_rng(3)
    xs = rng.standard_normal(300) * np.exp(rng.uniform(-30, 30, 300))
    got = round_to_storage(xs, "f32")
    for x, y in zip(xs, got):
        assert y == _nearest_even(float(x), 23)


def test_f64_is_identity():
    xs = np.random.default_rng(4).standard_normal(100)
    assert np.array_equal(round_to_storage(xs, "f64"), xs)
