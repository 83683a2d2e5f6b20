"""Pins for the oracle's own IEEE 754 binary16 conversion.

The oracle rounds every float16 result with a conversion written from the
binary16 format definition.  These tests pin it against facts that do not come
from the oracle: the exhaustive set of 65,536 patterns, numpy's and torch's
library conversions, and hand-derived boundary cases (largest finite value,
overflow midpoint, subnormal quantum, ties to even).
"""
import numpy as np
import pytest
import torch

import oracle


def _all_patterns():
    return np.arange(65536, dtype=np.uint32).astype(np.uint16)


def test_f16_to_f32_exhaustive_matches_numpy():
    bits = _all_patterns()
    ours = oracle.f16_to_f32(bits.view(np.float16))
    ref = bits.view(np.float16).astype(np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def test_f32_round_trip_exhaustive():
    bits = _all_patterns()
    f = bits.view(np.float16).astype(np.float32)
    back = oracle.f32_to_f16(f).view(np.uint16)
    nan = np.isnan(f)
    assert np.array_equal(back[~nan], bits[~nan])
    assert np.all(np.isnan(back[nan].view(np.float16)))


def test_f32_to_f16_random_bits_match_numpy_and_torch():
    rng = np.random.default_rng(123)
    # Random binary32 bit patterns concentrated on the binary16 range and its
    # neighbourhood (exponent fields 100..150), plus fully random patterns.
    n = 2_000_000
    exp = rng.integers(100, 151, size=n, dtype=np.uint32)
    man = rng.integers(0, 1 << 23, size=n, dtype=np.uint32)
    sign = rng.integers(0, 2, size=n, dtype=np.uint32)
    f = ((sign << 31) | (exp << 23) | man).view(np.float32)
    f = np.concatenate([f, rng.integers(0, 2**32, size=n, dtype=np.uint64)
                        .astype(np.uint32).view(np.float32)])
    f = f[~np.isnan(f)]
    ours = oracle.f32_to_f16(f).view(np.uint16)
    with np.errstate(over="ignore"):
        ref_np = f.astype(np.float16).view(np.uint16)
    assert np.array_equal(ours, ref_np)
    ref_torch = torch.from_numpy(f).to(torch.float16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref_torch)


def test_f64_to_f16_single_rounding_matches_numpy():
    """Double -> half must round once.  Values just above a half-way point
    between two float16 neighbours are the cases where going through float32
    would round twice and land on the wrong neighbour."""
    rng = np.random.default_rng(7)
    base = rng.integers(0, 0x7c00, size=200_000, dtype=np.uint16).view(np.float16)
    with np.errstate(over="ignore", invalid="ignore"):
        lo = base.astype(np.float64)
        hi = np.nextafter(base, np.float16(np.inf)).astype(np.float64)
        mid = (lo + hi) / 2
        tiny = np.abs(hi - lo) * 2.0 ** -30
        probes = np.concatenate([mid, mid + tiny, mid - tiny, -(mid + tiny),
                                 rng.standard_normal(200_000) * 1000.0])
    probes = probes[np.isfinite(probes)]
    ours = oracle.f64_to_f16(probes).view(np.uint16)
    ref = probes.astype(np.float16).view(np.uint16)
    assert np.array_equal(ours, ref)
    # the double-rounding case written out: 1 + 2^-11 + 2^-40 lies above the
    # midpoint between 1 and 1 + 2^-10, so it rounds up; via float32 it would
    # become exactly the midpoint and round down to 1.
    v = 1.0 + 2.0 ** -11 + 2.0 ** -40
    assert oracle.f64_to_f16(np.array([v])).view(np.uint16)[0] == 0x3C01


@pytest.mark.parametrize("value,bits", [
    (65504.0, 0x7BFF),                  # largest finite
    (65519.99, 0x7BFF),                 # below the overflow midpoint
    (65520.0, 0x7C00),                  # midpoint: ties to even -> overflow
    (-65520.0, 0xFC00),
    (2.0 ** -24, 0x0001),               # smallest subnormal
    (2.0 ** -25, 0x0000),               # half of it: tie to even -> +0
    (3 * 2.0 ** -26, 0x0001),           # 0.75 quantum -> 1 quantum
    (3 * 2.0 ** -25, 0x0002),           # 1.5 quanta: tie -> even (2)
    (2.0 ** -14, 0x0400),               # smallest normal
    (2.0 ** -14 - 2.0 ** -25, 0x0400),  # 1023.5 quanta: tie -> 1024 (normal)
    (1.0 + 2.0 ** -11, 0x3C00),         # tie between 1 and 1+2^-10 -> 1 (even)
    (1.0 + 3 * 2.0 ** -11, 0x3C02),     # tie -> even neighbour 1+2^-9
    (-0.0, 0x8000),
    (float("inf"), 0x7C00),
])
def test_f16_hand_boundaries(value, bits):
    assert oracle.f64_to_f16(np.array([value])).view(np.uint16)[0] == bits
