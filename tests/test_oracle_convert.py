"""Pins for the oracle's own binary16 converters (used for every scale and zero).

The reference points are independent implementations: numpy's float32 ->
float16 cast (round to nearest, ties to even) and numpy's float16 -> float32
widening, compared over every binary32 / binary16 bit pattern.
"""
import numpy as np
import pytest

import oracle


def test_f16_to_f32_exhaustive(oracle_lib):
    h = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ours = oracle.f16_bits_to_f32(h)
    ref = h.view(np.float16).astype(np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def test_f32_to_f16_exhaustive(oracle_lib):
    """Every binary32 pattern whose binary16 rounding is non-trivial (|x| in [2^-26, 2^16),
    both signs: 2 x 42 x 2^23 patterns) is bit-identical to numpy's cast; every pattern
    below 2^-26 gives a signed zero and every finite pattern from 2^16 up gives a signed
    infinity (checked on all exponents with a sample of fractions); NaN stays NaN."""
    chunk = 1 << 23
    for sign in (0, 1):
        for E in range(101, 143):
            start = (sign << 31) | (E << 23)
            u = np.arange(start, start + chunk, dtype=np.uint64).astype(np.uint32)
            x = u.view(np.float32)
            ours = oracle.f32_to_f16_bits(x)
            ref = x.astype(np.float16).view(np.uint16)
            bad = np.nonzero(ours != ref)[0]
            assert bad.size == 0, f"pattern {int(u[bad[0]]):#010x}: {ours[bad[0]]:#06x} vs {ref[bad[0]]:#06x}"
    rng = np.random.default_rng(0)
    frac = np.concatenate([[0, 1, 0x7FFFFF, 0x400000], rng.integers(0, 1 << 23, 252)]).astype(np.uint32)
    for sign in (0, 1):
        for E in list(range(0, 101)) + list(range(143, 256)):
            u = np.uint32((sign << 31) | (E << 23)) | frac
            ours = oracle.f32_to_f16_bits(u.view(np.float32))
            if E < 101:
                want = np.full_like(ours, sign << 15)
                assert np.array_equal(ours, want), E
            else:
                inf_or_nan = (ours & 0x7C00) == 0x7C00
                assert inf_or_nan.all(), E
                is_nan = (ours & 0x3FF) != 0
                assert np.array_equal(is_nan, (E == 255) & (frac != 0)), E
                assert np.all((ours >> 15) == sign)


def test_f32_to_f16_rounding_cases(oracle_lib):
    """Hand-picked boundaries: ties to even in the normal and subnormal ranges, overflow."""
    cases = {
        1.0 + 2.0 ** -11: 0x3C00,           # tie between 1 and 1+2^-10 -> even (1)
        1.0 + 3 * 2.0 ** -11: 0x3C02,       # tie -> even (1+2^-9)
        65504.0: 0x7BFF,
        65519.99: 0x7BFF,
        65520.0: 0x7C00,                    # tie at the top rounds to inf
        2.0 ** -24: 0x0001,
        2.0 ** -25: 0x0000,                 # tie between 0 and the least subnormal -> 0
        1.5 * 2.0 ** -24: 0x0002,           # tie between 1 and 2 subnormal units -> 2
        2.0 ** -14: 0x0400,
        -0.0: 0x8000,
    }
    for v, want in cases.items():
        got = int(oracle.f32_to_f16_bits(np.array([v], np.float32))[0])
        assert got == want, (v, hex(got), hex(want))
