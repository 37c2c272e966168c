"""Pins for the oracle's quantizer and packing (CPU only).

None of these re-types the oracle's formula. They check it against:
  * planted grids: inputs built as x = z + c*s with a power-of-two s, where the
    guide's min/max quantizer ("Step 1" of "KIVI: Asymmetric 2-Bit KV Cache
    Quantization Guide") must give back exactly (c, s, z);
  * brute force: every code is the nearest grid point c*s + z over all
    c in [0, qmax], evaluated in fp64;
  * invariants: codes in range, the error bound, min -> 0, max -> qmax,
    constant groups -> s = 0;
  * the packing rule, unpacked here with independent shift arithmetic.
"""
import numpy as np
import pytest

import oracle
from synth import bits_to_f32, to_dtype_bits

F16, BF16 = oracle.F16, oracle.BF16


def unpack(rows: np.ndarray, bits: int, D: int) -> np.ndarray:
    """Independent unpacker: code of channel d = (row[d*bits//8] >> ((d*bits) % 8)) & (2^bits-1)."""
    d = np.arange(D)
    byte = rows[..., (d * bits) // 8].astype(np.int64)
    return (byte >> ((d * bits) % 8)) & ((1 << bits) - 1)


def f16(bits_u16):
    return np.asarray(bits_u16, np.uint16).view(np.float16).astype(np.float64)


def planted_codes(rng, shape, qmax, axis):
    """Random codes in [0, qmax] where every group along `axis` holds a 0 and a qmax."""
    c = rng.integers(0, qmax + 1, size=shape)
    c = np.moveaxis(c, axis, -1)
    flat = c.reshape(-1, c.shape[-1])
    for row in flat:
        i, j = rng.choice(row.size, 2, replace=False)
        row[i], row[j] = 0, qmax
    return np.moveaxis(flat.reshape(c.shape), -1, axis)


@pytest.mark.parametrize("bits", [2, 4])
@pytest.mark.parametrize("dtype", [F16, BF16])
@pytest.mark.parametrize("G", [32, 64])
def test_planted_grid_keys(oracle_lib, bits, dtype, G):
    rng = np.random.default_rng(10 + bits + 7 * dtype + G)
    S, T, D = 3, 3 * G, 64
    cfg = oracle.Cfg(bits=bits, head_dim=D, dtype=dtype, group=G)
    qmax = (1 << bits) - 1
    # one power-of-two scale and one zero (a multiple of the scale) per (stream, group, channel)
    k = rng.integers(-6, 3, size=(S, T // G, D))
    s = np.ldexp(1.0, k)
    z = rng.integers(-48, 48, size=(S, T // G, D)) * s
    codes = planted_codes(rng, (S, T // G, G, D), qmax, axis=2).reshape(S, T, D)
    x = np.repeat(z, G, axis=1) + codes * np.repeat(s, G, axis=1)
    xb = to_dtype_bits(x, "bf16" if dtype == BF16 else "f16")
    assert np.array_equal(bits_to_f32(xb, "bf16" if dtype == BF16 else "f16").astype(np.float64), x)
    got_codes, got_s, got_z = oracle.quant_keys(cfg, xb)
    assert np.array_equal(unpack(got_codes, bits, D), codes)
    assert np.array_equal(f16(got_s), s)
    assert np.array_equal(f16(got_z), z)


@pytest.mark.parametrize("bits", [2, 4])
@pytest.mark.parametrize("dtype", [F16, BF16])
@pytest.mark.parametrize("G", [32, 64])
def test_planted_grid_values(oracle_lib, bits, dtype, G):
    rng = np.random.default_rng(20 + bits + 7 * dtype + G)
    S, T, D = 2, 40, 128
    cfg = oracle.Cfg(bits=bits, head_dim=D, dtype=dtype, group=G)
    qmax = (1 << bits) - 1
    k = rng.integers(-6, 3, size=(S, T, D // G))
    s = np.ldexp(1.0, k)
    z = rng.integers(-48, 48, size=(S, T, D // G)) * s
    codes = planted_codes(rng, (S, T, D // G, G), qmax, axis=3).reshape(S, T, D)
    x = np.repeat(z, G, axis=2) + codes * np.repeat(s, G, axis=2)
    xb = to_dtype_bits(x, "bf16" if dtype == BF16 else "f16")
    got_codes, got_s, got_z = oracle.quant_values(cfg, xb)
    assert np.array_equal(unpack(got_codes, bits, D), codes)
    assert np.array_equal(f16(got_s), s)
    assert np.array_equal(f16(got_z), z)


def test_round_half_to_even(oracle_lib):
    """x = z + (c + 1/2) s lies exactly between two grid points: the even code wins."""
    D, G = 32, 32
    cfg = oracle.Cfg(bits=2, head_dim=D)
    # one value group of 32 channels per token: min 0, max 3 (s = 1), half-way points in between
    x = np.zeros((1, 1, D))
    x[0, 0, 0], x[0, 0, 1] = 0.0, 3.0
    x[0, 0, 2:] = np.resize([0.5, 1.5, 2.5], D - 2)
    codes, s, z = oracle.quant_values(cfg, to_dtype_bits(x, "f16"))
    c = unpack(codes, 2, D)[0, 0]
    assert f16(s)[0, 0, 0] == 1.0 and f16(z)[0, 0, 0] == 0.0
    want = np.array([0, 3] + list(np.resize([0, 2, 2], D - 2)))
    assert np.array_equal(c, want)


def test_constant_group(oracle_lib):
    cfg = oracle.Cfg(bits=2, head_dim=64)
    x = np.full((1, 32, 64), 1.25)
    x[0, :, 5] = -3.0
    codes, s, z = oracle.quant_keys(cfg, to_dtype_bits(x, "f16"))
    assert np.all(f16(s) == 0.0)
    assert np.array_equal(f16(z)[0, 0], x[0, 0])
    assert np.all(codes == 0)


def _dequant_keys(cfg, codes, s, z):
    G = cfg.group
    c = unpack(codes, cfg.k_bits, cfg.head_dim)
    return c * np.repeat(f16(s), G, axis=1) + np.repeat(f16(z), G, axis=1)


def _structured_inputs(rng, S, T, D, dtype):
    x = rng.standard_normal((S, T, D))
    x[:, :, rng.choice(D, 3, replace=False)] *= 20.0        # outlier channels
    x[:, rng.random(T) < 0.05, :] *= 10.0                    # burst tokens
    name = "bf16" if dtype == BF16 else "f16"
    xb = to_dtype_bits(x, name)
    return xb, bits_to_f32(xb, name).astype(np.float64)


@pytest.mark.parametrize("bits", [2, 4])
@pytest.mark.parametrize("dtype", [F16, BF16])
@pytest.mark.parametrize("G", [32, 64])
def test_keys_brute_force_and_invariants(oracle_lib, bits, dtype, G):
    rng = np.random.default_rng(30 + bits + dtype + G)
    S, T, D = 2, 128, 64
    cfg = oracle.Cfg(bits=bits, head_dim=D, dtype=dtype, group=G)
    qmax = (1 << bits) - 1
    xb, x = _structured_inputs(rng, S, T, D, dtype)
    codes, sb, zb = oracle.quant_keys(cfg, xb)
    c = unpack(codes, bits, D)
    assert c.min() >= 0 and c.max() <= qmax
    s = np.repeat(f16(sb), G, axis=1)
    z = np.repeat(f16(zb), G, axis=1)
    grid = z[..., None] + np.arange(qmax + 1) * s[..., None]          # [S][T][D][qmax+1]
    err = np.abs(x[..., None] - grid)
    chosen = np.take_along_axis(err, c[..., None], axis=-1)[..., 0]
    best = err.min(axis=-1)
    # nearest grid point, up to fp32 rounding of (x - z) / s (a few ulps of the quotient)
    assert np.all(chosen - best <= s * 2.0 ** -20 + 1e-30)
    # error bound: half a step, or the clamp overshoot caused by rounding s and z to fp16
    xg = x.reshape(S, T // G, G, D)
    mn, mx = xg.min(axis=2), xg.max(axis=2)
    over = np.maximum.reduce([f16(zb) - mn, mx - (f16(zb) + qmax * f16(sb)), np.zeros_like(mn)])
    bound = np.maximum(0.5 * f16(sb) * (1 + 2.0 ** -20), over)
    assert np.all(np.abs(x - _dequant_keys(cfg, codes, sb, zb)).reshape(S, T // G, G, D)
                  <= bound[:, :, None, :] + 1e-30)
    # the group minimum gets code 0 and the maximum gets qmax
    cg = c.reshape(S, T // G, G, D)
    am, aM = xg.argmin(axis=2), xg.argmax(axis=2)
    assert np.all(np.take_along_axis(cg, am[:, :, None, :], axis=2) == 0)
    assert np.all(np.take_along_axis(cg, aM[:, :, None, :], axis=2) == qmax)


@pytest.mark.parametrize("bits", [2, 4])
@pytest.mark.parametrize("dtype", [F16, BF16])
@pytest.mark.parametrize("G", [32, 64])
def test_values_brute_force_and_invariants(oracle_lib, bits, dtype, G):
    rng = np.random.default_rng(40 + bits + dtype + G)
    S, T, D = 2, 37, 128
    cfg = oracle.Cfg(bits=bits, head_dim=D, dtype=dtype, group=G)
    qmax = (1 << bits) - 1
    xb, x = _structured_inputs(rng, S, T, D, dtype)
    codes, sb, zb = oracle.quant_values(cfg, xb)
    c = unpack(codes, bits, D)
    s = np.repeat(f16(sb), G, axis=2)
    z = np.repeat(f16(zb), G, axis=2)
    grid = z[..., None] + np.arange(qmax + 1) * s[..., None]
    err = np.abs(x[..., None] - grid)
    chosen = np.take_along_axis(err, c[..., None], axis=-1)[..., 0]
    assert np.all(chosen - err.min(axis=-1) <= s * 2.0 ** -20 + 1e-30)
    xg = x.reshape(S, T, D // G, G)
    cg = c.reshape(S, T, D // G, G)
    assert np.all(np.take_along_axis(cg, xg.argmin(axis=3)[..., None], axis=3) == 0)
    assert np.all(np.take_along_axis(cg, xg.argmax(axis=3)[..., None], axis=3) == qmax)
    # s is the fp16 rounding of (max - min) / qmax, z of the minimum
    assert np.allclose(f16(sb), (xg.max(3) - xg.min(3)) / qmax, rtol=2.0 ** -10, atol=0)
    assert np.allclose(f16(zb), xg.min(3), rtol=2.0 ** -10, atol=2.0 ** -24)


def test_packing_layout_2bit(oracle_lib):
    """Channel d of a row lands in byte d // 4 at bits 2*(d % 4): four 2-bit codes per byte."""
    D = 32
    cfg = oracle.Cfg(bits=2, head_dim=D)
    x = np.zeros((1, 1, D))
    x[0, 0, :] = [0, 3] + [1] * (D - 2)        # min 0, max 3, s = 1
    codes, _, _ = oracle.quant_values(cfg, to_dtype_bits(x, "f16"))
    assert codes.shape == (1, 1, 8)
    # byte 0 holds channels 0..3 = codes (0, 3, 1, 1) -> 0b01_01_11_00
    assert codes[0, 0, 0] == 0b01011100
    assert np.all(codes[0, 0, 1:] == 0b01010101)


@pytest.mark.parametrize("dtype", [F16, BF16])
def test_signed_zero_extreme_takes_first_seen(oracle_lib, dtype):
    """Where a group's minimum (or maximum) is a zero, z (or s) follows the zero seen
    first in scan order: tokens for keys, channels for values (the reading that
    ties keep the first value seen)."""
    name = "bf16" if dtype == BF16 else "f16"
    D = 32
    cfg = oracle.Cfg(bits=2, head_dim=D, dtype=dtype)
    x = np.abs(np.linspace(0.5, 3.0, 32))[:, None] * np.ones((1, D))    # [T=32][D], all > 0
    x[4, :] = -0.0
    x[9, :] = 0.0
    x[4, 1] = 0.0            # channel 1: +0 first (token 4), -0 never
    x[9, 2] = -0.0           # channel 2: -0 at token 4 and token 9
    xb = to_dtype_bits(x[None], name)
    _, _, zb = oracle.quant_keys(cfg, xb)
    zbits = np.asarray(zb, np.uint16)[0, 0]
    assert zbits[0] == 0x8000 and zbits[1] == 0x0000 and zbits[2] == 0x8000
    # values: channel order within a 32-channel group; all <= 0, so the maximum is a zero
    v = -np.abs(np.linspace(0.5, 3.0, 32))[None, :] * np.ones((3, 1))   # [T=3][D]
    v[0, 7], v[0, 20] = 0.0, -0.0
    v[1, 7], v[1, 20] = -0.0, 0.0
    v[2, 3] = -0.0
    vb = to_dtype_bits(v[None], name)
    _, sb, zb = oracle.quant_values(cfg, vb)
    mx_minus_mn = f16(sb)[0, :, 0] * 3
    assert np.allclose(mx_minus_mn, 3.0, rtol=2.0 ** -9)
    # min is -3 in every row; the stored zero is the fp16 of the minimum, the sign of the
    # maximum zero shows only through s, which is the same for either sign
    assert np.all(f16(zb)[0, :, 0] == -3.0)
    # keys again with every token of a channel a zero: the first token's sign wins
    y = np.zeros((32, D))
    y[0, :D // 2] = -0.0
    y[1:, D // 2:] = -0.0
    _, sb, zb = oracle.quant_keys(cfg, to_dtype_bits(y[None], name))
    zbits = np.asarray(zb, np.uint16)[0, 0]
    assert np.all(zbits[:D // 2] == 0x8000) and np.all(zbits[D // 2:] == 0x0000)
    assert np.all(np.asarray(sb, np.uint16) == 0)
