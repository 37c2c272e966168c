"""GPU parity of the codec entry points (kivi_quant_keys, kivi_quant_values):
codes, scales and zeros bit-exact against the oracle."""
import numpy as np
import pytest
import torch

import bit_asymmetric_kv_kivi_gb300 as kivi
import oracle
from gpu_util import configs, dev_tensor, host_bits
from synth import to_dtype_bits
from test_oracle_codec import planted_codes

pytestmark = pytest.mark.gpu


def structured(rng, S, T, D, dtype):
    x = rng.standard_normal((S, T, D))
    x[:, :, rng.choice(D, max(1, D // 32), replace=False)] *= 20.0
    x[:, rng.random(T) < 0.05, :] *= 10.0
    x[0, :3, :] = 0.0                       # exact zeros
    x[-1, 5, :] = 1.5                       # a constant value row (value groups with s = 0)
    return to_dtype_bits(x, dtype)


# (G, D): every slice width of each group size (D a multiple of G)
GD_KEYS = [(32, D) for D in (32, 64, 96, 128, 160, 192, 256)] + [(64, D) for D in (64, 128, 192, 256)]


@pytest.mark.parametrize("bits", [2, 4])
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("G,D", GD_KEYS)
def test_quant_keys_bitexact(bits, dtype, G, D):
    rng = np.random.default_rng(100 + bits + D + G)
    S, T = 3, 5 * G
    kcfg, ocfg = configs(bits, dtype, 1, 1, D, G=G)
    xb = structured(rng, S, T, D, dtype)
    xb[1, G:2 * G, :] = xb[1, G, :]         # a group of identical tokens: every channel constant
    codes, scale, zero = kivi.quant_keys(kcfg, dev_tensor(xb, dtype))
    rc, rs, rz = oracle.quant_keys(ocfg, xb)
    np.testing.assert_array_equal(codes.cpu().numpy(), rc)
    np.testing.assert_array_equal(host_bits(scale), rs)
    np.testing.assert_array_equal(host_bits(zero), rz)


@pytest.mark.parametrize("bits", [2, 4])
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("G,D,T", [(32, 32, 1), (32, 64, 45), (32, 96, 70), (32, 128, 97), (32, 192, 32),
                                   (32, 224, 5), (32, 256, 33), (64, 64, 3), (64, 128, 97), (64, 192, 40),
                                   (64, 256, 65)])
def test_quant_values_bitexact(bits, dtype, G, D, T):
    rng = np.random.default_rng(200 + bits + D + G)
    S = 4
    kcfg, ocfg = configs(bits, dtype, 1, 1, D, G=G)
    xb = structured(rng, S, max(T, 6), D, dtype)[:, :T].copy()
    codes, scale, zero = kivi.quant_values(kcfg, dev_tensor(xb, dtype))
    rc, rs, rz = oracle.quant_values(ocfg, xb)
    np.testing.assert_array_equal(codes.cpu().numpy(), rc)
    np.testing.assert_array_equal(host_bits(scale), rs)
    np.testing.assert_array_equal(host_bits(zero), rz)


@pytest.mark.parametrize("bits", [2, 4])
def test_planted_grid_recovered_exactly(bits):
    """x = z + c*s on exact grids: the kernel must return (c, s, z) themselves."""
    rng = np.random.default_rng(300 + bits)
    S, T, D, G = 2, 64, 128, 32
    qmax = (1 << bits) - 1
    kcfg, _ = configs(bits, "f16", 1, 1, D)
    s = np.ldexp(1.0, rng.integers(-6, 3, size=(S, T // G, D)))
    z = rng.integers(-48, 48, size=s.shape) * s
    c = planted_codes(rng, (S, T // G, G, D), qmax, axis=2).reshape(S, T, D)
    x = np.repeat(z, G, axis=1) + c * np.repeat(s, G, axis=1)
    codes, scale, zero = kivi.quant_keys(kcfg, dev_tensor(to_dtype_bits(x, "f16"), "f16"))
    d = np.arange(D)
    got_c = (codes.cpu().numpy()[..., (d * bits) // 8].astype(np.int64) >> ((d * bits) % 8)) & qmax
    np.testing.assert_array_equal(got_c, c)
    np.testing.assert_array_equal(host_bits(scale).view(np.float16).astype(np.float64), s)
    np.testing.assert_array_equal(host_bits(zero).view(np.float16).astype(np.float64), z)


def test_empty_inputs_are_noops():
    kcfg, _ = configs(2, "f16", 1, 1, 128)
    x = torch.empty((0, 32, 128), dtype=torch.float16, device="cuda")
    codes, scale, zero = kivi.quant_keys(kcfg, x)
    assert codes.numel() == 0
    x = torch.empty((2, 0, 128), dtype=torch.float16, device="cuda")
    codes, scale, zero = kivi.quant_values(kcfg, x)
    assert codes.numel() == 0


@pytest.mark.parametrize("bits", [2, 4])
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("G", [32, 64])
def test_exact_ties_take_the_exact_division(bits, dtype, G):
    """Values exactly half-way between two grid points (x = z + (c + 1/2) s) must round
    half to even like the oracle: the kernels divide exactly near such ties."""
    rng = np.random.default_rng(400 + bits + G)
    S, T, D = 2, 2 * G, 128
    qmax = (1 << bits) - 1
    kcfg, ocfg = configs(bits, dtype, 1, 1, D, G=G)
    s = np.ldexp(1.0, rng.integers(-4, 2, size=(S, T // G, D)))
    z = rng.integers(-20, 20, size=s.shape) * s
    c = rng.integers(0, qmax, size=(S, T, D)) + 0.5 * (rng.random((S, T, D)) < 0.5)
    c[:, ::G, :] = 0                          # every group keeps its min at z ...
    c[:, 1::G, :] = qmax                      # ... and its max at z + qmax s
    x = np.repeat(z, G, axis=1) + c * np.repeat(s, G, axis=1)
    xb = to_dtype_bits(x, dtype)
    codes, scale, zero = kivi.quant_keys(kcfg, dev_tensor(xb, dtype))
    rc, rs, rz = oracle.quant_keys(ocfg, xb)
    np.testing.assert_array_equal(codes.cpu().numpy(), rc)
    np.testing.assert_array_equal(host_bits(scale), rs)
    xv = np.transpose(x.reshape(S, T // G, G, D), (0, 1, 3, 2)).reshape(S, T, D)   # ties along channels too
    xvb = to_dtype_bits(xv, dtype)
    codes, scale, zero = kivi.quant_values(kcfg, dev_tensor(xvb, dtype))
    rc, rs, rz = oracle.quant_values(ocfg, xvb)
    np.testing.assert_array_equal(codes.cpu().numpy(), rc)
    np.testing.assert_array_equal(host_bits(scale), rs)


@pytest.mark.parametrize("bits", [2, 4])
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("G,D", [(32, 32), (32, 64), (32, 96), (32, 128), (32, 192), (32, 256), (64, 64), (64, 128)])
def test_signed_zero_extremes_bitexact(bits, dtype, G, D):
    """Groups whose minimum or maximum is a zero of either sign, at every channel-slice
    width: the stored zero must follow the first zero seen, like the oracle."""
    rng = np.random.default_rng(500 + bits + D + G)
    S, T = 2, 3 * G
    kcfg, ocfg = configs(bits, dtype, 1, 1, D, G=G)
    x = np.abs(rng.standard_normal((S, T, D))) + 0.25
    x[:, G:2 * G] *= -1.0                                       # middle group: maximum is a zero
    zeros = rng.random((S, T, D)) < 0.15
    x[zeros] = np.where(rng.random(zeros.sum()) < 0.5, 0.0, -0.0)
    x[1, 2 * G:, : D // 2] = np.where(rng.random((G, D // 2)) < 0.5, 0.0, -0.0)   # all-zero groups
    xb = to_dtype_bits(x, dtype)
    assert np.any(xb == 0x8000)
    codes, scale, zero = kivi.quant_keys(kcfg, dev_tensor(xb, dtype))
    rc, rs, rz = oracle.quant_keys(ocfg, xb)
    np.testing.assert_array_equal(host_bits(zero), rz)
    np.testing.assert_array_equal(host_bits(scale), rs)
    np.testing.assert_array_equal(codes.cpu().numpy(), rc)
    codes, scale, zero = kivi.quant_values(kcfg, dev_tensor(xb, dtype))
    rc, rs, rz = oracle.quant_values(ocfg, xb)
    np.testing.assert_array_equal(host_bits(zero), rz)
    np.testing.assert_array_equal(host_bits(scale), rs)
    np.testing.assert_array_equal(codes.cpu().numpy(), rc)


@pytest.mark.parametrize("bits", [2, 4])
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("G", [32, 64])
def test_tiny_magnitudes_bitexact(bits, dtype, G):
    """Groups whose scale falls in the fp16 subnormal range (and, for bf16, whose
    minimum does too): the rounded scale and zero can push a group's end codes past
    0 or qmax before the clamp, which the kernels must handle like the oracle."""
    rng = np.random.default_rng(600 + bits + G)
    S, T, D = 3, 2 * G, 128
    kcfg, ocfg = configs(bits, dtype, 1, 1, D, G=G)
    mag = 10.0 ** rng.uniform(-8.5, -4.0, size=(S, T // G, 1, D))
    x = (rng.standard_normal((S, T // G, G, D)) * mag).reshape(S, T, D)
    x[0] += 3e-6                                                    # offset groups: z rounds coarsely
    xb = to_dtype_bits(x, dtype)
    codes, scale, zero = kivi.quant_keys(kcfg, dev_tensor(xb, dtype))
    rc, rs, rz = oracle.quant_keys(ocfg, xb)
    np.testing.assert_array_equal(host_bits(scale), rs)
    np.testing.assert_array_equal(host_bits(zero), rz)
    np.testing.assert_array_equal(codes.cpu().numpy(), rc)
    xv = np.swapaxes(x.reshape(S, T // G, G, D), 2, 3).reshape(S, T, D)   # the same groups along channels
    xvb = to_dtype_bits(xv, dtype)
    codes, scale, zero = kivi.quant_values(kcfg, dev_tensor(xvb, dtype))
    rc, rs, rz = oracle.quant_values(ocfg, xvb)
    np.testing.assert_array_equal(host_bits(scale), rs)
    np.testing.assert_array_equal(host_bits(zero), rz)
    np.testing.assert_array_equal(codes.cpu().numpy(), rc)
