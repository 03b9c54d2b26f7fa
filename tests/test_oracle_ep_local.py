"""Pins of the MXFP8 quantiser and the combine + RMSNorm oracle."""

import math

import numpy as np
import torch

from oracle import codecs
from oracle.ep_local import combine_rmsnorm, mx_exponent, mxfp8_quantize


def test_exponent_closed_form():
    for amax, want in [(1.0, -8), (1.75, -8), (2.0, -7), (448.0, 0), (0.0, -127), (2.0 ** -130, -127),
                       (3.0e38, 119), (0.0009765625, -18)]:
        assert mx_exponent(amax) == want, amax
    rng = np.random.default_rng(0)
    for v in rng.uniform(-30, 30, 200):
        a = 2.0 ** v
        assert mx_exponent(a) == max(-127, min(127, math.floor(math.log2(a)) - 8))


def test_one_hot_block_and_zero_block():
    x = np.zeros((2, 64), np.float32)
    x[0, 5] = -3.0  # floor(log2 3) = 1 -> exponent -7, code of -3 * 2^7 = -384
    codes, scales = mxfp8_quantize(x)
    assert scales[0, 0] == 120 and scales[0, 1] == 0 and scales[1, 0] == 0
    assert codecs.e4m3_decode(codes[0, 5]) == -384.0
    assert (np.delete(codes[0], 5) == 0).all() and (codes[1] == 0).all()


def test_dequantised_error_within_half_ulp_and_saturation():
    rng = np.random.default_rng(1)
    x = codecs.bf16_round(rng.normal(size=(4, 256)).astype(np.float32) * 10)
    codes, scales = mxfp8_quantize(x)
    deq = codecs.e4m3_decode(codes).reshape(4, 8, 32) * np.exp2(scales.astype(np.float64) - 127)[:, :, None]
    xb = x.reshape(4, 8, 32).astype(np.float64)
    # E4M3 keeps 3 mantissa bits: error <= 2^-4 relative (half ulp), except values clamped at 448 * 2^e
    top = 448.0 * np.exp2(scales.astype(np.float64) - 127)[:, :, None]
    ok = np.abs(deq - xb) <= 2.0 ** -4 * np.abs(xb) + 2.0 ** -9 * np.exp2(scales.astype(np.float64) - 127)[:, :, None]
    sat = np.abs(xb) > top
    assert np.all(ok | sat)
    assert np.all(np.abs(deq[sat]) == top[sat.nonzero()[0], sat.nonzero()[1], 0])


def test_matches_torch_float8_for_in_range_values():
    rng = np.random.default_rng(2)
    x = codecs.bf16_round(rng.normal(size=(3, 128)).astype(np.float32))
    codes, scales = mxfp8_quantize(x)
    scaled = torch.from_numpy(x.reshape(3, 4, 32) * np.exp2(-(scales.astype(np.float32) - 127))[:, :, None])
    ref = scaled.clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8).numpy().reshape(3, 128)
    assert np.array_equal(codes, ref)


def test_combine_reduces_in_rank_order_then_normalises():
    H = 64
    big = np.full(H, 2.0 ** 24, np.float32)
    partials = np.stack([np.stack([big, -big, np.ones(H, np.float32)])])  # (2^24 - 2^24) + 1
    latent, normed = combine_rmsnorm(partials, np.ones(H, np.float32))
    assert np.all(latent == 1.0)
    assert np.allclose(normed, codecs.bf16_round(np.full(H, 1.0 / math.sqrt(1.0 + 1e-5))))
    partials2 = partials[:, [2, 0, 1], :]  # (1 + 2^24) - 2^24 loses the 1
    latent2, normed2 = combine_rmsnorm(partials2, np.ones(H, np.float32))
    assert np.all(latent2 == 0.0) and np.all(normed2 == 0.0)


def test_rmsnorm_closed_form():
    rng = np.random.default_rng(3)
    H = 3584
    x = codecs.bf16_round(rng.normal(size=(2, 1, H)).astype(np.float32))
    g = codecs.bf16_round(rng.uniform(0.5, 1.5, H).astype(np.float32))
    latent, normed = combine_rmsnorm(x, g, 1e-5)
    assert np.array_equal(latent, x[:, 0, :])
    r = 1.0 / np.sqrt((x[:, 0, :].astype(np.float64) ** 2).mean(axis=1, keepdims=True) + 1e-5)
    assert np.array_equal(normed, codecs.bf16_round(x[:, 0, :].astype(np.float64) * r * g))
    # scale invariance: 2x the input gives the same normed output (up to eps)
    _, normed2 = combine_rmsnorm(2 * x, g, 0.0)
    _, normed1 = combine_rmsnorm(x, g, 0.0)
    assert np.array_equal(normed1, normed2)
