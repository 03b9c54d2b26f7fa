"""Pins of the finalize oracle against closed forms and exact cases."""

import numpy as np

from oracle import codecs
from oracle.finalize import finalize


def _bf16(a):
    return codecs.bf16_round(np.asarray(a, dtype=np.float32))


def test_one_hot_weights_select_the_row():
    rng = np.random.default_rng(1)
    M, k, H = 3, 4, 64
    out = _bf16(rng.normal(size=(M * k, H)))
    for r in range(k):
        w = np.zeros((M, k), np.float32)
        w[:, r] = 1.0
        y = finalize(out, w)
        assert np.array_equal(y, out.reshape(M, k, H)[:, r, :])


def test_zero_weights_give_the_shared_row():
    rng = np.random.default_rng(2)
    M, k, H = 2, 8, 32
    out = _bf16(rng.normal(size=(M * k, H)))
    sh = _bf16(rng.normal(size=(M, H)))
    assert np.array_equal(finalize(out, np.zeros((M, k), np.float32), sh), sh)


def test_power_of_two_scaling_is_exact():
    rng = np.random.default_rng(3)
    M, k, H = 4, 6, 128
    out = _bf16(rng.normal(size=(M * k, H)))
    w = rng.uniform(0.05, 1.0, size=(M, k)).astype(np.float32)
    assert np.array_equal(finalize(out, 2 * w), 2 * finalize(out, w))


def test_matches_exact_sum_within_fp32_bound():
    rng = np.random.default_rng(4)
    M, k, H = 5, 8, 256
    out = _bf16(rng.normal(size=(M * k, H)))
    sh = _bf16(rng.normal(size=(M, H)))
    w = rng.uniform(0.0, 1.0, size=(M, k)).astype(np.float32)
    exact = (w.astype(np.float64)[:, :, None] * out.reshape(M, k, H).astype(np.float64)).sum(1) + sh
    terms = (np.abs(w)[:, :, None] * np.abs(out.reshape(M, k, H))).sum(1) + np.abs(sh)
    # at most 2k + 1 FP32 roundings before the final BF16 rounding (half an ulp of BF16 = 2^-8 relative)
    bound = (2 * k + 1) * 2.0 ** -24 * terms + 2.0 ** -8 * np.abs(exact) + 1e-30
    assert np.all(np.abs(finalize(out, w, sh) - exact) <= bound)


def test_order_is_ascending_route_then_shared():
    # 1 + 2^24 - 2^24 in FP32 depends on the order: ascending r keeps the 1 only
    # if it is added after the cancellation.
    H = 8
    rows = np.array([[2.0 ** 24] * H, [-(2.0 ** 24)] * H, [1.0] * H], np.float32)
    w = np.ones((1, 3), np.float32)
    assert np.all(finalize(rows, w) == 1.0)           # (2^24 - 2^24) + 1
    rows2 = rows[[2, 0, 1]]
    assert np.all(finalize(rows2, w) == 0.0)          # (1 + 2^24) - 2^24: the 1 is lost
    sh = np.full((1, H), 1.0, np.float32)
    assert np.all(finalize(rows2, w, sh) == 1.0)      # shared row added last
