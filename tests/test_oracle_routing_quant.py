"""Pins of the oracle's routing and activation quantisers."""

import numpy as np
import pytest
from scipy.special import expit

from oracle import codecs, quant, routing


def _iterative_topk(keys_row, k):
    """The selection as the mega_moe page describes it: k rounds of 'largest
    key, lowest expert among equals', removing the winner each round."""
    keys = [float(v) for v in keys_row]
    taken = set()
    out = []
    for _ in range(k):
        best = None
        for e, v in enumerate(keys):
            if e in taken:
                continue
            if best is None or v > keys[best]:
                best = e
        taken.add(best)
        out.append(best)
    return out


@pytest.mark.parametrize("M,E,k", [(1, 8, 2), (5, 40, 3), (4, 256, 8), (2, 896, 16)])
def test_route_matches_iterative_selection(M, E, k):
    rng = np.random.default_rng(M * 1000 + E)
    logits = rng.standard_normal((M, E)).astype(np.float32)
    bias = (rng.standard_normal(E) * 0.1).astype(np.float32)
    ids, w, keys = routing.route(logits, bias, k, 2.5)
    for t in range(M):
        assert ids[t].tolist() == _iterative_topk(keys[t], k)


def test_sigmoid_matches_scipy():
    x = np.linspace(-30, 30, 10001).astype(np.float32)
    ref = expit(x.astype(np.float64)).astype(np.float32)
    assert (routing.sigmoid_f32(x) == ref).all()


def test_one_hot_logit_is_picked_first():
    rng = np.random.default_rng(7)
    logits = rng.standard_normal((3, 64)).astype(np.float32)
    logits[0, 17] = 12.0
    logits[1, 63] = 12.0
    logits[2, 0] = 12.0
    ids, _, _ = routing.route(logits, np.zeros(64, np.float32), 4, 1.0)
    assert ids[:, 0].tolist() == [17, 63, 0]


def test_weights_sum_to_scale_and_ignore_bias():
    rng = np.random.default_rng(8)
    logits = rng.standard_normal((6, 256)).astype(np.float32)
    bias = (rng.standard_normal(256) * 0.05).astype(np.float32)
    ids, w, _ = routing.route(logits, bias, 8, 2.5)
    assert np.allclose(w.sum(axis=1), 2.5, rtol=1e-6, atol=0)
    # Weights depend on the unbiased scores of the picked experts only.
    s = expit(logits.astype(np.float64))
    for t in range(6):
        sc = s[t, ids[t]]
        assert np.allclose(w[t], sc / sc.sum() * 2.5, rtol=1e-6)


def test_ties_go_to_lower_expert():
    logits = np.zeros((2, 40), np.float32)
    ids, w, _ = routing.route(logits, np.zeros(40, np.float32), 5, 1.0)
    assert ids.tolist() == [[0, 1, 2, 3, 4]] * 2
    assert (w == np.float32(np.float32(0.5) / np.float32(2.5))).all()


def test_bias_changes_selection_only():
    rng = np.random.default_rng(9)
    logits = rng.standard_normal((1, 32)).astype(np.float32)
    bias = np.zeros(32, np.float32)
    bias[5] = 100.0  # forces expert 5 in, with its own small score
    ids, w, _ = routing.route(logits, bias, 3, 1.0)
    assert ids[0, 0] == 5
    s = expit(logits[0].astype(np.float64))
    assert np.isclose(w[0, 0], s[5] / s[ids[0]].sum(), rtol=1e-6)


def test_expert_permutation_invariance():
    rng = np.random.default_rng(10)
    E = 48
    logits = rng.standard_normal((3, E)).astype(np.float32)
    bias = (rng.standard_normal(E) * 0.1).astype(np.float32)
    perm = rng.permutation(E)
    ids, w, _ = routing.route(logits, bias, 4, 2.0)
    ids_p, w_p, _ = routing.route(logits[:, perm], bias[perm], 4, 2.0)
    assert (perm[ids_p] == ids).all()
    assert (w_p == w).all()


# ------------------------------------------------------------------- FP8 quant
def test_one_hot_block_quantises_to_fp8_max():
    x = np.zeros((1, 256), np.float32)
    x[0, 5] = -3.0
    x[0, 200] = 0.125
    codes, s = quant.fp8_quant_mul(x, ue8m0=False)
    assert codes[0, 5] == 0xFE and codes[0, 200] == 0x7E
    assert (np.delete(codes[0], [5, 200]) == 0).all()
    assert s[0, 0] == np.float32(3.0) / np.float32(448.0)
    assert s[0, 1] == np.float32(0.125) / np.float32(448.0)


def test_zero_block_scale_floor():
    x = np.zeros((1, 128), np.float32)
    c, s = quant.fp8_quant_mul(x, ue8m0=False)
    assert (c == 0).all() and s[0, 0] == np.float32(1e-10) / np.float32(448.0)
    c, s = quant.fp8_quant_mul(x, ue8m0=True)
    # max(1e-10/448, 1e-10) = 1e-10, rounded up to a power of two: 2^-33
    assert s[0, 0] == np.float32(2.0**-33)


def test_fp8_quant_error_is_half_ulp():
    rng = np.random.default_rng(11)
    x = (rng.standard_normal((4, 1024)) * rng.uniform(0.01, 100, (4, 1))).astype(np.float32)
    for ue in (False, True):
        codes, s = quant.fp8_quant_mul(x, ue)
        deq = codecs.e4m3_decode(codes).reshape(4, 8, 128)
        target = x.reshape(4, 8, 128) / s[..., None].astype(np.float64)
        table = codecs.e4m3_decode(np.arange(0x7F, dtype=np.uint8))
        a = np.abs(target)
        hi = np.searchsorted(table, a)
        gap = table[np.minimum(hi, 126)] - table[np.maximum(hi - 1, 0)]
        assert (np.abs(deq - target) <= gap / 2 + 1e-6 * a + 1e-30).all()
        assert (np.abs(deq) <= 448).all()


def test_ue8m0_scales_are_powers_of_two_and_div_equals_mul():
    rng = np.random.default_rng(12)
    x = (rng.standard_normal((3, 512)) * 7).astype(np.float32)
    c1, s1 = quant.fp8_quant_mul(x, True)
    c2, s2 = quant.fp8_quant_div(x, True)
    m, _ = np.frexp(s1)
    assert (m == 0.5).all()
    assert (c1 == c2).all() and (s1 == s2).all()
    _, s0 = quant.fp8_quant_mul(x, False)
    assert (s1 >= s0).all() and (s1 < 2 * s0).all()


# ------------------------------------------------------------------- NVFP4 quant
def test_nvfp4_one_hot_and_sign():
    x = np.zeros((1, 32), np.float32)
    x[0, 3] = 6.0
    x[0, 4] = -3.0
    x[0, 20] = -0.75
    nib, sb = quant.nvfp4_quant(x)
    assert sb[0, 0] == 0x38  # 6/6 = 1.0
    assert nib[0, 3] == 0x7 and nib[0, 4] == 0xD  # 6 and -3: negatives survive (Bug A)
    # second group: amax 0.75 -> scale e4m3(0.125) = 0x28; -0.75/0.125 = -6
    assert codecs.e4m3_decode(sb[0, 1:2])[0] == 0.125
    assert nib[0, 20] == 0xF


def test_nvfp4_stored_scale_is_divisor_and_zero_groups():
    rng = np.random.default_rng(13)
    x = (rng.standard_normal((2, 64)) * 3).astype(np.float32)
    x[1, 16:32] = 0.0
    nib, sb = quant.nvfp4_quant(x)
    d = codecs.e4m3_decode(sb)
    amax = np.abs(x.reshape(2, 4, 16)).max(-1)
    # stored scale ~ amax / 6 (E4M3 relative spacing 1/8), never amax itself (Bug B)
    nz = amax > 0
    assert np.all(np.abs(d[nz] * 6 / amax[nz] - 1) <= 1 / 16 + 1e-9)
    assert (nib[1, 16:32] == 0).all() and d[1, 1] == 0
    deq = codecs.e2m1_decode(nib).reshape(2, 4, 16) * d[..., None]
    assert np.all(np.abs(deq).max(-1) <= 6 * d + 1e-12)


# ------------------------------------------------------------------- exact divide quantiser
def _f32_round(q):
    """Nearest float32 to the rational q, ties to the even significand
    (subnormals included, no overflow handling needed here)."""
    from fractions import Fraction
    q = Fraction(q)
    if q == 0:
        return Fraction(0)
    a = abs(q)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    ulp = Fraction(2) ** max(e - 23, -149)
    n = round(a / ulp)  # Fraction.__round__: half to even
    v = n * ulp
    return v if q > 0 else -v


def _e4m3_code_exact(q):
    """E4M3 byte of the rational q: nearest finite magnitude by brute force over
    the 127 non-negative codes, ties to the even code, saturating at 448."""
    from fractions import Fraction
    mags = [Fraction(codecs.e4m3_value(c)) for c in range(0x7F)]
    a = abs(Fraction(q))
    if a >= mags[-1]:
        c = 0x7E
    else:
        best = None
        for c0 in range(0x7F):
            d = abs(mags[c0] - a)
            if best is None or d < best[0] or (d == best[0] and c0 % 2 == 0):
                best = (d, c0)
        c = best[1]
    return c | 0x80 if q < 0 else c


def test_quant_div_is_an_ieee_divide_not_an_inverse_multiply():
    """"mega_moe" ``hidden_block`` quantises the routed hidden by dividing by its
    scale (``act / scale``). With a non-power-of-two scale (ue8m0 False) the
    float32 quotient h / sh can differ from h * float32(1 / sh); the values below
    are picked where the two land on different sides of an E4M3 rounding
    midpoint, so an oracle quantising by the inverse fails this exact check."""
    from fractions import Fraction
    amax = np.float32(300.0)
    sh = _f32_round(Fraction(float(amax)) / 448)  # float32(max(amax, 1e-10) / 448)
    inv = np.float32(1.0) / np.float32(float(sh))
    mags = [Fraction(codecs.e4m3_value(c)) for c in range(0x7F)]
    mids = [(mags[i] + mags[i + 1]) / 2 for i in range(40, 120)]
    picked = []
    for m in mids:
        centre = np.float32(float(m * sh))
        h = centre
        for _ in range(6):  # a few float32 steps either side of m * sh
            h = np.nextafter(h, np.float32(-np.inf), dtype=np.float32)
        for _ in range(13):
            div = _e4m3_code_exact(_f32_round(Fraction(float(h)) / sh))
            mul = _e4m3_code_exact(Fraction(float(np.float32(h * inv))))
            if div != mul:
                picked.append(float(h))
                break
            h = np.nextafter(h, np.float32(np.inf), dtype=np.float32)
        if len(picked) >= 8:
            break
    assert len(picked) >= 4, "no discriminating values found"
    block = np.zeros(128, np.float32)
    block[0] = amax
    block[1:1 + len(picked)] = picked
    block[64:64 + len(picked)] = -np.asarray(picked, np.float32)
    codes, scale = quant.fp8_quant_div(block[None, :], False)
    assert Fraction(float(scale[0, 0])) == sh
    want = [_e4m3_code_exact(_f32_round(Fraction(float(v)) / sh)) for v in block]
    assert codes[0].tolist() == want
    # and the same block quantised by the inverse differs (the check can fail)
    codes_mul, _ = quant.fp8_quant_mul(block[None, :], False)
    assert (codes_mul[0] != codes[0]).sum() >= len(picked)
