"""Pins of the oracle's GEMMs and whole layers: a dense dequantised reference,
exact brute force with Fractions on tiny shapes, one-hot block scales,
constant scales, and invariances."""

from fractions import Fraction

import numpy as np
import pytest
from scipy.special import expit

from oracle import codecs, moe_fp8, moe_nvfp4, quant, routing


def _fp8_codes(rng, shape):
    """Random finite E4M3 bytes (any code but the NaNs)."""
    c = rng.integers(0, 256, size=shape, dtype=np.uint8)
    return np.where((c & 0x7F) == 0x7F, c ^ 0x01, c).astype(np.uint8)


def _normalish_codes(rng, shape):
    return codecs.e4m3_encode(rng.standard_normal(shape).astype(np.float32))


def _scales(rng, shape, lo=-10, hi=-6):
    return np.exp2(rng.uniform(lo, hi, shape)).astype(np.float32)


# ------------------------------------------------------------------- GEMM pins
def test_block_gemv_equals_dense_dequantised_matmul():
    rng = np.random.default_rng(20)
    N, K = 384, 640
    W = _fp8_codes(rng, (N, K))
    ws = _scales(rng, (N // 128, K // 128))
    a = _fp8_codes(rng, K)
    sa = _scales(rng, K // 128, -3, 3)
    y = moe_fp8.block_scaled_gemv(W, ws, a, sa)
    Wd = codecs.e4m3_decode(W) * np.repeat(np.repeat(ws.astype(np.float64), 128, 0), 128, 1)
    ad = codecs.e4m3_decode(a) * np.repeat(sa.astype(np.float64), 128)
    dense = Wd @ ad
    mag = np.abs(Wd) @ np.abs(ad)
    # Same sum in another order; the only difference is the float32 rounding
    # of each (w_scale * a_scale) product.
    assert np.all(np.abs(y - dense) <= 1e-6 * mag)


def test_block_gemv_constant_scales_exact_brute_force():
    rng = np.random.default_rng(21)
    N, K = 8, 256
    W = _fp8_codes(rng, (N, K))
    a = _fp8_codes(rng, K)
    y = moe_fp8.block_scaled_gemv(W, np.ones((1, 2), np.float32), a, np.ones(2, np.float32))
    for n in range(N):
        exact = sum(Fraction(float(codecs.e4m3_value(W[n, k]))) * Fraction(float(codecs.e4m3_value(a[k])))
                    for k in range(K))
        assert Fraction(float(y[n])) == exact


def test_one_hot_block_scale_changes_only_its_block():
    rng = np.random.default_rng(22)
    N, K = 256, 384
    W = _normalish_codes(rng, (N, K))
    ws = _scales(rng, (2, 3))
    a = _normalish_codes(rng, K)
    sa = _scales(rng, 3, -3, 0)
    y0 = moe_fp8.block_scaled_gemv(W, ws, a, sa)
    ws2 = ws.copy()
    ws2[1, 2] *= 2
    y1 = moe_fp8.block_scaled_gemv(W, ws2, a, sa)
    assert (y1[:128] == y0[:128]).all()
    # rows 128..255 gain exactly their block-2 contribution once more
    for n in range(128, 256, 17):
        blk = sum(Fraction(float(codecs.e4m3_value(W[n, k]))) * Fraction(float(codecs.e4m3_value(a[k])))
                  for k in range(256, 384))
        contrib = float(blk * Fraction(float(np.float32(ws[1, 2] * sa[2]))))
        assert np.isclose(y1[n] - y0[n], contrib, rtol=1e-12, atol=1e-300)


def test_swiglu_closed_forms():
    g = np.array([-30.0, -1.0, 0.0, 0.5, 3.0, 10.0])
    u = np.array([2.0, -9.0, 5.0, 0.25, 8.0, -8.0])
    ref = g * expit(g) * u
    assert np.allclose(moe_fp8.clamped_swiglu(g, u, np.inf), ref, rtol=1e-15)
    L = 7.0
    got = moe_fp8.clamped_swiglu(g, u, L)
    gc = np.minimum(g, L)
    uc = np.clip(u, -L, L)
    assert np.allclose(got, gc * expit(gc) * uc, rtol=1e-15)
    assert got[-1] == pytest.approx(7.0 * expit(7.0) * -7.0)


# ------------------------------------------------------------------- routed layer
def _tiny_routed(rng, M=2, E=8, H=256, I=128):
    w13 = _normalish_codes(rng, (E, 2 * I, H))
    s13 = _scales(rng, (E, 2 * I // 128, H // 128))
    w2 = _normalish_codes(rng, (E, H, I))
    s2 = _scales(rng, (E, H // 128, I // 128))
    x = codecs.bf16_round(rng.standard_normal((M, H)))
    logits = rng.standard_normal((M, E)).astype(np.float32)
    bias = (rng.standard_normal(E) * 0.1).astype(np.float32)
    return x, logits, bias, w13, s13, w2, s2


def _brute_gemv(W, ws, a, sa):
    """Exact sum over blocks of Fraction partials times float32 scale products."""
    N, K = W.shape
    out = []
    for n in range(N):
        acc = Fraction(0)
        for b in range(K // 128):
            part = sum(Fraction(codecs.e4m3_value(W[n, k])) * Fraction(codecs.e4m3_value(a[k]))
                       for k in range(b * 128, (b + 1) * 128))
            acc += part * Fraction(float(np.float32(ws[n // 128, b] * sa[b])))
        out.append(float(acc))
    return np.array(out)


@pytest.mark.parametrize("ue8m0", [False, True])
def test_routed_layer_brute_force_tiny(ue8m0):
    rng = np.random.default_rng(23 + ue8m0)
    M, E, H, I, k = 2, 8, 256, 128, 2
    x, logits, bias, w13, s13, w2, s2 = _tiny_routed(rng, M, E, H, I)
    out, ids, w, _ = moe_fp8.routed_fp8(x, logits, bias, w13, s13, w2, s2, k, 7.0, 2.5, ue8m0)
    xq, sx = quant.fp8_quant_mul(x, ue8m0)
    for t in range(M):
        for r in range(k):
            e = ids[t, r]
            y = _brute_gemv(w13[e], s13[e], xq[t], sx[t]).astype(np.float32)
            up, gate = y[:I], y[I:]  # W31: up rows first, then gate rows
            g = np.minimum(gate.astype(np.float64), 7.0)
            uu = np.clip(up.astype(np.float64), -7.0, 7.0)
            h = (g * expit(g) * uu).astype(np.float32)
            qh, sh = quant.fp8_quant_div(h, ue8m0)
            ref = codecs.bf16_round(_brute_gemv(w2[e], s2[e], qh, sh))
            got = out[t * k + r]
            # Brute force and oracle agree up to the float32 rounding of the
            # GEMM1 sums (silu evaluated by another library): allow 1 BF16 ulp.
            ulp = np.abs(ref).astype(np.float64) * 2.0**-7 + 1e-30
            assert np.all(np.abs(got - ref) <= ulp), (t, r)


def test_routed_gate_up_row_order():
    """Gate rows forced very negative make silu(gate) ~ 0, so the output
    vanishes only if the oracle reads gate from the second half of W31."""
    rng = np.random.default_rng(25)
    M, E, H, I, k = 1, 8, 128, 128, 2
    x, logits, bias, w13, s13, w2, s2 = _tiny_routed(rng, M, E, H, I)
    x[:] = np.abs(x)
    w13[:, :I, :] = codecs.e4m3_encode(np.full((E, I, H), 0.5, np.float32))  # up: positive, big
    w13[:, I:, :] = codecs.e4m3_encode(np.full((E, I, H), -4.0, np.float32))  # gate: very negative
    s13[:] = 1.0
    out, *_ = moe_fp8.routed_fp8(x, logits, bias, w13, s13, w2, s2, k, 1000.0, 1.0, False)
    assert np.all(np.abs(out) < 1e-6 * np.abs(out).max() + 1e-3)


def test_routed_outputs_unweighted_and_identical_tokens():
    rng = np.random.default_rng(26)
    x, logits, bias, w13, s13, w2, s2 = _tiny_routed(rng, 3, 8, 256, 128)
    x[1] = x[0]
    logits[1] = logits[0]
    o1, ids, w1, _ = moe_fp8.routed_fp8(x, logits, bias, w13, s13, w2, s2, 2, 7.0, 1.0, False)
    o2, _, w2_, _ = moe_fp8.routed_fp8(x, logits, bias, w13, s13, w2, s2, 2, 7.0, 4.0, False)
    assert np.array_equal(o1, o2)  # routing weights are not applied to the route rows
    assert np.allclose(w2_, 4 * w1, rtol=1e-6)
    assert np.array_equal(o1[0:2], o1[2:4]) and (ids[0] == ids[1]).all()


def test_routed_sampled_rows_match_full():
    rng = np.random.default_rng(27)
    x, logits, bias, w13, s13, w2, s2 = _tiny_routed(rng, 2, 8, 384, 256)
    full, *_ = moe_fp8.routed_fp8(x, logits, bias, w13, s13, w2, s2, 2, 7.0, 2.5, False)
    rows = np.array([0, 5, 130, 383])
    part, *_ = moe_fp8.routed_fp8(x, logits, bias, w13, s13, w2, s2, 2, 7.0, 2.5, False,
                                  routes=[1, 2], rows=rows)
    assert np.array_equal(part[[1, 2]][:, rows], full[[1, 2]][:, rows])
    assert np.isnan(part[0]).all()


# ------------------------------------------------------------------- shared expert
def test_shared_expert_brute_force_tiny():
    rng = np.random.default_rng(28)
    M, H, I = 2, 256, 128
    w13 = _normalish_codes(rng, (2 * I, H))
    s13 = np.exp2(rng.integers(-10, -5, (2, 2))).astype(np.float32)
    w2 = _normalish_codes(rng, (H, I))
    s2 = np.exp2(rng.integers(-10, -5, (2, 1))).astype(np.float32)
    x = codecs.bf16_round(rng.standard_normal((M, H)))
    out, gu = moe_fp8.shared_fp8(x, w13, s13, w2, s2, 7.0, True)
    xq, sx = quant.fp8_quant_mul(x, True)
    for t in range(M):
        g_u = codecs.bf16_round(_brute_gemv(w13, s13, xq[t], sx[t]))
        assert np.array_equal(g_u, gu[t])
        gate, up = g_u[:I], g_u[I:]  # shared expert: gate rows first
        g = np.minimum(gate.astype(np.float64), 7.0)
        h = codecs.bf16_round(g * expit(g) * np.clip(up, -7.0, 7.0))
        qh, sh = quant.fp8_quant_mul(h, True)
        ref = codecs.bf16_round(_brute_gemv(w2, s2, qh, sh))
        ulp = np.abs(ref).astype(np.float64) * 2.0**-7 + 1e-30
        assert np.all(np.abs(out[t] - ref) <= ulp)


def _golden_ue8m0():
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "ue8m0_packed.txt")
    vals = {}
    for line in open(path):
        if line.startswith("#") or not line.strip():
            continue
        key, *rest = line.split()
        vals[key] = rest
    return [int(v) for v in vals["exponents"]], [float(v) for v in vals["scales"]]


def test_ue8m0_unpack_golden_layout():
    exps, scales = _golden_ue8m0()
    n, k = 128, 1024
    packed = np.zeros((n, k // 512), np.uint32)
    for g, e in enumerate(exps):
        packed[:, g // 4] |= np.uint32(e) << np.uint32(8 * (g % 4))
    got = moe_fp8.ue8m0_unpack(packed.view(np.int32), n, k)
    assert got.shape == (1, 8)
    assert got[0].tolist() == scales
    for e, s in zip(exps, scales):
        assert s == np.ldexp(1.0, e - 127)
    packed[7, 0] ^= np.uint32(1)  # one row of the block disagrees
    with pytest.raises(ValueError):
        moe_fp8.ue8m0_unpack(packed.view(np.int32), n, k)


# ------------------------------------------------------------------- NVFP4
def _nvfp4_weights(rng, L, N2, K, const_scale=False):
    packed = rng.integers(0, 256, size=(L, N2, K // 2), dtype=np.uint8)
    if const_scale:
        sc = np.full((L, N2, K // 16), 0x38, np.uint8)
    else:
        sc = codecs.e4m3_encode(np.exp2(rng.uniform(-8, 0, (L, N2, K // 16))).astype(np.float32))
    return packed, sc


def test_fp4_gemv_constant_scales_exact():
    rng = np.random.default_rng(30)
    N, K = 6, 64
    Wp, Ws = _nvfp4_weights(rng, 1, N, K, const_scale=True)
    a = rng.integers(0, 16, K, dtype=np.uint8)
    y = moe_nvfp4.fp4_block_scaled_gemv(Wp[0], Ws[0], a, np.full(K // 16, 0x38, np.uint8))
    nib = codecs.fp4_unpack(Wp[0], K)
    for n in range(N):
        exact = sum(Fraction(codecs.e2m1_value(nib[n, i])) * Fraction(codecs.e2m1_value(a[i])) for i in range(K))
        assert Fraction(float(y[n])) == exact


def test_fp4_gemv_dense_dequantised():
    rng = np.random.default_rng(31)
    N, K = 64, 256
    Wp, Ws = _nvfp4_weights(rng, 1, N, K)
    a = rng.integers(0, 16, K, dtype=np.uint8)
    sa = codecs.e4m3_encode(np.exp2(rng.uniform(-4, 4, K // 16)).astype(np.float32))
    y = moe_nvfp4.fp4_block_scaled_gemv(Wp[0], Ws[0], a, sa)
    Wd = codecs.e2m1_decode(codecs.fp4_unpack(Wp[0], K)) * np.repeat(codecs.e4m3_decode(Ws[0]), 16, axis=1)
    ad = codecs.e2m1_decode(a) * np.repeat(codecs.e4m3_decode(sa), 16)
    assert np.allclose(y, Wd @ ad, rtol=1e-12, atol=1e-300)


def _nvfp4_case(rng, M=3, k=3, H=64, N=32, L=4, E=12):
    w13, s13 = _nvfp4_weights(rng, L, 2 * N, H)
    w2, s2 = _nvfp4_weights(rng, L, H, N)
    x = codecs.bf16_round(rng.standard_normal((M, H)))
    logits = rng.standard_normal((M, E)).astype(np.float32)
    ids, weights, _ = routing.route(logits, np.zeros(E, np.float32), k, 1.0)
    return x, ids, weights, w13, s13, w2, s2


def test_nvfp4_no_local_routes_is_zero():
    rng = np.random.default_rng(32)
    x, ids, weights, w13, s13, w2, s2 = _nvfp4_case(rng)
    y = moe_nvfp4.routed_nvfp4(x, ids, weights, w13, s13, w2, s2, e0=100, n_local=4)
    assert (y == 0).all()


def test_nvfp4_weights_applied_once():
    rng = np.random.default_rng(33)
    x, ids, weights, w13, s13, w2, s2 = _nvfp4_case(rng, L=12)
    y1 = moe_nvfp4.routed_nvfp4(x, ids, weights, w13, s13, w2, s2, 0, 12)
    y2 = moe_nvfp4.routed_nvfp4(x, ids, 2 * weights, w13, s13, w2, s2, 0, 12)
    assert np.array_equal(y2, 2 * y1)  # linear in the weights: applied exactly once


def test_nvfp4_per_slot_silu_brute_force():
    rng = np.random.default_rng(34)
    M, k, H, N, L = 2, 3, 64, 32, 6
    x, ids, weights, w13, s13, w2, s2 = _nvfp4_case(rng, M, k, H, N, L, E=6)
    y = moe_nvfp4.routed_nvfp4(x, ids, weights, w13, s13, w2, s2, 0, L)
    xq, xs = quant.nvfp4_quant(x)
    for t in range(M):
        acc = np.float32(0) * np.zeros(H, np.float32)
        for r in range(k):
            e = ids[t, r]
            Wd = codecs.e2m1_decode(codecs.fp4_unpack(w13[e], H)) * np.repeat(codecs.e4m3_decode(s13[e]), 16, 1)
            xd = codecs.e2m1_decode(xq[t]) * np.repeat(codecs.e4m3_decode(xs[t]), 16)
            g1 = codecs.bf16_round(Wd @ xd)
            gate, up = g1[:N], g1[N:]  # [gate; up]
            h = codecs.bf16_round(gate * expit(gate.astype(np.float64)) * up)  # SiLU per slot
            hq, hs = quant.nvfp4_quant(h)
            W2d = codecs.e2m1_decode(codecs.fp4_unpack(w2[e], N)) * np.repeat(codecs.e4m3_decode(s2[e]), 16, 1)
            hd = codecs.e2m1_decode(hq) * np.repeat(codecs.e4m3_decode(hs), 16)
            o = codecs.bf16_round(W2d @ hd)
            acc = (acc + (weights[t, r] * o).astype(np.float32)).astype(np.float32)
        assert np.array_equal(y[t], codecs.bf16_round(acc))


def test_mx_gemv_reduces_to_block_gemv_and_matches_dense_dequant():
    from oracle import codecs
    from oracle.moe_fp8 import block_scaled_gemv, mx_block_scaled_gemv
    rng = np.random.default_rng(11)
    N, K = 256, 512
    w = rng.integers(0, 0x7E, size=(N, K), dtype=np.uint8) | (rng.integers(0, 2, size=(N, K), dtype=np.uint8) << 7)
    w[(w & 0x7F) == 0x7F] = 0
    ws = np.exp2(rng.uniform(-12, -6, size=(N // 128, K // 128))).astype(np.float32)
    a = rng.integers(0, 0x7E, size=K, dtype=np.uint8)
    # equal exponents inside each 128-block: the per-128 GEMV with scale 2^(e-127)
    e128 = rng.integers(110, 140, size=K // 128).astype(np.uint8)
    e32 = np.repeat(e128, 4)
    got = mx_block_scaled_gemv(w, ws, a, e32)
    ref = block_scaled_gemv(w, ws, a, np.exp2(e128.astype(np.float64) - 127).astype(np.float32))
    assert np.allclose(got, ref, rtol=1e-12, atol=0)
    # any exponents: the dense dequantised product (power-of-two scales: exact scale products)
    e = rng.integers(100, 150, size=K // 32).astype(np.uint8)
    W = codecs.e4m3_decode(w) * np.repeat(np.repeat(ws.astype(np.float64), 128, 0), 128, 1)
    av = codecs.e4m3_decode(a) * np.repeat(np.exp2(e.astype(np.float64) - 127), 32)
    assert np.allclose(mx_block_scaled_gemv(w, ws, a, e), W @ av, rtol=1e-12, atol=1e-300)


def test_shared_gate_up_row_order():
    """"shared_expert" ``_DownKernel`` reads gates at the row base and ups at
    base + inter, so gate_up rows [0, I) are the gate. Gate rows forced very
    negative make silu(gate) = 0 and the output vanishes; an oracle that took
    gate from the second half would give large outputs."""
    rng = np.random.default_rng(35)
    M, H, I = 2, 256, 128
    x = codecs.bf16_round(np.abs(rng.standard_normal((M, H))) + 0.1)
    w13 = np.empty((2 * I, H), np.uint8)
    w13[:I] = codecs.e4m3_encode(np.full((I, H), -4.0, np.float32))  # gate: very negative
    w13[I:] = codecs.e4m3_encode(np.full((I, H), 0.5, np.float32))  # up: positive
    s13 = np.ones((2, 2), np.float32)
    w2 = _normalish_codes(rng, (H, I))
    s2 = np.ones((2, 1), np.float32)
    out, gu = moe_fp8.shared_fp8(x, w13, s13, w2, s2, 7.0, False)
    assert (gu[:, :I] < -100).all() and (gu[:, I:] > 10).all()
    assert (out == 0).all()
    # the mirror image: gate rows positive, up rows negative -> clamped, non-zero
    out2, _ = moe_fp8.shared_fp8(x, w13[np.r_[I:2 * I, 0:I]], s13, w2, s2, 7.0, False)
    assert np.abs(out2).max() > 1.0


def test_nvfp4_gate_up_row_order():
    """"nvfp4-megamoe-kernel README.md", Bugs Found & Fixed §4: L1 rows are the
    plain concatenation [gate; up]. Gate rows forced very negative make every
    slot's SiLU zero, so y vanishes; reading gate from the second half would
    not."""
    rng = np.random.default_rng(36)
    M, k, H, N, L = 2, 2, 64, 32, 4
    x = codecs.bf16_round(np.abs(rng.standard_normal((M, H))) + 0.5)
    neg4, half = 0xE, 0x1  # E2M1 nibbles of -4.0 and +0.5
    w13 = np.empty((L, 2 * N, H // 2), np.uint8)
    w13[:, :N] = neg4 | (neg4 << 4)
    w13[:, N:] = half | (half << 4)
    s13 = np.full((L, 2 * N, H // 16), 0x38, np.uint8)  # UE4M3 1.0
    w2, s2 = _nvfp4_weights(rng, L, H, N)
    ids = np.array([[0, 1], [2, 3]], np.int32)
    weights = np.full((M, k), 0.5, np.float32)
    y = moe_nvfp4.routed_nvfp4(x, ids, weights, w13, s13, w2, s2, 0, L)
    assert (y == 0).all()
    swapped = w13[:, np.r_[N:2 * N, 0:N]]
    y2 = moe_nvfp4.routed_nvfp4(x, ids, weights, swapped, s13, w2, s2, 0, L)
    assert np.abs(y2).max() > 1.0
