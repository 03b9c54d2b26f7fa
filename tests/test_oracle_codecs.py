"""Pins of the oracle's number formats against things other than itself:
torch's float8 / bfloat16 casts (library), golden points with citations,
exhaustive tables and brute-force nearest search."""

import os

import numpy as np
import pytest
import torch

from oracle import codecs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden_points():
    pts = []
    with open(os.path.join(GOLDEN, "format_points.txt")) as f:
        for line in f:
            line = line.split("|")[0].strip()
            if not line or line.startswith("#"):
                continue
            fmt, code, val = line.split()
            pts.append((fmt, int(code, 16), float(val)))
    return pts


@pytest.mark.parametrize("fmt,code,val", _golden_points())
def test_golden_format_points(fmt, code, val):
    dec = codecs.e4m3_decode if fmt == "e4m3" else codecs.e2m1_decode
    assert dec(np.array([code]))[0] == val
    enc = codecs.e4m3_encode if fmt == "e4m3" else codecs.e2m1_encode
    if val != 0.0:
        assert int(enc(np.array([val], dtype=np.float32))[0]) == code


def test_e4m3_decode_matches_torch_all_codes():
    ours = codecs.e4m3_decode(np.arange(256, dtype=np.uint8))
    lib = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    nan = np.isnan(lib)
    assert (np.isnan(ours) == nan).all()
    assert set(np.nonzero(nan)[0].tolist()) == {0x7F, 0xFF}
    assert (ours[~nan] == lib[~nan]).all()


def test_e4m3_roundtrip_every_finite_code():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    assert (codecs.e4m3_encode(codecs.e4m3_decode(codes).astype(np.float32)) == codes).all()


def test_e4m3_encode_matches_torch_cast_in_range():
    rng = np.random.default_rng(1)
    v = np.concatenate([
        rng.standard_normal(20000) * 50,
        rng.uniform(-448, 448, 20000),
        rng.standard_normal(20000) * 1e-2,  # subnormal range
    ]).astype(np.float32)
    ours = codecs.e4m3_encode(v)
    lib = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    # torch keeps the sign of values that round to zero as well
    assert (ours == lib).all()


def test_e4m3_encode_ties_to_even_and_saturates():
    table = codecs.e4m3_decode(np.arange(0x7F, dtype=np.uint8))
    mids = ((table[:-1] + table[1:]) / 2).astype(np.float32)
    # every midpoint between neighbours is exact in float32; brute force the tie rule
    got = codecs.e4m3_encode(mids)
    for i, m in enumerate(mids):
        cands = [i, i + 1]
        want = [c for c in cands if c % 2 == 0][0]
        assert got[i] == want, (i, m)
    sat = codecs.e4m3_encode(np.array([449.0, 464.0, 1e6, -500.0, -1e30], dtype=np.float32))
    assert sat.tolist() == [0x7E, 0x7E, 0x7E, 0xFE, 0xFE]


def test_e2m1_is_the_ocp_value_list_and_embeds_in_e4m3():
    vals = codecs.e2m1_decode(np.arange(8, dtype=np.uint8))
    assert vals.tolist() == [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    # Every E2M1 value is an E4M3 value: exponent rebias 1 -> 7, mantissa << 2.
    for n in range(1, 8):
        e, m = n >> 1, n & 1
        if e == 0:
            continue
        e4 = ((e - 1 + 7) << 3) | (m << 2)
        assert codecs.e4m3_decode(np.array([e4]))[0] == vals[n]
    neg = codecs.e2m1_decode(np.arange(8, 16, dtype=np.uint8))
    assert (neg[1:] == -vals[1:]).all()


def test_e2m1_encode_brute_force():
    rng = np.random.default_rng(2)
    v = np.concatenate([rng.uniform(-8, 8, 5000),
                        np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, -0.25, -5.0, 7.0, -100.0])]
                       ).astype(np.float32)
    got = codecs.e2m1_encode(v)
    mags = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    for x, g in zip(v, got):
        a = min(abs(float(x)), 6.0)
        d = [abs(a - m) for m in mags]
        best = min(d)
        cands = [i for i in range(8) if d[i] == best]
        want = cands[0] if len(cands) == 1 else [c for c in cands if c % 2 == 0][0]
        if x < 0:
            want |= 8
        assert g == want, (x, g, want)


def test_bf16_round_matches_torch():
    rng = np.random.default_rng(3)
    v = np.concatenate([rng.standard_normal(50000) * 10, rng.standard_normal(1000) * 1e-30]).astype(np.float32)
    # include exact ties: bf16 value + half a bf16 ulp
    base = codecs.bf16_round(rng.standard_normal(1000)).astype(np.float32)
    ties = (base.view(np.uint32) | np.uint32(0x8000)).view(np.float32)
    v = np.concatenate([v, ties])
    lib = torch.from_numpy(v).to(torch.bfloat16).float().numpy()
    assert (codecs.bf16_round(v) == lib).all()


def test_ue8m0_round_up_against_page_bit_rule():
    rng = np.random.default_rng(4)
    s = np.exp2(rng.uniform(-40, 20, 20000)).astype(np.float32)
    s = np.concatenate([s, np.exp2(np.arange(-30, 20)).astype(np.float32), np.float32([1e-12, 1e-10])])
    ours = codecs.ue8m0_round_up(s)
    # The pages' rule: bits of max(s, 1e-10); exponent field plus one if any
    # mantissa bit is set, shifted back into place.
    b = np.maximum(s, np.float32(1e-10)).view(np.uint32)
    e = (b >> 23) + ((b & 0x7FFFFF) != 0).astype(np.uint32)
    page = (e << 23).view(np.float32)
    assert (ours == page).all()
    assert (ours >= np.maximum(s, np.float32(1e-10))).all()
    assert (ours < 2 * np.maximum(s, np.float32(1e-10))).all()


def test_fp4_unpack_nibble_order():
    packed = np.array([[0x21, 0xF7]], dtype=np.uint8)
    assert codecs.fp4_unpack(packed, 4).tolist() == [[0x1, 0x2, 0x7, 0xF]]
