"""Parity criteria between the CUDA path and the oracle.

Routed FP8 (stated accuracy target): ids bit-exact; weights within 1e-6
relative; per route row max-abs error <= 0.02 x the oracle row's RMS; at least
99.9% of elements within 2 BF16 ulp of the oracle value (ulp taken at the
oracle value). The same output criteria are applied to the shared expert and
the NVFP4 layer.

Rounding ties. The outputs are BF16 roundings of FP32 sums. Where the exact
value sits within FP32 summation noise of the midpoint between two BF16
values, a kernel that sums in another order may round to the other neighbour:
one BF16 ulp, which for an element above about 2.6 x the row RMS exceeds
0.02 x RMS although both sides are correct. Given the oracle's unrounded
values, such one-ulp tie flips (exact value within TIE_REL x max(|exact|, row
RMS) of the midpoint) are left out of the row max; they still count in the
2-ulp fraction.
"""

import numpy as np

ROW_RMS_FRAC = 0.02
ULP_FRAC = 0.999
ULPS = 2.0
WEIGHT_RTOL = 1e-6
TIE_REL = 2.0**-18


def bf16_ulp(v):
    """BF16 ulp at |v| (8 significant bits); subnormal spacing near zero."""
    a = np.abs(np.asarray(v, dtype=np.float64))
    e = np.floor(np.log2(np.maximum(a, 2.0**-126)))
    return np.exp2(e - 7)


def tie_flips(got, ref, exact, rms):
    """Elements where got and ref are neighbouring BF16 values and the exact
    value lies within TIE_REL x max(|exact|, rms) of their midpoint."""
    got, ref, exact = (np.asarray(v, dtype=np.float64) for v in (got, ref, exact))
    lo, hi = np.minimum(got, ref), np.maximum(got, ref)
    neighbours = (hi > lo) & (hi - lo <= np.minimum(bf16_ulp(lo), bf16_ulp(hi)) * 1.0000001)
    near = np.abs(exact - 0.5 * (lo + hi)) <= TIE_REL * np.maximum(np.abs(exact), rms[..., None])
    return neighbours & near


def output_report(got, ref, exact=None):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    err = np.abs(got - ref)
    within = err <= ULPS * bf16_ulp(ref)
    rms = np.sqrt(np.mean(ref**2, axis=-1))
    ties = np.zeros(err.shape, dtype=bool) if exact is None else tie_flips(got, ref, exact, rms)
    row_ratio = np.where(ties, 0.0, err).max(axis=-1) / np.maximum(rms, 1e-30)
    return {"frac_within_2ulp": float(within.mean()), "worst_row_maxerr_over_rms": float(row_ratio.max()),
            "max_abs_err": float(err.max()), "n": int(err.size), "tie_flips": int(ties.sum())}


def assert_outputs(got, ref, what="out", exact=None):
    r = output_report(got, ref, exact)
    assert np.isfinite(np.asarray(got, dtype=np.float64)).all(), f"{what}: non-finite values"
    assert r["frac_within_2ulp"] >= ULP_FRAC, f"{what}: {r}"
    assert r["worst_row_maxerr_over_rms"] <= ROW_RMS_FRAC, f"{what}: {r}"
    return r


GAP_ULPS = 4  # near-tie excuse of the routing comparison, in float32 ulps of the keys


def decisive_gap_ulps(keys, ids):
    """Per token, the smallest gap that decides its picks or their order (between
    consecutive picked keys, and between the k-th pick and the best unpicked
    key), in float32 ulps at the larger key of each pair, from the oracle's
    float32 keys [M, E] and ids [M, k]."""
    keys = np.asarray(keys, dtype=np.float32)
    ids = np.asarray(ids)
    M, E = keys.shape
    out = np.full(M, np.inf)
    for t in range(M):
        ordered = [keys[t, int(e)] for e in ids[t]]
        picked = set(int(e) for e in ids[t])
        rest = [keys[t, e] for e in range(E) if e not in picked]
        pairs = list(zip(ordered, ordered[1:]))
        if rest:
            pairs.append((min(ordered), max(rest)))
        for a, b in pairs:
            ulp = float(np.spacing(np.float32(max(abs(a), abs(b)))))
            out[t] = min(out[t], (float(a) - float(b)) / ulp)
    return out


def assert_routing(ids, weights, ref_ids, ref_weights, keys=None, max_ulps=GAP_ULPS):
    """ids must match the oracle's exactly. The one excuse: a token whose
    decisive key gap (decisive_gap_ulps, from the oracle's keys) is below
    `max_ulps` float32 ulps, where the kernel's sigmoid (CUDA expf, IEEE add
    and divide) and the oracle's correctly rounded one may order two keys
    differently; such a token must still pick the same set up to the one
    swapped boundary pick. Weights at matching picks are within 1e-6 relative.
    Returns the number of excused tokens (also printed when non-zero)."""
    ids, ref_ids = np.asarray(ids), np.asarray(ref_ids)
    gaps = None if keys is None else decisive_gap_ulps(keys, ref_ids)
    excused = 0
    for t in range(ids.shape[0]):
        if gaps is not None and gaps[t] < max_ulps:
            excused += 1
            assert len(set(ids[t].tolist()) ^ set(ref_ids[t].tolist())) <= 2, f"token {t}"
            continue
        assert (ids[t] == ref_ids[t]).all(), f"token {t}: {ids[t]} vs {ref_ids[t]}"
    w, rw = np.asarray(weights, np.float64), np.asarray(ref_weights, np.float64)
    same = ids == ref_ids
    assert np.all(np.abs(w - rw)[same] <= WEIGHT_RTOL * np.abs(rw)[same] + 1e-30), \
        f"weights: max rel err {np.max(np.abs(w - rw)[same] / np.abs(rw)[same])}"
    if excused:
        print(f"routing: {excused} of {ids.shape[0]} tokens excused (decisive key gap < {max_ulps} ulp)")
    return excused
