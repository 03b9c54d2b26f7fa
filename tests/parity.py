"""Parity criteria between the CUDA path and the oracle.

Routed FP8 (stated accuracy target): ids bit-exact; weights within 1e-6
relative; per route row max-abs error <= 0.02 x the oracle row's RMS; at least
99.9% of elements within 2 BF16 ulp of the oracle value (ulp taken at the
oracle value). The same output criteria are applied to the shared expert and
the NVFP4 layer.
"""

import numpy as np

ROW_RMS_FRAC = 0.02
ULP_FRAC = 0.999
ULPS = 2.0
WEIGHT_RTOL = 1e-6


def bf16_ulp(v):
    """BF16 ulp at |v| (8 significant bits); subnormal spacing near zero."""
    a = np.abs(np.asarray(v, dtype=np.float64))
    e = np.floor(np.log2(np.maximum(a, 2.0**-126)))
    return np.exp2(e - 7)


def output_report(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    err = np.abs(got - ref)
    within = err <= ULPS * bf16_ulp(ref)
    rms = np.sqrt(np.mean(ref**2, axis=-1))
    row_ratio = err.max(axis=-1) / np.maximum(rms, 1e-30)
    return {"frac_within_2ulp": float(within.mean()), "worst_row_maxerr_over_rms": float(row_ratio.max()),
            "max_abs_err": float(err.max()), "n": int(err.size)}


def assert_outputs(got, ref, what="out"):
    r = output_report(got, ref)
    assert np.isfinite(np.asarray(got, dtype=np.float64)).all(), f"{what}: non-finite values"
    assert r["frac_within_2ulp"] >= ULP_FRAC, f"{what}: {r}"
    assert r["worst_row_maxerr_over_rms"] <= ROW_RMS_FRAC, f"{what}: {r}"
    return r


def assert_routing(ids, weights, ref_ids, ref_weights, gaps=None, min_gap=1e-6):
    """ids must match exactly except for tokens whose decisive key gap (from the
    oracle, in float32) is below `min_gap`: there a few-ulp sigmoid difference
    may legitimately swap two picks, and only the set/weights are checked."""
    ids, ref_ids = np.asarray(ids), np.asarray(ref_ids)
    for t in range(ids.shape[0]):
        if gaps is not None and gaps[t] < min_gap:
            # a near-tie may swap at most the boundary pick
            assert len(set(ids[t].tolist()) ^ set(ref_ids[t].tolist())) <= 2, f"token {t}"
            continue
        assert (ids[t] == ref_ids[t]).all(), f"token {t}: {ids[t]} vs {ref_ids[t]}"
    w, rw = np.asarray(weights, np.float64), np.asarray(ref_weights, np.float64)
    same = ids == ref_ids
    assert np.all(np.abs(w - rw)[same] <= WEIGHT_RTOL * np.abs(rw)[same] + 1e-30), \
        f"weights: max rel err {np.max(np.abs(w - rw)[same] / np.abs(rw)[same])}"
