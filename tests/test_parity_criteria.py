"""The parity criteria themselves (CPU): the stated output tolerance, and the
rounding-tie rule that leaves one-ulp flips at a BF16 midpoint out of the row
maximum and nothing else."""

import numpy as np

from oracle import moe_fp8
from oracle.codecs import bf16_round
from synth import workloads as W
from tests.parity import ROW_RMS_FRAC, bf16_ulp, output_report


def _row():
    rng = np.random.default_rng(0)
    ref = bf16_round(rng.normal(0, 1e-3, 256)).astype(np.float64)
    ref[7] = bf16_round(np.array([5.5e-3]))[0]  # a large element, about 5 x the row RMS
    return ref


def test_one_ulp_flip_on_a_large_element_breaks_the_plain_row_criterion():
    ref = _row()
    got = ref.copy()
    got[7] = ref[7] - bf16_ulp(ref[7])
    r = output_report(got[None], ref[None])
    assert r["frac_within_2ulp"] == 1.0
    assert r["worst_row_maxerr_over_rms"] > ROW_RMS_FRAC


def test_tie_flip_is_excused_only_at_the_midpoint():
    ref = _row()
    got = ref.copy()
    got[7] = ref[7] - bf16_ulp(ref[7])
    mid = 0.5 * (got[7] + ref[7])
    exact = ref.copy()
    exact[7] = mid * (1 + 1e-7)  # rounds to ref[7]; a reordered FP32 sum may land below the midpoint
    r = output_report(got[None], ref[None], exact[None])
    assert r["tie_flips"] == 1 and r["worst_row_maxerr_over_rms"] == 0.0
    exact[7] = mid * (1 + 1e-3)  # far from the midpoint: the flip is an error
    r = output_report(got[None], ref[None], exact[None])
    assert r["tie_flips"] == 0 and r["worst_row_maxerr_over_rms"] > ROW_RMS_FRAC


def test_two_ulp_errors_are_never_excused():
    ref = _row()
    got = ref.copy()
    got[7] = ref[7] - 2 * bf16_ulp(ref[7])
    exact = ref.copy()
    exact[7] = ref[7] - bf16_ulp(ref[7])
    r = output_report(got[None], ref[None], exact[None])
    assert r["tie_flips"] == 0 and r["worst_row_maxerr_over_rms"] > ROW_RMS_FRAC


def test_oracle_exact_output_rounds_to_its_output():
    cfg = W.TINY
    w13h, w2h = W.fp8_weights_host(cfg, 3)
    s13, s2 = W.fp8_weight_scales(cfg, 3)
    x, logits, bias = W.fp8_activations(cfg, 2, 3)
    out, _, _, _, exact = moe_fp8.routed_fp8(x, logits, bias, w13h, s13, w2h, s2, cfg.top_k, cfg.limit, cfg.scale,
                                             cfg.ue8m0, exact=True)
    assert np.array_equal(bf16_round(exact), out)
    assert not np.array_equal(exact, out.astype(np.float64))


def test_routing_excuse_is_a_few_ulps_of_the_keys():
    """A swap of two picks is excused only where the oracle's deciding keys
    are within GAP_ULPS float32 ulps of each other; the count is returned."""
    import pytest
    from tests.parity import GAP_ULPS, assert_routing, decisive_gap_ulps
    one = np.float32(0.75)
    ulp = float(np.spacing(one))
    keys = np.array([[0.9, 0.75, 0.75 - 2 * ulp, 0.1],       # ranks 2/3 two ulps apart
                     [0.9, 0.75, 0.75 - 10 * ulp, 0.1]], np.float32)
    ref = np.array([[0, 1, 2], [0, 1, 2]], np.int32)
    w = np.full((2, 3), 1 / 3, np.float32)
    g = decisive_gap_ulps(keys, ref)
    assert g[0] == pytest.approx(2.0) and g[1] == pytest.approx(10.0)
    swapped = np.array([[0, 2, 1], [0, 1, 2]], np.int32)
    assert assert_routing(swapped, w, ref, w, keys) == 1
    with pytest.raises(AssertionError):
        assert_routing(np.array([[0, 1, 2], [0, 2, 1]], np.int32), w, ref, w, keys)
    assert GAP_ULPS <= 4
