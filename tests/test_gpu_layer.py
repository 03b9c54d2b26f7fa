"""GPU parity of the one-launch FP8 layer (routed experts + shared expert)
against the oracle, and agreement with the two separate calls."""

import dataclasses

import numpy as np
import pytest
import torch

from oracle import moe_fp8, routing
from synth import workloads as W
from tests.parity import assert_outputs, assert_routing

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module")
def fme():
    import fp4_moe_expert_gb300 as m
    return m


def _dev(a):
    return torch.from_numpy(a).to(DEV)


def _small_problem(cfg, scfg, M, seed):
    w13h, w2h = W.fp8_weights_host(cfg, seed)
    s13, s2 = W.fp8_weight_scales(cfg, seed)
    x, logits, bias = W.fp8_activations(cfg, M, seed)
    shared = W.shared_weights_host(scfg, seed + 100)
    return w13h, w2h, s13, s2, x, logits, bias, shared


def _close(a, b, what):
    """Same values up to FP32 summation order: |a - b| <= 2 BF16 ulp of |b|."""
    a, b = a.float(), b.float()
    ulp = torch.clamp(b.abs(), min=2.0 ** -126) * 2.0 ** -7
    bad = int(((a - b).abs() > 2 * ulp).sum().item())
    assert bad <= max(1, b.numel() // 1000), f"{what}: {bad} of {b.numel()} differ by more than 2 ulp"


def _check_layer(fme, cfg, scfg, M, seed, ws=None, shared_ws=None):
    w13h, w2h, s13, s2, x, logits, bias, (sw13, ss13, sw2, ss2) = _small_problem(cfg, scfg, M, seed)
    xd = _dev(x).to(torch.bfloat16)
    ld = _dev(logits).to(torch.bfloat16) if cfg.logits_bf16 else _dev(logits)
    routed = (xd, ld, _dev(bias), _dev(w13h.full()), _dev(s13), _dev(w2h.full()), _dev(s2), cfg.top_k, cfg.limit,
              cfg.scale, cfg.ue8m0)
    shared = (_dev(sw13), _dev(ss13), _dev(sw2), _dev(ss2), scfg.limit, scfg.ue8m0)
    if ws is None:
        ws = fme.Workspace(fme.moe_layer_fp8_workspace(M, cfg.H, cfg.I, cfg.E, cfg.top_k), DEV)
    out, ids, wts, sout = fme.moe_layer_fp8(*routed, *shared, workspace=ws)
    torch.cuda.synchronize()
    assert ws.error() == 0
    ref, rids, rw, keys = moe_fp8.routed_fp8(x, logits, bias, w13h, s13, w2h, s2, cfg.top_k, cfg.limit, cfg.scale,
                                             cfg.ue8m0)
    assert_routing(ids.cpu().numpy(), wts.cpu().numpy(), rids, rw, keys)
    assert_outputs(out.float().cpu().numpy(), ref, "routed")
    sref, _ = moe_fp8.shared_fp8(x, sw13, ss13, sw2, ss2, scfg.limit, scfg.ue8m0)
    assert_outputs(sout.float().cpu().numpy(), sref, "shared")
    # the one-launch layer agrees with the two separate calls
    if shared_ws is None:
        shared_ws = fme.Workspace(fme.shared_expert_fp8_workspace(M, cfg.H, cfg.I), DEV)
    out2, ids2, wts2 = fme.moe_routed_fp8(*routed, workspace=ws)
    sout2 = fme.shared_expert_fp8(xd, *shared, workspace=shared_ws)
    torch.cuda.synchronize()
    assert ws.error() == 0 and shared_ws.error() == 0
    assert torch.equal(ids, ids2) and torch.equal(wts, wts2)
    _close(out, out2, "routed")
    _close(sout, sout2, "shared")


@pytest.mark.parametrize("M", [1, 4, 5, 16, 17, 64])
@pytest.mark.parametrize("shared_ue8m0", [False, True])
def test_layer_small_matches_oracle_and_separate_calls(fme, M, shared_ue8m0):
    scfg = W.SharedConfig("small_shared", W.RAGGED.H, W.RAGGED.I, 5.0, shared_ue8m0)
    _check_layer(fme, W.RAGGED, scfg, M, seed=31)


def test_layer_tiny_single_token(fme):
    scfg = W.SharedConfig("tiny_shared", W.TINY.H, W.TINY.I, 6.0, True)
    _check_layer(fme, W.TINY, scfg, 1, seed=32)


def test_layer_workspace_shared_with_routed_calls(fme):
    """One workspace serves one-launch and routed-only calls in any order and
    with any token count up to its size (the shared-expert call has its own)."""
    cfg = W.RAGGED
    scfg = W.SharedConfig("small_shared", cfg.H, cfg.I, 7.0, True)
    ws = fme.Workspace(fme.moe_layer_fp8_workspace(8, cfg.H, cfg.I, cfg.E, cfg.top_k), DEV)
    sws = fme.Workspace(fme.shared_expert_fp8_workspace(8, cfg.H, cfg.I), DEV)
    for step, M in enumerate((8, 3, 8, 1)):
        _check_layer(fme, cfg, scfg, M, seed=40 + step, ws=ws, shared_ws=sws)


def test_layer_one_and_two_launch_calls_share_a_workspace(fme):
    """Above 16 tokens the layer call runs the shared expert, then the routed
    experts, as two launches; calls on either side of that line, in any order,
    share one workspace sized for the largest."""
    cfg = W.RAGGED
    scfg = W.SharedConfig("small_shared", cfg.H, cfg.I, 7.0, False)
    ws = fme.Workspace(fme.moe_layer_fp8_workspace(32, cfg.H, cfg.I, cfg.E, cfg.top_k), DEV)
    sws = fme.Workspace(fme.shared_expert_fp8_workspace(32, cfg.H, cfg.I), DEV)
    for step, M in enumerate((32, 8, 17, 16, 1)):
        _check_layer(fme, cfg, scfg, M, seed=50 + step, ws=ws, shared_ws=sws)


def test_layer_dsv3_full_size(fme):
    cfg, scfg = W.DSV3, W.SHARED
    M, seed = 4, 33
    w13, s13, w2, s2 = W.fp8_weights_device(cfg, seed, DEV)
    w13h, w2h = W.fp8_weights_host(cfg, seed)
    sw13, ss13, sw2, ss2 = W.shared_weights_host(scfg, seed)
    x, logits, bias = W.fp8_activations(cfg, M, seed)
    xd, ld = _dev(x).to(torch.bfloat16), _dev(logits).to(torch.bfloat16)
    routed = (xd, ld, _dev(bias), w13, s13, w2, s2, cfg.top_k, cfg.limit, cfg.scale, cfg.ue8m0)
    shared = (_dev(sw13), _dev(ss13), _dev(sw2), _dev(ss2), scfg.limit, scfg.ue8m0)
    ws = fme.Workspace(fme.moe_layer_fp8_workspace(M, cfg.H, cfg.I, cfg.E, cfg.top_k), DEV)
    out, ids, wts, sout = fme.moe_layer_fp8(*routed, *shared, workspace=ws)
    torch.cuda.synchronize()
    assert ws.error() == 0
    routes = [0, 9, 22, 31]
    ref, rids, rw, keys = moe_fp8.routed_fp8(x, logits, bias, w13h, s13.cpu().numpy(), w2h, s2.cpu().numpy(),
                                             cfg.top_k, cfg.limit, cfg.scale, cfg.ue8m0, routes=routes,
                                             rows=np.arange(7168))
    assert_routing(ids.cpu().numpy(), wts.cpu().numpy(), rids, rw, keys)
    assert_outputs(out.float().cpu().numpy()[routes], ref[routes], "routed")
    sref, _ = moe_fp8.shared_fp8(x, sw13, ss13, sw2, ss2, scfg.limit, scfg.ue8m0)
    assert_outputs(sout.float().cpu().numpy(), sref, "shared")
    sws = fme.Workspace(fme.shared_expert_fp8_workspace(M, cfg.H, cfg.I), DEV)
    out2, _, _ = fme.moe_routed_fp8(*routed, workspace=ws)
    sout2 = fme.shared_expert_fp8(xd, *shared, workspace=sws)
    torch.cuda.synchronize()
    assert ws.error() == 0 and sws.error() == 0
    _close(out, out2, "routed")
    _close(sout, sout2, "shared")
