"""GPU parity of the routed FP8 layer with MXFP8 activations (E4M3 values, one
E8M0 scale per 32) against the oracle, through the C ABI."""

import dataclasses

import numpy as np
import pytest
import torch

from oracle import ep_local, moe_fp8, routing
from synth import workloads as W
from tests.parity import assert_outputs, assert_routing

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module")
def fme():
    import fp4_moe_expert_gb300 as m
    return m


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def _logits(cfg, logits):
    ld = _dev(logits)
    return ld.to(torch.bfloat16) if cfg.logits_bf16 else ld


def _run(fme, cfg, M, seed, w13h, w2h, s13, s2, dev_weights=None, routes=None, rows=None, workspace=None, step=0):
    x, logits, bias = W.fp8_activations(cfg, M, seed, step)
    codes, scales = ep_local.mxfp8_quantize(x)
    if dev_weights is None:
        dev_weights = (_dev(w13h.full()), _dev(s13), _dev(w2h.full()), _dev(s2))
    w13, s13d, w2, s2d = dev_weights
    out, ids, wts = fme.moe_routed_fp8_mx(_dev(codes), _dev(scales), _logits(cfg, logits), _dev(bias), w13, s13d, w2,
                                          s2d, cfg.top_k, cfg.limit, cfg.scale, cfg.ue8m0, workspace=workspace)
    torch.cuda.synchronize()
    ref, rids, rw, keys, exact = moe_fp8.routed_fp8(x, logits, bias, w13h, s13, w2h, s2, cfg.top_k, cfg.limit,
                                                    cfg.scale, cfg.ue8m0, routes=routes, rows=rows,
                                                    x_mx=(codes, scales), exact=True)
    assert_routing(ids.cpu().numpy(), wts.cpu().numpy(), rids, rw, keys)
    got = out.float().cpu().numpy()
    if routes is not None:
        got, ref, exact = got[routes], ref[routes], exact[routes]
    if rows is not None:
        got, ref, exact = got[:, rows], ref[:, rows], exact[:, rows]
    assert_outputs(got, ref, "routed mx", exact)
    return out, ids


@pytest.mark.parametrize("cfg_name,M", [("tiny_fp8", 1), ("ragged_fp8", 5), ("ragged_fp8", 16), ("ragged_fp8", 24)])
@pytest.mark.parametrize("ue8m0", [False, True])
def test_mx_small_full_parity(fme, cfg_name, M, ue8m0):
    cfg = dataclasses.replace(W.FP8_CONFIGS[cfg_name], ue8m0=ue8m0)
    w13h, w2h = W.fp8_weights_host(cfg, 21)
    s13, s2 = W.fp8_weight_scales(cfg, 21)
    _run(fme, cfg, M, 21, w13h, w2h, s13, s2)


def test_mx_max_tokens_and_workspace_reuse(fme):
    """M = 64 (the large-token kernel) and fewer tokens on the same workspace,
    interleaved with BF16-input calls."""
    cfg = dataclasses.replace(W.TINY, H=256, I=128, E=16, top_k=4, name="mx_max_tokens")
    w13h, w2h = W.fp8_weights_host(cfg, 22)
    s13, s2 = W.fp8_weight_scales(cfg, 22)
    dw = (_dev(w13h.full()), _dev(s13), _dev(w2h.full()), _dev(s2))
    ws = fme.Workspace(fme.moe_routed_fp8_workspace(64, cfg.H, cfg.I, cfg.E, cfg.top_k), DEV)
    for step, M in enumerate((64, 3, 17)):
        _run(fme, cfg, M, 22, w13h, w2h, s13, s2, dev_weights=dw, workspace=ws, step=step)
        assert ws.error() == 0
        x, logits, bias = W.fp8_activations(cfg, M, 23, step)
        fme.moe_routed_fp8(_dev(x).to(torch.bfloat16), _logits(cfg, logits), _dev(bias), *dw, cfg.top_k, cfg.limit,
                           cfg.scale, cfg.ue8m0, workspace=ws)
        torch.cuda.synchronize()
        assert ws.error() == 0


def test_mx_device_quantiser_feeds_the_gemm(fme):
    """fme_mxfp8_quantize output goes straight into the MX entry: same result as
    the oracle's codes (the quantiser is bit-exact), and close to the BF16-input
    call (the two activation formats differ by their rounding only)."""
    cfg = W.RAGGED
    M = 4
    w13h, w2h = W.fp8_weights_host(cfg, 24)
    s13, s2 = W.fp8_weight_scales(cfg, 24)
    dw = (_dev(w13h.full()), _dev(s13), _dev(w2h.full()), _dev(s2))
    x, logits, bias = W.fp8_activations(cfg, M, 24)
    xd = _dev(x).to(torch.bfloat16)
    q, sc = fme.mxfp8_quantize(xd)
    out, ids, _ = fme.moe_routed_fp8_mx(q, sc, _logits(cfg, logits), _dev(bias), *dw, cfg.top_k, cfg.limit, cfg.scale,
                                        cfg.ue8m0)
    torch.cuda.synchronize()
    codes, scales = ep_local.mxfp8_quantize(x)
    assert np.array_equal(q.cpu().numpy(), codes) and np.array_equal(sc.cpu().numpy(), scales)
    ref, _, _, _, exact = moe_fp8.routed_fp8(x, logits, bias, w13h, s13, w2h, s2, cfg.top_k, cfg.limit, cfg.scale,
                                             cfg.ue8m0, x_mx=(codes, scales), exact=True)
    assert_outputs(out.float().cpu().numpy(), ref, "routed mx", exact)
    out_bf16, ids2, _ = fme.moe_routed_fp8(xd, _logits(cfg, logits), _dev(bias), *dw, cfg.top_k, cfg.limit, cfg.scale,
                                           cfg.ue8m0)
    torch.cuda.synchronize()
    assert torch.equal(ids, ids2)
    a, b = out.float(), out_bf16.float()
    rel = float((a - b).norm() / b.norm())
    assert rel < 0.08, rel


def test_mx_dsv3_m1_full_size(fme):
    cfg = W.DSV3
    w13, s13, w2, s2 = W.fp8_weights_device(cfg, 25, DEV)
    w13h, w2h = W.fp8_weights_host(cfg, 25)
    _run(fme, cfg, 1, 25, w13h, w2h, s13.cpu().numpy(), s2.cpu().numpy(), dev_weights=(w13, s13, w2, s2),
         routes=list(range(8)), rows=np.arange(7168))


def test_mx_dsv3_ue8m0_m8_sampled(fme):
    cfg = W.DSV3_UE8M0
    w13, s13, w2, s2 = W.fp8_weights_device(cfg, 26, DEV)
    w13h, w2h = W.fp8_weights_host(cfg, 26)
    rng = np.random.default_rng(3)
    routes = sorted(rng.choice(64, 3, replace=False).tolist())
    _run(fme, cfg, 8, 26, w13h, w2h, s13.cpu().numpy(), s2.cpu().numpy(), dev_weights=(w13, s13, w2, s2),
         routes=routes, rows=np.arange(0, 7168, 5))
