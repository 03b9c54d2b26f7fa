"""The workspace entry points inside a CUDA graph: every call is asynchronous on
the caller's stream and allocates nothing, so a call captured once replays with
new inputs copied into the captured buffers and gives, bit for bit, what a
direct call on those inputs gives (the kernels are deterministic, and each call
leaves its workspace counters at zero for the next)."""

import pytest
import torch

from oracle import routing
from synth import workloads as W
from tests.parity import assert_routing

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module")
def fme():
    import fp4_moe_expert_gb300 as m
    return m


def _capture(fn):
    """Warm up on a side stream, then capture one call of fn()."""
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for _ in range(2):
            fn()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    return g


def test_routed_fp8_and_layer_replay_match_direct_calls(fme):
    cfg = W.RAGGED
    scfg = W.SharedConfig("small_shared", cfg.H, cfg.I, 7.0, True)
    M = 5
    w13h, w2h = W.fp8_weights_host(cfg, 61)
    s13, s2 = W.fp8_weight_scales(cfg, 61)
    weights = [torch.from_numpy(a).to(DEV) for a in (w13h.full(), s13, w2h.full(), s2)]
    shared = [torch.from_numpy(a).to(DEV) for a in W.shared_weights_host(scfg, 62)]
    x0, l0, bias = W.fp8_activations(cfg, M, 63)
    x = torch.from_numpy(x0).to(DEV).to(torch.bfloat16)
    lg = torch.from_numpy(l0).to(DEV).to(torch.bfloat16)
    bd = torch.from_numpy(bias).to(DEV)
    out = torch.empty(M * cfg.top_k, cfg.H, dtype=torch.bfloat16, device=DEV)
    ids = torch.empty(M, cfg.top_k, dtype=torch.int32, device=DEV)
    wts = torch.empty(M, cfg.top_k, dtype=torch.float32, device=DEV)
    sout = torch.empty(M, cfg.H, dtype=torch.bfloat16, device=DEV)
    ws = fme.Workspace(fme.moe_layer_fp8_workspace(M, cfg.H, cfg.I, cfg.E, cfg.top_k), DEV)
    w13, s13d, w2, s2d = weights
    routed_args = (w13, s13d, w2, s2d, cfg.top_k, cfg.limit, cfg.scale, cfg.ue8m0)

    g_routed = _capture(lambda: fme.moe_routed_fp8(x, lg, bd, *routed_args, out=out, ids=ids, weights=wts,
                                                   workspace=ws))
    g_layer = _capture(lambda: fme.moe_layer_fp8(x, lg, bd, *routed_args, *shared, scfg.limit, scfg.ue8m0,
                                                 out=out, ids=ids, weights=wts, shared_out=sout, workspace=ws))
    for step in range(3):
        xn, ln, _ = W.fp8_activations(cfg, M, 70 + step)
        x.copy_(torch.from_numpy(xn).to(DEV).to(torch.bfloat16))
        lg.copy_(torch.from_numpy(ln).to(DEV).to(torch.bfloat16))
        g_routed.replay()
        torch.cuda.synchronize()
        assert ws.error() == 0
        ref_out, ref_ids, ref_w = fme.moe_routed_fp8(x, lg, bd, *routed_args)
        torch.cuda.synchronize()
        assert torch.equal(ids, ref_ids) and torch.equal(wts, ref_w) and torch.equal(out, ref_out)
        # the routing the replay used is the oracle's for these inputs
        oid, ow, okeys = routing.route(lg.float().cpu().numpy(), bias, cfg.top_k, cfg.scale)
        assert_routing(ids.cpu().numpy(), wts.cpu().numpy(), oid, ow, okeys)

        g_layer.replay()
        torch.cuda.synchronize()
        assert ws.error() == 0
        lo, lids, lw, lso = fme.moe_layer_fp8(x, lg, bd, *routed_args, *shared, scfg.limit, scfg.ue8m0)
        torch.cuda.synchronize()
        assert torch.equal(ids, lids) and torch.equal(wts, lw)
        assert torch.equal(out, lo) and torch.equal(sout, lso)


def test_nvfp4_layer_replay_matches_direct_calls(fme):
    cfg = W.Nvfp4Config("nvfp4_ragged", 1024, 384, 10, 40, 20, 4, float("inf"), (7,))
    M = 7
    nw = [torch.from_numpy(h.full()).to(DEV) for h in W.nvfp4_weights_host(cfg, 81)]
    x0, l0, b0 = W.nvfp4_activations(cfg, M, 82)
    x = torch.from_numpy(x0).to(DEV).to(torch.bfloat16)
    lg = torch.from_numpy(l0).to(DEV)
    bd = torch.from_numpy(b0).to(DEV)
    y = torch.empty(M, cfg.H, dtype=torch.bfloat16, device=DEV)
    ws = fme.Workspace(fme.moe_routed_nvfp4_workspace(M, cfg.H, cfg.N, cfg.L, cfg.top_k), DEV)
    box = {}

    def call():
        box["r"] = fme.moe_layer_nvfp4(x, lg, bd, *nw, cfg.e0, cfg.top_k, 1.0, cfg.limit, y=y, workspace=ws)

    g = _capture(call)
    for step in range(3):
        xn, ln, _ = W.nvfp4_activations(cfg, M, 90 + step)
        x.copy_(torch.from_numpy(xn).to(DEV).to(torch.bfloat16))
        lg.copy_(torch.from_numpy(ln).to(DEV))
        g.replay()
        torch.cuda.synchronize()
        ry, rids, rw = fme.moe_layer_nvfp4(x, lg, bd, *nw, cfg.e0, cfg.top_k, 1.0, cfg.limit)
        torch.cuda.synchronize()
        _, gids, gw = box["r"]
        assert torch.equal(gids, rids) and torch.equal(gw, rw) and torch.equal(y, ry)
        assert ws.error() == 0
