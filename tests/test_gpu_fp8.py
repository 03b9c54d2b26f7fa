"""GPU parity of the routed FP8 layer and the FP8 shared expert against the
oracle, through the C ABI (via the thin binding)."""

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


def _device_problem(cfg, M, seed, step=0):
    w13h, w2h = W.fp8_weights_host(cfg, seed)
    s13, s2 = W.fp8_weight_scales(cfg, seed)
    x, logits, bias = W.fp8_activations(cfg, M, seed, step)
    return w13h, w2h, s13, s2, x, logits, bias


def _to_dev(cfg, x, logits, bias):
    xd = torch.from_numpy(x).to(DEV).to(torch.bfloat16)
    ld = torch.from_numpy(logits).to(DEV)
    if cfg.logits_bf16:
        ld = ld.to(torch.bfloat16)
    return xd, ld, torch.from_numpy(bias).to(DEV)


def _run_small(fme, cfg, M, seed, top_k=None, **over):
    top_k = top_k or cfg.top_k
    w13h, w2h, s13, s2, x, logits, bias = _device_problem(cfg, M, seed)
    w13 = torch.from_numpy(w13h.full()).to(DEV)
    w2 = torch.from_numpy(w2h.full()).to(DEV)
    xd, ld, bd = _to_dev(cfg, x, logits, bias)
    out, ids, wts = fme.moe_routed_fp8(xd, ld, bd, w13, torch.from_numpy(s13).to(DEV), w2,
                                       torch.from_numpy(s2).to(DEV), top_k, cfg.limit, cfg.scale, cfg.ue8m0)
    torch.cuda.synchronize()
    ref, rids, rw, keys = moe_fp8.routed_fp8(x, logits, bias, w13h, s13, w2h, s2, top_k, cfg.limit, cfg.scale,
                                             cfg.ue8m0)
    assert_routing(ids.cpu().numpy(), wts.cpu().numpy(), rids, rw, keys)
    got = out.float().cpu().numpy()
    return got, ref, ids.cpu().numpy(), rids


@pytest.mark.parametrize("cfg_name,M", [("tiny_fp8", 1), ("ragged_fp8", 5), ("ragged_fp8", 24)])
@pytest.mark.parametrize("ue8m0", [False, True])
def test_routed_small_full_parity(fme, cfg_name, M, ue8m0):
    import dataclasses
    cfg = dataclasses.replace(W.FP8_CONFIGS[cfg_name], ue8m0=ue8m0)
    got, ref, ids, rids = _run_small(fme, cfg, M, seed=3)
    assert_outputs(got, ref)


@pytest.mark.parametrize("M,E,k", [(1, 256, 8), (1, 40, 3), (1, 256, 1), (2, 96, 32), (3, 256, 8), (4, 200, 16),
                                   (4, 33, 32), (1, 1024, 32), (2, 300, 8), (5, 896, 16), (9, 128, 8),
                                   (17, 1024, 32)])
def test_routing_small_m_with_key_ties(fme, M, E, k):
    """The kernel routes in three ways: up to 4 tokens (one token up to 1024
    experts) it splits each token's experts over several warps of every CTA and
    merges their picks; with more tokens or experts each CTA routes its own
    share of the tokens that way and all CTAs read every pick back; otherwise a
    warp routes a token. ids must equal the oracle's bit for bit in all three,
    including exact key ties between experts of different 32-expert blocks
    (equal logits and equal bias: the lower expert id goes first)."""
    import dataclasses
    cfg = dataclasses.replace(W.TINY, H=256, I=128, E=E, top_k=k, name=f"route_{E}_{k}")
    w13h, w2h, s13, s2, x, logits, bias = _device_problem(cfg, M, seed=40 + E + k)
    tied = [e for e in (3, 35, 67, 99, 131, 163, 291, 899) if e < E]
    bias[tied] = bias[tied[0]]
    for t in range(M):
        logits[t, tied] = logits[t].max() + 0.5
        if t % 2:
            logits[t, tied[-1]] = logits[t].max() + 0.25  # a single winner ahead of the tie
    w13 = torch.from_numpy(w13h.full()).to(DEV)
    w2 = torch.from_numpy(w2h.full()).to(DEV)
    xd, ld, bd = _to_dev(cfg, x, logits, bias)
    out, ids, wts = fme.moe_routed_fp8(xd, ld, bd, w13, torch.from_numpy(s13).to(DEV), w2,
                                       torch.from_numpy(s2).to(DEV), k, cfg.limit, cfg.scale, cfg.ue8m0)
    torch.cuda.synchronize()
    ref, rids, rw, keys = moe_fp8.routed_fp8(x, logits, bias, w13h, s13, w2h, s2, k, cfg.limit, cfg.scale, cfg.ue8m0)
    assert np.array_equal(ids.cpu().numpy(), rids)  # no excuse: ties are exact, gaps elsewhere are wide
    assert np.allclose(wts.cpu().numpy(), rw, rtol=1e-6, atol=0)
    assert_outputs(out.float().cpu().numpy(), ref)


def test_routed_top_k_equals_E_and_max_tokens(fme):
    import dataclasses
    cfg = dataclasses.replace(W.TINY, H=256, I=128, E=8, top_k=8, name="topk_all")
    got, ref, ids, _ = _run_small(fme, cfg, 3, seed=4)
    assert_outputs(got, ref)
    assert sorted(ids[0].tolist()) == list(range(8))
    cfg = dataclasses.replace(W.TINY, H=256, I=128, E=16, top_k=4, name="max_tokens")
    got, ref, _, _ = _run_small(fme, cfg, 64, seed=5)
    assert_outputs(got, ref)


def test_routed_deterministic_and_identical_tokens(fme):
    cfg = W.RAGGED
    w13h, w2h, s13, s2, x, logits, bias = _device_problem(cfg, 4, 6)
    x[2] = x[0]
    logits[2] = logits[0]
    w13 = torch.from_numpy(w13h.full()).to(DEV)
    w2 = torch.from_numpy(w2h.full()).to(DEV)
    xd, ld, bd = _to_dev(cfg, x, logits, bias)
    args = (xd, ld, bd, w13, torch.from_numpy(s13).to(DEV), w2, torch.from_numpy(s2).to(DEV), cfg.top_k,
            cfg.limit, cfg.scale, cfg.ue8m0)
    outs = [fme.moe_routed_fp8(*args)[0].clone() for _ in range(5)]
    for o in outs[1:]:
        assert torch.equal(o, outs[0])
    k = cfg.top_k
    assert torch.equal(outs[0][0:k], outs[0][2 * k:3 * k])


def test_routed_workspace_stays_clean(fme):
    cfg = W.TINY
    w13h, w2h, s13, s2, x, logits, bias = _device_problem(cfg, 1, 7)
    ws = fme.Workspace(fme.moe_routed_fp8_workspace(1, cfg.H, cfg.I, cfg.E, cfg.top_k), DEV)
    w13 = torch.from_numpy(w13h.full()).to(DEV)
    w2 = torch.from_numpy(w2h.full()).to(DEV)
    xd, ld, bd = _to_dev(cfg, x, logits, bias)
    for _ in range(3):
        fme.moe_routed_fp8(xd, ld, bd, w13, torch.from_numpy(s13).to(DEV), w2, torch.from_numpy(s2).to(DEV),
                           cfg.top_k, cfg.limit, cfg.scale, cfg.ue8m0, workspace=ws)
    torch.cuda.synchronize()
    assert ws.error() == 0
    counters = ws.buf[256:256 + 2 * 256].view(torch.int32)
    assert int(counters.abs().sum().item()) == 0


def test_routed_one_workspace_serves_every_token_count(fme):
    """A workspace sized for the largest M is reused by calls with fewer tokens."""
    cfg = W.RAGGED
    w13h, w2h = W.fp8_weights_host(cfg, 8)
    s13, s2 = W.fp8_weight_scales(cfg, 8)
    w13 = torch.from_numpy(w13h.full()).to(DEV)
    w2 = torch.from_numpy(w2h.full()).to(DEV)
    ws = fme.Workspace(fme.moe_routed_fp8_workspace(8, cfg.H, cfg.I, cfg.E, cfg.top_k), DEV)
    for step, M in enumerate((8, 1, 5, 2, 8)):
        x, logits, bias = W.fp8_activations(cfg, M, 8, step)
        xd, ld, bd = _to_dev(cfg, x, logits, bias)
        out, ids, wts = fme.moe_routed_fp8(xd, ld, bd, w13, torch.from_numpy(s13).to(DEV), w2,
                                           torch.from_numpy(s2).to(DEV), cfg.top_k, cfg.limit, cfg.scale,
                                           cfg.ue8m0, workspace=ws)
        torch.cuda.synchronize()
        assert ws.error() == 0, (step, M)
        ref, rids, rw, keys = moe_fp8.routed_fp8(x, logits, bias, w13h, s13, w2h, s2, cfg.top_k, cfg.limit,
                                                 cfg.scale, cfg.ue8m0)
        assert_routing(ids.cpu().numpy(), wts.cpu().numpy(), rids, rw, keys)
        assert_outputs(out.float().cpu().numpy(), ref)


def _full_size(fme, cfg, M, seed, routes, rows):
    w13, s13, w2, s2 = W.fp8_weights_device(cfg, seed, DEV)
    s13h, s2h = s13.cpu().numpy(), s2.cpu().numpy()
    w13h, w2h = W.fp8_weights_host(cfg, seed)
    x, logits, bias = W.fp8_activations(cfg, M, seed)
    xd, ld, bd = _to_dev(cfg, x, logits, bias)
    out, ids, wts = fme.moe_routed_fp8(xd, ld, bd, w13, s13, w2, s2, cfg.top_k, cfg.limit, cfg.scale, cfg.ue8m0)
    torch.cuda.synchronize()
    ref, rids, rw, keys = moe_fp8.routed_fp8(x, logits, bias, w13h, s13h, w2h, s2h, cfg.top_k, cfg.limit,
                                             cfg.scale, cfg.ue8m0, routes=routes, rows=rows)
    assert_routing(ids.cpu().numpy(), wts.cpu().numpy(), rids, rw, keys)
    # the device-filled weights are the generator's bytes
    e = int(rids.reshape(-1)[routes[0]])
    assert np.array_equal(w13[e, :64].cpu().numpy(), w13h[e][:64])
    got = out.float().cpu().numpy()
    assert_outputs(got[routes][:, rows], ref[routes][:, rows])
    return out


def test_dsv3_m1_full_size_all_routes(fme):
    _full_size(fme, W.DSV3, 1, seed=11, routes=list(range(8)), rows=np.arange(7168))


def test_dsv3_m8_sampled_routes(fme):
    rng = np.random.default_rng(1)
    routes = sorted(rng.choice(64, 4, replace=False).tolist())
    _full_size(fme, W.DSV3, 8, seed=12, routes=routes, rows=np.arange(7168))


def test_dsv3_ue8m0_m4_sampled(fme):
    _full_size(fme, W.DSV3_UE8M0, 4, seed=13, routes=[0, 13, 31], rows=np.arange(0, 7168, 7))


def test_latent_m32_sampled_routes(fme):
    rng = np.random.default_rng(2)
    routes = sorted(rng.choice(32 * 16, 5, replace=False).tolist())
    _full_size(fme, W.LATENT, 32, seed=14, routes=routes, rows=np.arange(3584))


@pytest.mark.parametrize("M", [1, 5, 16])
def test_latent_full_size(fme, M):
    """Latent-MoE shape (H 3584, I 2048, 896 experts, top_k 16, FP32 logits, skewed
    bias N(0, 0.5)) at full size: every route at M = 1; at M = 5 and 16 the
    routes of the expert picked by the most tokens (expert sharing) plus
    others, each compared on all 3584 rows."""
    cfg = W.LATENT
    x, logits, bias = W.fp8_activations(cfg, M, 15 + M)
    ids, _, _ = routing.route(logits, bias, cfg.top_k, cfg.scale)
    if M == 1:
        routes = list(range(cfg.top_k))
    else:
        flat = ids.reshape(-1)
        vals, counts = np.unique(flat, return_counts=True)
        shared = int(vals[np.argmax(counts)])
        assert counts.max() >= 2, "the skewed bias should make some expert shared"
        routes = [int(r) for r in np.nonzero(flat == shared)[0][:3]]
        rng = np.random.default_rng(M)
        rest = [r for r in range(M * cfg.top_k) if r not in routes]
        routes = sorted(routes + rng.choice(rest, 3, replace=False).tolist())
    _full_size(fme, cfg, M, seed=15 + M, routes=routes, rows=np.arange(cfg.H))


@pytest.mark.parametrize("M", [1, 3])
def test_shared_expert_full_size(fme, M):
    cfg = W.SHARED
    w13, s13, w2, s2 = W.shared_weights_host(cfg, seed=21)
    x, _, _ = W.fp8_activations(W.DSV3, M, seed=21)
    out, gu = fme.shared_expert_fp8(torch.from_numpy(x).to(DEV).to(torch.bfloat16), torch.from_numpy(w13).to(DEV),
                                    torch.from_numpy(s13).to(DEV), torch.from_numpy(w2).to(DEV),
                                    torch.from_numpy(s2).to(DEV), cfg.limit, cfg.ue8m0, want_gate_up=True)
    torch.cuda.synchronize()
    ref, ref_gu = moe_fp8.shared_fp8(x, w13, s13, w2, s2, cfg.limit, cfg.ue8m0)
    assert_outputs(gu.float().cpu().numpy(), ref_gu, "gate_up")
    assert_outputs(out.float().cpu().numpy(), ref, "out")


def test_shared_expert_small_non_ue8m0(fme):
    cfg = W.SharedConfig("small_shared", 1024, 384, 7.0, False)
    w13, s13, w2, s2 = W.shared_weights_host(cfg, seed=22)
    x, _, _ = W.fp8_activations(W.RAGGED, 5, seed=22)
    out = fme.shared_expert_fp8(torch.from_numpy(x).to(DEV).to(torch.bfloat16), torch.from_numpy(w13).to(DEV),
                                torch.from_numpy(s13).to(DEV), torch.from_numpy(w2).to(DEV),
                                torch.from_numpy(s2).to(DEV), cfg.limit, cfg.ue8m0)
    torch.cuda.synchronize()
    ref, _ = moe_fp8.shared_fp8(x, w13, s13, w2, s2, cfg.limit, cfg.ue8m0)
    assert_outputs(out.float().cpu().numpy(), ref)


def test_device_generator_matches_host(fme):
    import synth
    t = synth.e4m3_normal_table()
    buf = torch.empty(3, 40, 96, dtype=torch.uint8, device=DEV)
    synth.fill_codes_device(buf, 5, synth.T_W2, t, expert0=7)
    for e in range(3):
        assert np.array_equal(buf[e].cpu().numpy(), synth.expert_bytes(5, synth.T_W2, 7 + e, 40, 96, t))
