"""GPU parity of the NVFP4 slot MoE and of the packed-UE8M0 scale unpacking
against the oracle, through the C ABI."""

import dataclasses

import numpy as np
import pytest
import torch

from oracle import moe_fp8, moe_nvfp4, routing
from synth import workloads as W
from tests.parity import assert_outputs

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module")
def fme():
    import fp4_moe_expert_gb300 as m
    return m


def _host_weights(cfg, seed):
    w13, s13, w2, s2 = W.nvfp4_weights_host(cfg, seed)
    return w13, s13, w2, s2


def _run(fme, cfg, M, seed, weights_scale=1.0, tokens=None, device_weights=False):
    w13h, s13h, w2h, s2h = _host_weights(cfg, seed)
    if device_weights:
        w13, s13, w2, s2 = W.nvfp4_weights_device(cfg, seed, DEV)
    else:
        w13, s13, w2, s2 = (torch.from_numpy(h.full()).to(DEV) for h in (w13h, s13h, w2h, s2h))
    x, logits, bias = W.nvfp4_activations(cfg, M, seed)
    ids, wts, _ = routing.route(logits, bias, cfg.top_k, 1.0)
    wts = (wts * np.float32(weights_scale)).astype(np.float32)
    y = fme.moe_routed_nvfp4(torch.from_numpy(x).to(DEV).to(torch.bfloat16), torch.from_numpy(ids).to(DEV),
                             torch.from_numpy(wts).to(DEV), w13, s13, w2, s2, cfg.e0, cfg.limit)
    torch.cuda.synchronize()
    sel = np.arange(M) if tokens is None else np.asarray(tokens)
    ref = moe_nvfp4.routed_nvfp4(x[sel], ids[sel], wts[sel], w13h, s13h, w2h, s2h, cfg.e0, cfg.L, cfg.limit)
    return y.float().cpu().numpy()[sel], ref, ids


SMALL = W.Nvfp4Config("nvfp4_small", 256, 128, 6, 12, 3, 3, float("inf"), (5,))
RAGGED = W.Nvfp4Config("nvfp4_ragged", 1024, 384, 10, 40, 20, 4, float("inf"), (7,))
# H and N odd multiples of 128: the last 256-value K block of both GEMMs is half past the row.
ODD = W.Nvfp4Config("nvfp4_odd", 384, 640, 7, 14, 2, 3, float("inf"), (9,))


@pytest.mark.parametrize("cfg,M", [(SMALL, 5), (RAGGED, 7), (dataclasses.replace(SMALL, limit=2.0), 6),
                                   (ODD, 9), (ODD, 24), (ODD, 33)])
def test_nvfp4_small_full_parity(fme, cfg, M):
    got, ref, ids = _run(fme, cfg, M, seed=41)
    local = ((ids >= cfg.e0) & (ids < cfg.e0 + cfg.L)).any(axis=1)
    assert (got[~local] == 0).all()
    nz = local
    if nz.any():
        assert_outputs(got[nz], ref[nz])


def test_nvfp4_weights_applied_once_on_gpu(fme):
    got1, ref1, _ = _run(fme, RAGGED, 6, seed=42)
    got2, ref2, _ = _run(fme, RAGGED, 6, seed=42, weights_scale=2.0)
    assert np.array_equal(got2, 2 * got1)  # exact: power-of-two scaling of FP32 sums before one BF16 rounding
    assert np.array_equal(ref2, 2 * ref1)


def test_nvfp4_no_local_slots_gives_zeros(fme):
    cfg = dataclasses.replace(SMALL, e0=100)
    got, ref, _ = _run(fme, cfg, 4, seed=43)
    assert (got == 0).all() and (ref == 0).all()


def test_nvfp4_full_size_m8(fme):
    got, ref, ids = _run(fme, W.NVFP4, 8, seed=44, device_weights=True)
    local = ((ids >= 0) & (ids < W.NVFP4.L)).any(axis=1)
    assert local.any()
    assert_outputs(got[local], ref[local])


def test_nvfp4_full_size_m64_sampled_tokens(fme):
    got, ref, ids = _run(fme, W.NVFP4, 64, seed=45, tokens=[3, 40], device_weights=True)
    for i, t in enumerate([3, 40]):
        if ((ids[t] >= 0) & (ids[t] < W.NVFP4.L)).any():
            assert_outputs(got[i:i + 1], ref[i:i + 1])
        else:
            assert (got[i] == 0).all()


def test_ue8m0_unpack_matches_oracle_and_detects_mismatch(fme):
    rng = np.random.default_rng(46)
    n, k = 512, 2048
    exps = rng.integers(100, 140, size=(n // 128, k // 128)).astype(np.uint32)
    per_row = np.repeat(exps, 128, axis=0)  # uniform inside each 128-row block
    packed = np.zeros((n, k // 512), np.uint32)
    for g in range(k // 128):
        packed[:, g // 4] |= per_row[:, g] << np.uint32(8 * (g % 4))
    dev = torch.from_numpy(packed.view(np.int32)).to(DEV)
    got = fme.ue8m0_unpack(dev, n, k).cpu().numpy()
    assert np.array_equal(got, moe_fp8.ue8m0_unpack(packed.view(np.int32), n, k))
    packed[300, 1] ^= np.uint32(1 << 8)
    with pytest.raises(ValueError):
        fme.ue8m0_unpack(torch.from_numpy(packed.view(np.int32)).to(DEV), n, k)


# ---------------------------------------------------------------- fused routing
@pytest.mark.parametrize("cfg,M,logits_bf16", [(SMALL, 5, False), (RAGGED, 7, True), (ODD, 20, True),
                                                (ODD, 33, False)])
def test_nvfp4_fused_routing_matches_oracle_and_unfused_call(fme, cfg, M, logits_bf16):
    from tests.parity import assert_routing
    w13h, s13h, w2h, s2h = _host_weights(cfg, 51)
    w13, s13, w2, s2 = (torch.from_numpy(h.full()).to(DEV) for h in (w13h, s13h, w2h, s2h))
    x, logits, bias = W.nvfp4_activations(cfg, M, 51)
    if logits_bf16:
        logits = codecs_bf16(logits)
    scale = 1.5
    xd = torch.from_numpy(x).to(DEV).to(torch.bfloat16)
    ld = torch.from_numpy(logits).to(DEV)
    ld = ld.to(torch.bfloat16) if logits_bf16 else ld
    y, ids, wts = fme.moe_layer_nvfp4(xd, ld, torch.from_numpy(bias).to(DEV), w13, s13, w2, s2, cfg.e0, cfg.top_k,
                                      scale, cfg.limit)
    rids, rw, keys = routing.route(logits, bias, cfg.top_k, scale)
    assert_routing(ids.cpu().numpy(), wts.cpu().numpy(), rids, rw, keys)
    # the slot MoE on the kernel's own picks: the oracle, and the unfused entry bit for bit
    gi, gw = ids.cpu().numpy(), wts.cpu().numpy()
    ref = moe_nvfp4.routed_nvfp4(x, gi, gw, w13h, s13h, w2h, s2h, cfg.e0, cfg.L, cfg.limit)
    local = ((gi >= cfg.e0) & (gi < cfg.e0 + cfg.L)).any(axis=1)
    got = y.float().cpu().numpy()
    assert (got[~local] == 0).all()
    if local.any():
        assert_outputs(got[local], ref[local])
    y2 = fme.moe_routed_nvfp4(xd, ids, wts, w13, s13, w2, s2, cfg.e0, cfg.limit)
    assert torch.equal(y, y2)


def codecs_bf16(a):
    from oracle import codecs
    return codecs.bf16_round(np.asarray(a, dtype=np.float32))


def test_nvfp4_fused_routing_full_size_m64_sampled_tokens(fme):
    # 384-expert router, 48 local experts, BF16 logits: picks against the oracle for
    # every token, y against the oracle for two sampled tokens on the kernel's picks
    from tests.parity import assert_routing
    cfg = W.NVFP4
    M, seed = 64, 46
    w13h, s13h, w2h, s2h = _host_weights(cfg, seed)
    w13, s13, w2, s2 = W.nvfp4_weights_device(cfg, seed, DEV)
    x, logits, bias = W.nvfp4_activations(cfg, M, seed)
    logits = codecs_bf16(logits)
    y, ids, wts = fme.moe_layer_nvfp4(torch.from_numpy(x).to(DEV).to(torch.bfloat16),
                                      torch.from_numpy(logits).to(DEV).to(torch.bfloat16),
                                      torch.from_numpy(bias).to(DEV), w13, s13, w2, s2, cfg.e0, cfg.top_k, 1.0,
                                      cfg.limit)
    rids, rw, keys = routing.route(logits, bias, cfg.top_k, 1.0)
    gi, gw = ids.cpu().numpy(), wts.cpu().numpy()
    assert_routing(gi, gw, rids, rw, keys)
    tokens = [t for t in range(M) if ((gi[t] >= cfg.e0) & (gi[t] < cfg.e0 + cfg.L)).any()][:2]
    assert tokens
    ref = moe_nvfp4.routed_nvfp4(x[tokens], gi[tokens], gw[tokens], w13h, s13h, w2h, s2h, cfg.e0, cfg.L, cfg.limit)
    assert_outputs(y.float().cpu().numpy()[tokens], ref)
