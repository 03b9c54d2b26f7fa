"""GPU parity of the local finalize against the oracle, through the C ABI:
standalone on seeded rows, and chained after the routed FP8 and layer calls."""

import numpy as np
import pytest
import torch

from oracle import codecs
from oracle.finalize import finalize as oracle_finalize
from synth import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module")
def fme():
    import fp4_moe_expert_gb300 as m
    return m


def _bf16_rows(rng, shape):
    return codecs.bf16_round(rng.normal(size=shape).astype(np.float32))


@pytest.mark.parametrize("M,k,H,shared", [(1, 8, 7168, False), (8, 8, 7168, True), (5, 3, 136, True),
                                          (64, 16, 3584, False), (2, 1, 8, True), (33, 32, 256, True)])
def test_finalize_bit_exact(fme, M, k, H, shared):
    rng = np.random.default_rng(M * 1000 + k * 10 + H)
    out = _bf16_rows(rng, (M * k, H))
    w = rng.uniform(0.0, 1.0, size=(M, k)).astype(np.float32)
    sh = _bf16_rows(rng, (M, H)) if shared else None
    ref = oracle_finalize(out, w, sh)
    got = fme.moe_finalize(torch.from_numpy(out).to(DEV).to(torch.bfloat16), torch.from_numpy(w).to(DEV),
                           None if sh is None else torch.from_numpy(sh).to(DEV).to(torch.bfloat16))
    assert np.array_equal(got.float().cpu().numpy(), ref)


def test_finalize_after_routed_and_shared_calls(fme):
    # DSv3 shape: the routed call's unweighted rows and weights, and the shared expert's out
    cfg, scfg = W.DSV3, W.SHARED
    M, seed = 4, 7
    w13, s13, w2, s2 = W.fp8_weights_device(cfg, seed, DEV)
    sw13, ss13, sw2, ss2 = (torch.from_numpy(np.asarray(t)).to(DEV) for t in W.shared_weights_host(scfg, seed))
    x, logits, bias = W.fp8_activations(cfg, M, seed)
    xd = torch.from_numpy(x).to(DEV).to(torch.bfloat16)
    out, ids, wts = fme.moe_routed_fp8(xd, torch.from_numpy(logits).to(DEV).to(torch.bfloat16),
                                       torch.from_numpy(bias).to(DEV), w13, s13, w2, s2, cfg.top_k, cfg.limit,
                                       cfg.scale, cfg.ue8m0)
    shared = fme.shared_expert_fp8(xd, sw13, ss13, sw2, ss2, scfg.limit, scfg.ue8m0)
    y = fme.moe_finalize(out, wts, shared)
    ref = oracle_finalize(out.float().cpu().numpy(), wts.cpu().numpy(), shared.float().cpu().numpy())
    assert np.array_equal(y.float().cpu().numpy(), ref)
