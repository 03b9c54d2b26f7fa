"""Failure detection on the GPU without a fault: the kernels' bounded waits
give up on a flag nothing sets and report through the workspace error word,
and the context stays usable afterwards."""

import ctypes
import time

import numpy as np
import pytest
import torch

from oracle import moe_fp8
from synth import workloads as W
from tests.parity import assert_outputs

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module")
def fme():
    import fp4_moe_expert_gb300 as m
    return m


def test_bounded_waits_time_out_and_report(fme):
    ws = fme.Workspace(4096, DEV)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    t0 = time.perf_counter()
    assert fme.lib.fme_selftest_wait_timeout(ws.ptr(), 4096, 20, stream) == 0
    code = ws.error()  # synchronises
    elapsed = time.perf_counter() - t0
    assert code == 3, code  # cross-CTA wait (2) and mbarrier wait (1) both gave up
    assert elapsed < 5.0
    assert ws.error() == 0  # reading cleared it
    # The context is intact: a normal layer call still matches the oracle.
    cfg = W.TINY
    w13h, w2h = W.fp8_weights_host(cfg, 1)
    s13, s2 = W.fp8_weight_scales(cfg, 1)
    x, logits, bias = W.fp8_activations(cfg, 1, 1)
    out, ids, wts = fme.moe_routed_fp8(torch.from_numpy(x).to(DEV).to(torch.bfloat16),
                                       torch.from_numpy(logits).to(DEV), torch.from_numpy(bias).to(DEV),
                                       torch.from_numpy(w13h.full()).to(DEV), torch.from_numpy(s13).to(DEV),
                                       torch.from_numpy(w2h.full()).to(DEV), torch.from_numpy(s2).to(DEV),
                                       cfg.top_k, cfg.limit, cfg.scale, cfg.ue8m0)
    torch.cuda.synchronize()
    ref, rids, _, _ = moe_fp8.routed_fp8(x, logits, bias, w13h, s13, w2h, s2, cfg.top_k, cfg.limit, cfg.scale,
                                         cfg.ue8m0)
    assert np.array_equal(ids.cpu().numpy(), rids)
    assert_outputs(out.float().cpu().numpy(), ref)


def test_selftest_argument_checks(fme):
    ws = fme.Workspace(4096, DEV)
    assert fme.lib.fme_selftest_wait_timeout(ws.ptr(), 100, 20, None) == -6
    assert fme.lib.fme_selftest_wait_timeout(ws.ptr(), 4096, 0, None) == -1
