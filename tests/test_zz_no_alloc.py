"""The allocation-free routed FP8 entry point (fme_moe_routed_fp8_noalloc).

It serves callers that cannot call cudaMalloc (they run inside someone
else's memory pool, in a host that forbids device allocations, or during
graph capture) and so cannot pass a workspace. The test calls it through the
C ABI twice in a row, with different inputs, and checks each result against
the regular entry point's on the same inputs. This file is collected last so
that a run stopping at the first failure has run every other test already.
"""

import ctypes

import numpy as np
import pytest
import torch

from synth import workloads as W
from tests.parity import assert_outputs

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module")
def fme():
    import __graft_entry__
    __graft_entry__.build()
    import fp4_moe_expert_gb300 as m
    return m


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def test_noalloc_matches_workspace_entry_point_twice(fme):
    cfg = W.RAGGED  # H 1024, I 384, 40 experts, top_k 3
    M = 5
    w13h, w2h = W.fp8_weights_host(cfg, 31)
    s13, s2 = W.fp8_weight_scales(cfg, 31)
    w13 = torch.from_numpy(w13h.full()).to(DEV)
    w2 = torch.from_numpy(w2h.full()).to(DEV)
    s13d, s2d = torch.from_numpy(s13).to(DEV), torch.from_numpy(s2).to(DEV)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for step in range(2):
        x, logits, bias = W.fp8_activations(cfg, M, 31, step)
        xd = torch.from_numpy(x).to(DEV).to(torch.bfloat16)
        ld = torch.from_numpy(logits).to(DEV)
        bd = torch.from_numpy(bias).to(DEV)
        ref_out, ref_ids, ref_w = fme.moe_routed_fp8(xd, ld, bd, w13, s13d, w2, s2d, cfg.top_k, cfg.limit,
                                                     cfg.scale, cfg.ue8m0)
        out = torch.empty(M * cfg.top_k, cfg.H, dtype=torch.bfloat16, device=DEV)
        ids = torch.empty(M, cfg.top_k, dtype=torch.int32, device=DEV)
        wts = torch.empty(M, cfg.top_k, dtype=torch.float32, device=DEV)
        rc = fme.lib.fme_moe_routed_fp8_noalloc(_p(xd), _p(ld), fme.FME_F32, _p(bd), _p(w13), _p(s13d), _p(w2),
                                                _p(s2d), M, cfg.H, cfg.I, cfg.E, cfg.top_k, cfg.limit, cfg.scale,
                                                int(cfg.ue8m0), _p(out), _p(ids), _p(wts), stream)
        assert rc == 0, fme.lib.fme_last_error().decode()
        torch.cuda.synchronize()
        assert torch.equal(ids, ref_ids)
        assert np.allclose(wts.cpu().numpy(), ref_w.cpu().numpy(), rtol=1e-6, atol=0)
        assert_outputs(out.float().cpu().numpy(), ref_out.float().cpu().numpy(), f"call {step}")
    # Both calls finished without a device-side error: the variant's own error
    # word (in the static array, not in any workspace) reads zero.
    code = ctypes.c_int(-1)
    rc = fme.lib.fme_moe_routed_fp8_noalloc_error(ctypes.byref(code), stream)
    assert rc == 0 and code.value == 0, fme.lib.fme_last_error().decode()


def test_noalloc_rejects_requests_beyond_its_scratch(fme):
    null = ctypes.c_void_p(16)
    # Latent shape, 64 tokens x top_k 16: about 68.4 MiB of workspace > 64 MiB
    rc = fme.lib.fme_moe_routed_fp8_noalloc(null, null, 0, null, null, null, null, null, 64, 3584, 2048, 896,
                                            16, 7.0, 1.0, 0, null, null, null, None)
    assert rc == -2
    assert "64 MiB" in fme.lib.fme_last_error().decode()
