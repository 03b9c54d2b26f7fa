"""GPU parity of the MXFP8 quantiser and the combine + RMSNorm against the oracle."""

import numpy as np
import pytest
import torch

from oracle import codecs
from oracle.ep_local import combine_rmsnorm as oracle_combine, mxfp8_quantize as oracle_mx

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module")
def fme():
    import fp4_moe_expert_gb300 as m
    return m


@pytest.mark.parametrize("T,H,scale", [(1, 3584, 1.0), (5, 3584, 1e3), (16, 96, 1e-30), (3, 7168, 2.0 ** 100)])
def test_mxfp8_bit_exact(fme, T, H, scale):
    rng = np.random.default_rng(T * 7 + H)
    x = codecs.bf16_round((rng.normal(size=(T, H)) * scale).astype(np.float32))
    x[0, :32] = 0.0                      # a zero block
    x[-1, 32:64] = x[-1, 32:64] * 1e-38  # a (sub)normal-amax block
    x = codecs.bf16_round(x)
    q, sc = fme.mxfp8_quantize(torch.from_numpy(x).to(DEV).to(torch.bfloat16))
    rq, rsc = oracle_mx(x)
    assert np.array_equal(sc.cpu().numpy(), rsc)
    assert np.array_equal(q.cpu().numpy(), rq)


@pytest.mark.parametrize("T,N,H", [(1, 1, 3584), (5, 16, 3584), (3, 4, 136), (2, 2, 8192)])
def test_combine_rmsnorm(fme, T, N, H):
    rng = np.random.default_rng(T * 100 + N)
    p = codecs.bf16_round(rng.normal(size=(T, N, H)).astype(np.float32))
    g = codecs.bf16_round(rng.uniform(0.5, 1.5, size=H).astype(np.float32))
    lat, nrm = fme.combine_rmsnorm(torch.from_numpy(p).to(DEV).to(torch.bfloat16),
                                   torch.from_numpy(g).to(DEV).to(torch.bfloat16), 1e-5)
    rl, rn = oracle_combine(p, g, 1e-5)
    assert np.array_equal(lat.float().cpu().numpy(), rl)  # rank-order FP32 sum, one rounding: exact
    got = nrm.float().cpu().numpy()
    ulp = np.maximum(np.abs(rn), 2.0 ** -126) * 2.0 ** -7
    assert np.all(np.abs(got - rn) <= 2 * ulp)  # approximate rsqrt and summation order of the squares
