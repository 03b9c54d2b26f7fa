"""The single-GPU forms of the expert-parallel dispatch quantiser and of the
combine's reduction with RMSNorm.

Oracle (test infrastructure only; see the package docstring).

"vllm.models.kimi_k3.nvidia.specialized_decode.cutedsl.moe.ep.comm":
EpDispatch quantises the BF16 latent to MXFP8 (E4M3 values, one E8M0 scale per
32 values, scales in row order); EpCombine sums the per-rank BF16 partials of a
token in rank order in FP32, rounds once to BF16 (the routed latent), then
applies vLLM's RMSNorm: the FP32 sum of squares of the BF16 latent,
rstd = rsqrt(sum / H + eps), out = x * rstd * w rounded once to BF16.

Readings where the page is silent (``mx_exponent`` and ``mx_rescale`` are not
printed): the shared exponent follows the OCP MX rule, floor(log2(amax)) minus
8 (the largest E4M3 exponent), clamped to the E8M0 range [-127, 127]; a block
whose amax is zero (or subnormal below 2^-119) takes exponent -127; each value
is multiplied by 2^-exponent and encoded as E4M3 round-to-nearest-even with
saturation at 448. RMSNorm: the page takes an approximate rsqrt, so its
result is the exact one within a few FP32 ulp; the oracle evaluates the sum of
squares and rsqrt in float64.
"""

import math

import numpy as np

from .codecs import bf16_round, e4m3_encode

MX_BLOCK = 32
E4M3_EMAX = 8


def mx_exponent(amax: float) -> int:
    """Shared exponent of one block: floor(log2(amax)) - 8, clamped to [-127, 127]."""
    if not amax > 0.0:
        return -127
    m, e = math.frexp(amax)  # amax = m * 2^e, m in [0.5, 1)
    return max(-127, min(127, (e - 1) - E4M3_EMAX))


def mxfp8_quantize(x):
    """x [T, H] float32 holding BF16 values, H a multiple of 32 ->
    (codes [T, H] uint8 E4M3, scales [T, H/32] uint8 E8M0 = exponent + 127)."""
    x = np.asarray(x, dtype=np.float32)
    T, H = x.shape
    blocks = x.reshape(T, H // MX_BLOCK, MX_BLOCK)
    codes = np.zeros_like(blocks, dtype=np.uint8)
    scales = np.zeros((T, H // MX_BLOCK), dtype=np.uint8)
    for t in range(T):
        for b in range(H // MX_BLOCK):
            v = blocks[t, b].astype(np.float64)
            e = mx_exponent(float(np.max(np.abs(v))))
            scales[t, b] = e + 127
            codes[t, b] = e4m3_encode((v * 2.0 ** -e).astype(np.float32))
    return codes.reshape(T, H), scales


def combine_rmsnorm(partials, gamma, eps: float = 1e-5):
    """partials [T, N, H] float32 holding BF16 values (rank order), gamma [H]
    (BF16 values) -> (latent [T, H], normed [T, H]), both BF16 values as float32."""
    p = np.asarray(partials, dtype=np.float32)
    T, N, H = p.shape
    acc = np.zeros((T, H), dtype=np.float32)
    for d in range(N):
        acc = (acc + p[:, d, :]).astype(np.float32)
    latent = bf16_round(acc)
    lat = latent.astype(np.float64)
    rstd = 1.0 / np.sqrt((lat * lat).sum(axis=1, keepdims=True) / H + eps)
    normed = bf16_round(lat * rstd * np.asarray(gamma, dtype=np.float64)[None, :])
    return latent, normed
