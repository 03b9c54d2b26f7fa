"""Local finalize of the routed layer: the routing-weighted sum of a token's
unweighted expert rows, plus the shared expert's row.

Oracle (test infrastructure only; see the package docstring).

"vllm.models.glm5next.nvidia.specialized_decode.mega_moe" (the routed kernel
writes unweighted rows t * top_k + r and the routing weights; a finalize step
publishes the weighted sum) and
"vllm.models.kimi_k3.nvidia.specialized_decode.cutedsl.moe.ep.comm"
(EpCombine: the routing-weighted sum, an FP32 sum in a fixed order, rounded
once to BF16). Readings where the pages are silent: products and sums are
separate FP32 operations (no fused multiply-add), in ascending r; the shared
expert's row is added after the routed sum; one BF16 rounding at the end.
"""

import numpy as np

from .codecs import bf16_round


def finalize(out, weights, shared_out=None):
    """y[t, m] = bf16(((w[t,0]*out[t*k+0, m] + w[t,1]*out[t*k+1, m]) + ...) + shared_out[t, m]).

    Args:
        out: [M * k, H] float32 holding BF16 values (rows in route order).
        weights: [M, k] float32 routing weights.
        shared_out: [M, H] float32 holding BF16 values, or None.
    Returns: y [M, H] float32 holding BF16 values.
    """
    w = np.asarray(weights, dtype=np.float32)
    M, k = w.shape
    o = np.asarray(out, dtype=np.float32).reshape(M, k, -1)
    acc = np.zeros((M, o.shape[2]), dtype=np.float32)
    for r in range(k):
        term = (w[:, r:r + 1] * o[:, r, :]).astype(np.float32)  # one FP32 rounding
        acc = (acc + term).astype(np.float32)                   # one FP32 rounding
    if shared_out is not None:
        acc = (acc + np.asarray(shared_out, dtype=np.float32)).astype(np.float32)
    return bf16_round(acc)
