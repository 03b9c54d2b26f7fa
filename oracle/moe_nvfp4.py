"""NVFP4 slot MoE over one local expert range.

Oracle (test infrastructure only; see the package docstring).

"nvfp4-megamoe-kernel README.md": a slot is one (token, top-k expert) pair and
only slots whose expert is local exist; per slot: L1 GEMM (gate; up), SiLU*Mul,
re-quant to FP4, L2 GEMM; the routing weights are applied once, in the final
index-add scatter to [M, hidden] ("Why slots?", Bugs Found & Fixed §6 and §7).
Formats per "Data Formats": packed E2M1 [E_local, N, K/2] (two values per
byte, K-major) with UE4M3 scales [E_local, N, K/16]; L1 rows are a plain
concatenation [gate; up] (Bugs Found & Fixed §4).

Readings where the page is silent: both GEMMs return BF16 (the page re-quantises
"L1 BF16 output"); SiLU*Mul is computed in float64 and rounded once to BF16;
``limit`` clamps like the FP8 path when finite and is +inf by default (the page
states no clamp); the scatter sums the slots of a token in ascending top-k
order in float32 (weight times BF16 slot output) and rounds once to BF16.
"""

import numpy as np

from .codecs import e2m1_decode, e4m3_decode, fp4_unpack, bf16_round
from .quant import FP4_GROUP, nvfp4_quant
from .moe_fp8 import clamped_swiglu


def fp4_block_scaled_gemv(w_packed, w_sbytes, a_nibbles, a_sbytes):
    """y[n] = sum_g (sum_{k in g} dec(w[n,k]) * dec(a[k])) * dec(sw[n,g]) * dec(sa[g]).

    The native NVFP4 block-scaled product: every E2M1 weight and activation
    carries its own UE4M3 group-16 scale ("Data Formats"). Per-group partial
    sums and scale products are exact in float64.

    Args: w_packed [N, K/2] uint8, w_sbytes [N, K/16] uint8 (E4M3 bytes),
        a_nibbles [K] uint8, a_sbytes [K/16] uint8.
    Returns: [N] float64.
    """
    w_packed = np.asarray(w_packed)
    N = w_packed.shape[0]
    K = w_packed.shape[1] * 2
    ng = K // FP4_GROUP
    W = e2m1_decode(fp4_unpack(w_packed, K)).reshape(N, ng, FP4_GROUP)
    a = e2m1_decode(a_nibbles).reshape(ng, FP4_GROUP)
    P = np.einsum("ngk,gk->ng", W, a)
    S = e4m3_decode(w_sbytes) * e4m3_decode(a_sbytes)[None, :]
    return (P * S).sum(axis=1)


def routed_nvfp4(x, ids, weights, w13, s13, w2, s2, e0: int, n_local: int,
                 limit: float = float("inf")):
    """Slot MoE for experts [e0, e0 + n_local).

    Args:
        x: [M, H] float32 holding BF16 tokens.
        ids: [M, k] int32 global expert ids; weights: [M, k] float32.
        w13: indexable by local expert -> packed [2N, H/2] uint8 (gate; up).
        s13: -> [2N, H/16] uint8 UE4M3.  w2: -> [H, N/2] uint8.  s2: -> [H, N/16].
        e0, n_local: the local expert range.
        limit: SwiGLU clamp (+inf: none).

    Returns: y [M, H] float32 holding BF16 values (zero rows for tokens with no
        local slot).
    """
    x = np.asarray(x, dtype=np.float32)
    ids = np.asarray(ids)
    weights = np.asarray(weights, dtype=np.float32)
    M, H = x.shape
    k = ids.shape[1]
    xq, xs = nvfp4_quant(x)
    y = np.zeros((M, H), dtype=np.float32)
    for t in range(M):
        acc = np.zeros(H, dtype=np.float32)
        for r in range(k):
            e = int(ids[t, r])
            if not (e0 <= e < e0 + n_local):
                continue  # non-local slot: does not exist on this rank
            le = e - e0
            W1 = np.asarray(w13[le])
            n_inter = W1.shape[0] // 2
            g1 = bf16_round(fp4_block_scaled_gemv(W1, s13[le], xq[t], xs[t]))
            gate, up = g1[:n_inter], g1[n_inter:]
            h = bf16_round(clamped_swiglu(gate, up, limit))
            hq, hs = nvfp4_quant(h)
            o = bf16_round(fp4_block_scaled_gemv(w2[le], s2[le], hq, hs))
            acc = (acc + (weights[t, r] * o).astype(np.float32)).astype(np.float32)
        y[t] = bf16_round(acc)
    return y
