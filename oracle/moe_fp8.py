"""Routed FP8 MoE layer and the FP8 shared expert.

Oracle (test infrastructure only; see the package docstring).

Block sums of decoded E4M3 products are taken in float64, where every product
and every partial sum of 128 of them is exact; the FP32 block-scale products
are formed in float32 as on the pages; the scaled block sums are added in
float64 and rounded once.
"""

import numpy as np

from .codecs import e4m3_decode, bf16_round
from .quant import GROUP, fp8_quant_mul, fp8_quant_div
from .routing import route


def block_scaled_gemv(w_codes, w_scales, a_codes, a_scales, row_idx=None):
    """y[n] = sum_b P[n, b] * float32(w_scale[n/128, b] * a_scale[b]).

    P[n, b] = sum over the 128 k of block b of dec(W[n, k]) * dec(a[k]).
    "mega_moe" ``_MegaKernel.epilogue`` (GEMM1: per K-block column times
    ``w_scale * x_scale``, summed; GEMM2 likewise with the hidden scale) and
    "shared_expert" ``_GateUpKernel`` / ``_DownKernel`` (``part * combined``).

    Args:
        w_codes: [N, K] uint8 E4M3, w_scales: [N/128, K/128] float32,
        a_codes: [K] uint8 E4M3, a_scales: [K/128] float32.
        row_idx: when w_codes holds a subset of rows, their row numbers n
            (each row keeps the scale of its own 128-row block).
    Returns: [N] float64 (not yet rounded).
    """
    w_codes = np.asarray(w_codes)
    N, K = w_codes.shape
    nb = K // GROUP
    W = e4m3_decode(w_codes).reshape(N, nb, GROUP)
    a = e4m3_decode(a_codes).reshape(nb, GROUP)
    P = np.einsum("nbk,bk->nb", W, a)
    ws = np.asarray(w_scales, dtype=np.float32)
    rows = (np.arange(N) if row_idx is None else np.asarray(row_idx)) // GROUP
    S = (ws[rows, :] * np.asarray(a_scales, dtype=np.float32)[None, :]).astype(np.float32)
    return (P * S.astype(np.float64)).sum(axis=1)


def mx_block_scaled_gemv(w_codes, w_scales, a_codes, a_e8m0):
    """y[n] = sum over K blocks b and their 32-value blocks s of
    P[n, b, s] * float32(w_scale[n/128, b] * 2^(a_e8m0[b, s] - 127)).

    The GEMV of MXFP8 activations (E4M3 values, one E8M0 scale per 32 values,
    "vllm.models.kimi_k3.nvidia.specialized_decode.cutedsl.moe.ep.comm"
    EpDispatch's format) with the routed weights' FP32 block-128 scales
    ("mega_moe"). Reading: the pages do not print this product; each 32-value
    block's exact partial sum takes its own scale product, as the MX format
    defines, and the sums are exact (float64 here).

    Args: w_codes [N, K] uint8 E4M3, w_scales [N/128, K/128] float32,
        a_codes [K] uint8 E4M3, a_e8m0 [K/32] uint8.
    Returns: [N] float64.
    """
    w_codes = np.asarray(w_codes)
    N, K = w_codes.shape
    nb = K // GROUP
    W = e4m3_decode(w_codes).reshape(N, nb, 4, GROUP // 4)
    a = e4m3_decode(a_codes).reshape(nb, 4, GROUP // 4)
    P = np.einsum("nbsk,bsk->nbs", W, a)
    ws = np.asarray(w_scales, dtype=np.float32)[np.arange(N) // GROUP, :]
    ax = np.exp2(np.asarray(a_e8m0, dtype=np.float64).reshape(nb, 4) - 127.0)
    S = (ws[:, :, None].astype(np.float64) * ax[None, :, :]).astype(np.float32)
    return (P * S.astype(np.float64)).sum(axis=(1, 2))


def clamped_swiglu(gate, up, limit):
    """silu(min(gate, limit)) * clamp(up, -limit, limit) in float64.

    "mega_moe" ``_MegaKernel.hidden_block``: gate = min(g, limit), up clamped to
    [-limit, limit], act = gate / (1 + exp(-gate)) * up. ``limit = inf`` gives
    the unclamped textbook silu(g) * u.
    """
    g = np.minimum(np.asarray(gate, dtype=np.float64), limit)
    u = np.clip(np.asarray(up, dtype=np.float64), -limit, limit)
    with np.errstate(over="ignore"):
        return g / (1.0 + np.exp(-g)) * u


def routed_fp8(x, logits, bias, w13, s13, w2, s2, top_k, limit, scale, ue8m0,
               hidden_ue8m0=None, routes=None, rows=None, x_mx=None, exact=False):
    """Routed experts of a few decode tokens ("mega_moe" ``MegaExperts.__call__``).

    Args:
        x: [M, H] float32 holding BF16 tokens.
        logits: [M, E] float32 (BF16 logits widen exactly); bias: [E] float32.
        w13: indexable by expert -> [2I, H] uint8 E4M3, up rows then gate rows.
        s13: indexable by expert -> [2I/128, H/128] float32.
        w2: indexable by expert -> [H, I] uint8 E4M3; s2 -> [H/128, I/128].
        top_k, limit, scale, ue8m0: as on the page's constructor.
        hidden_ue8m0: rounding of the hidden scale (default: ``ue8m0``).
        routes: optional iterable of route indices t*top_k + r to evaluate.
        rows: optional array of output rows m to evaluate (sampling).
        x_mx: optional MXFP8 activations (codes [M, H] uint8 E4M3, scales
            [M, H/32] uint8 E8M0) used by GEMM1 instead of quantising x
            (x then only gives M and H).
        exact: also return the float64 GEMM2 results before their BF16
            rounding (where a BF16 rounding decision sits on a tie, which of
            the two neighbours a summation in another order picks is open).

    Returns:
        out [M*top_k, H] float32 holding BF16 values (NaN where not evaluated),
        ids [M, top_k] int32, weights [M, top_k] float32, keys [M, E] float32
        (and with ``exact`` the unrounded out [M*top_k, H] float64).
    """
    x = np.asarray(x, dtype=np.float32)
    M, H = x.shape
    if hidden_ue8m0 is None:
        hidden_ue8m0 = ue8m0
    ids, weights, keys = route(logits, bias, top_k, scale)
    # x-quant: "mega_moe" epilogue head, per 128-K block, values * inverse.
    xq, sx = fp8_quant_mul(x, ue8m0)
    out = np.full((M * top_k, H), np.nan, dtype=np.float32)
    unrounded = np.full((M * top_k, H), np.nan, dtype=np.float64)
    routes = range(M * top_k) if routes is None else routes
    row_idx = np.arange(H) if rows is None else np.asarray(rows)
    for route_i in routes:
        t, r = divmod(int(route_i), top_k)
        e = int(ids[t, r])
        W1 = np.asarray(w13[e])
        inter = W1.shape[0] // 2
        if x_mx is None:
            y = block_scaled_gemv(W1, s13[e], xq[t], sx[t]).astype(np.float32)
        else:
            y = mx_block_scaled_gemv(W1, s13[e], x_mx[0][t], x_mx[1][t]).astype(np.float32)
        # W31 row order: up rows, then gate rows ("mega_moe" module docstring).
        up, gate = y[:inter], y[inter:]
        h = clamped_swiglu(gate, up, limit).astype(np.float32)
        qh, sh = fp8_quant_div(h, hidden_ue8m0)
        W2 = np.asarray(w2[e])[row_idx]
        S2 = np.asarray(s2[e])
        y2 = block_scaled_gemv(W2, S2, qh, sh, row_idx=row_idx)
        out[route_i, row_idx] = bf16_round(y2)
        unrounded[route_i, row_idx] = y2
    if exact:
        return out, ids, weights, keys, unrounded
    return out, ids, weights, keys


def shared_fp8(x, w13, s13, w2, s2, limit, ue8m0):
    """Shared expert ("shared_expert" ``SharedExpert.__call__``).

    gate_up = BF16(block-scaled GEMV of FP8 x), gate rows first then up rows
    (``_DownKernel``: gates at the row base, ups at base + inter); h =
    BF16(silu(min(g, L)) * clamp(u)) with an IEEE divide and accurate exp;
    FP8 per-128 re-quant by ``_group_scale`` (ue8m0 per flag, times the
    inverse); out = BF16(block-scaled GEMV of the down weight).

    Args: x [M, H] float32 (BF16 values); w13 [2I, H] uint8; s13 [2I/128, H/128];
        w2 [H, I] uint8; s2 [H/128, I/128].
    Returns: out [M, H] float32 (BF16 values), gate_up [M, 2I] float32 (BF16).
    """
    x = np.asarray(x, dtype=np.float32)
    M, H = x.shape
    w13 = np.asarray(w13)
    inter = w13.shape[0] // 2
    xq, sx = fp8_quant_mul(x, ue8m0)
    gate_up = np.stack([bf16_round(block_scaled_gemv(w13, s13, xq[t], sx[t]))
                        for t in range(M)])
    gate, up = gate_up[:, :inter], gate_up[:, inter:]
    h = bf16_round(clamped_swiglu(gate, up, limit))
    qh, sh = fp8_quant_mul(h, ue8m0)
    out = np.stack([bf16_round(block_scaled_gemv(w2, s2, qh[t], sh[t]))
                    for t in range(M)])
    return out, gate_up


def ue8m0_unpack(packed, n: int, k: int):
    """FP32 [n/128, k/128] block scales from packed UE8M0 int32 [n, k/512].

    "shared_expert" ``block_scales``: byte g % 4 of column g // 4 holds the
    exponent of K group g; the exponent must be uniform inside each 128-row
    block; the value is the float32 whose bits are exponent << 23.
    Raises ValueError when a 128-row block is not uniform.
    """
    p = np.ascontiguousarray(np.asarray(packed, dtype=np.int32)).view(np.uint32)
    groups = k // GROUP
    g = np.arange(groups)
    exps = (p[:, g // 4] >> (8 * (g % 4)).astype(np.uint32)) & 0xFF  # [n, groups]
    blocks = exps.reshape(n // GROUP, GROUP, groups)
    if not (blocks == blocks[:, :1, :]).all():
        raise ValueError("scales vary inside a 128-row block")
    return (blocks[:, 0, :].astype(np.uint32) << 23).view(np.float32)
