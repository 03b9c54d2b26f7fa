"""Per-token top-k routing with a selection-only score-correction bias.

Oracle (test infrastructure only; see the package docstring).

Follows "vllm.models.glm5next.nvidia.specialized_decode.mega_moe",
``_MegaKernel.top_k_pick`` and its docstring: sigmoid scores of the router
logits; top-k by score plus bias with ties going to the lower expert; the
picked experts in descending key order; each weight is its unbiased score over
the float sum of the picked scores (summed in pick order), times ``scale``.

Reading (the page uses an approximate exp/divide "a few ulp" off): the oracle
takes the correctly rounded float32 sigmoid (computed in float64, rounded once).
The key is ``float32(score + bias)``; the weight is ``float32(score / total)``
then a float32 multiply by ``scale``.
"""

import numpy as np


def sigmoid_f32(logits) -> np.ndarray:
    """float32(1 / (1 + exp(-l))) computed in float64 and rounded once."""
    l = np.asarray(logits, dtype=np.float32).astype(np.float64)
    with np.errstate(over="ignore"):
        s = 1.0 / (1.0 + np.exp(-l))
    return s.astype(np.float32)


def route(logits, bias, top_k: int, scale: float):
    """Route every token.

    Args:
        logits: [M, E] router logits as float32 (BF16 logits widen exactly).
        bias: [E] float32 score-correction bias, used for selection only.
        top_k: experts per token.
        scale: routed scaling factor applied after renormalisation.

    Returns:
        ids [M, top_k] int32 in descending key order, weights [M, top_k] float32,
        keys [M, E] float32 (for tie-gap diagnostics).
    """
    logits = np.asarray(logits, dtype=np.float32)
    bias = np.asarray(bias, dtype=np.float32)
    M, E = logits.shape
    scores = sigmoid_f32(logits)
    keys = (scores + bias[None, :]).astype(np.float32)  # float32 add, RN
    ids = np.empty((M, top_k), dtype=np.int32)
    weights = np.empty((M, top_k), dtype=np.float32)
    for t in range(M):
        # Descending key, ties to the lower expert id.
        order = sorted(range(E), key=lambda e: (-float(keys[t, e]), e))[:top_k]
        ids[t] = order
        total = np.float32(0.0)
        for e in order:  # float sum in pick order
            total = np.float32(total + scores[t, e])
        for r, e in enumerate(order):
            w = np.float32(scores[t, e] / total)
            weights[t, r] = np.float32(w * np.float32(scale))
    return ids, weights, keys


def selection_gap(keys, ids) -> np.ndarray:
    """Per token, the float gap between the k-th picked key and the best
    unpicked key (inf when every expert is picked). A gap of a few float32 ulp
    means a sigmoid evaluated a few ulp differently could swap the pick."""
    keys = np.asarray(keys, dtype=np.float32)
    M, E = keys.shape
    gaps = np.full(M, np.inf)
    for t in range(M):
        picked = set(int(e) for e in ids[t])
        rest = [keys[t, e] for e in range(E) if e not in picked]
        kth = min(keys[t, e] for e in picked)
        if rest:
            gaps[t] = float(kth) - float(max(rest))
        # Gaps between consecutive picked keys decide the order of ids too.
        ordered = [float(keys[t, e]) for e in ids[t]]
        for a, b in zip(ordered, ordered[1:]):
            gaps[t] = min(gaps[t], a - b)
    return gaps
