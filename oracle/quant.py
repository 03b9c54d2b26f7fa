"""Activation quantisers: FP8 E4M3 per 128 and NVFP4 E2M1 per 16.

Oracle (test infrastructure only; see the package docstring).
"""

import numpy as np

from .codecs import FP8_MAX, FP4_MAX, e4m3_encode, e4m3_decode, e2m1_encode, ue8m0_round_up

GROUP = 128  # FP8 block size of every K and row block on both FP8 pages
FP4_GROUP = 16  # NVFP4 scale group ("Data Formats": 1 scale per 16 FP4 values)


def fp8_group_scale(amax, ue8m0: bool):
    """Scale and its inverse for blocks with the given |max|.

    "shared_expert" ``_group_scale`` (and the same rule in "mega_moe"
    ``_MegaKernel.epilogue`` x-quant): scale = max(amax, 1e-10) / 448 divided
    in float32; when ue8m0, rounded up to a power of two from
    max(scale, 1e-10); inverse = float32(1 / scale), exact for a power of two.
    """
    amax = np.maximum(np.asarray(amax, dtype=np.float32), np.float32(1e-10))
    scale = (amax / np.float32(FP8_MAX)).astype(np.float32)
    if ue8m0:
        scale = ue8m0_round_up(scale)
    inverse = (np.float32(1.0) / scale).astype(np.float32)
    return scale, inverse


def fp8_quant_mul(values, ue8m0: bool):
    """Per-128 FP8 quantisation by multiplying with the inverse scale.

    Used for the routed x ("mega_moe" epilogue head: ``values * inverse``) and
    for both quantisations of "shared_expert" (``v * inverse``).

    Args: values [..., K] float32 (K a multiple of 128).
    Returns: codes uint8 [..., K], scales float32 [..., K/128].
    """
    v = np.asarray(values, dtype=np.float32)
    blocks = v.reshape(v.shape[:-1] + (v.shape[-1] // GROUP, GROUP))
    amax = np.abs(blocks).max(axis=-1)
    scale, inverse = fp8_group_scale(amax, ue8m0)
    scaled = (blocks * inverse[..., None]).astype(np.float32)
    codes = e4m3_encode(scaled).reshape(v.shape)
    return codes, scale


def fp8_quant_div(values, ue8m0: bool):
    """Per-128 FP8 quantisation by dividing by the scale.

    "mega_moe" ``_MegaKernel.hidden_block``: scale = max(amax, 1e-10) / 448 and
    codes of ``act / scale``. The page does not round this scale; here it is
    rounded up to a power of two when ue8m0 (the workload states that every
    activation scale is rounded), where division and inverse-multiply agree.
    """
    v = np.asarray(values, dtype=np.float32)
    blocks = v.reshape(v.shape[:-1] + (v.shape[-1] // GROUP, GROUP))
    amax = np.abs(blocks).max(axis=-1)
    scale, _ = fp8_group_scale(amax, ue8m0)
    scaled = (blocks / scale[..., None]).astype(np.float32)
    codes = e4m3_encode(scaled).reshape(v.shape)
    return codes, scale


def nvfp4_quant(values):
    """BF16 -> E2M1 per group of 16 with a UE4M3 scale.

    "nvfp4-megamoe-kernel README.md", Bugs Found & Fixed §2 (``stage_activation``):
    the stored scale is block_max / 6 as a UE4M3 byte and the same stored value
    is the divisor; values are signed E2M1 by nearest neighbour. Readings:
    block_max / 6 is a float32 division, rounded to E4M3 (RN-even, saturating);
    the divisor is the decoded stored byte; a group whose stored scale decodes
    to zero quantises to zeros.

    Args: values [..., K] float32 (K a multiple of 16).
    Returns: nibbles uint8 [..., K], scale bytes uint8 [..., K/16].
    """
    v = np.asarray(values, dtype=np.float32)
    g = v.reshape(v.shape[:-1] + (v.shape[-1] // FP4_GROUP, FP4_GROUP))
    amax = np.abs(g).max(axis=-1).astype(np.float32)
    sbytes = e4m3_encode((amax / np.float32(FP4_MAX)).astype(np.float32))
    divisor = e4m3_decode(sbytes).astype(np.float32)
    safe = np.where(divisor > 0, divisor, np.float32(1.0)).astype(np.float32)
    scaled = (g / safe[..., None]).astype(np.float32)
    scaled = np.where((divisor > 0)[..., None], scaled, np.float32(0.0))
    nibbles = e2m1_encode(scaled).reshape(v.shape)
    return nibbles, sbytes
