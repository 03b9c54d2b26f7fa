"""Number formats used by the pages: FP8 E4M3, FP4 E2M1, UE8M0, BF16.

Oracle (test infrastructure only; see the package docstring).

Each decoder is the format's closed form written out; each encoder picks the
nearest representable value by search over the decoded table, with ties to the
even code and saturation at the largest finite magnitude. These are the
readings of the pages' unprinted ``pack_fp8`` helper ("mega_moe":
``_MegaKernel.epilogue`` x-quant and ``hidden_block``) and of "nearest-neighbor
E2M1 quantization" ("nvfp4-megamoe-kernel README.md", Bugs Found & Fixed §2).
"""

import numpy as np

FP8_MAX = 448.0  # largest finite E4M3 magnitude (scale = amax / 448 on both FP8 pages)
FP4_MAX = 6.0  # largest E2M1 magnitude (scale = block_max / 6, nvfp4 README §2)


# --------------------------------------------------------------------------- E4M3
def e4m3_value(code: int) -> float:
    """Value of one E4M3 byte: sign bit 7, exponent bits 6..3 (bias 7), mantissa
    bits 2..0. Exponent 0 is subnormal (m/8 * 2^-6). 0x7F/0xFF are NaN."""
    code = int(code) & 0xFF
    sign = -1.0 if code & 0x80 else 1.0
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return float("nan")
    if e == 0:
        return sign * (m / 8.0) * 2.0**-6
    return sign * (1.0 + m / 8.0) * 2.0 ** (e - 7)


_E4M3_TABLE = np.array([e4m3_value(c) for c in range(256)], dtype=np.float64)
# Non-negative finite magnitudes in code order 0x00..0x7E; strictly increasing.
_E4M3_POS = _E4M3_TABLE[:0x7F].copy()


def e4m3_decode(codes) -> np.ndarray:
    """float64 values of an array of E4M3 bytes."""
    return _E4M3_TABLE[np.asarray(codes, dtype=np.uint8)]


def _nearest_code(mag: np.ndarray, table: np.ndarray) -> np.ndarray:
    """Index into increasing ``table`` nearest to each ``mag`` (>= 0); exact ties
    go to the even index (the even mantissa); beyond the end saturates."""
    hi = np.searchsorted(table, mag, side="left")
    hi = np.minimum(hi, len(table) - 1)
    lo = np.maximum(hi - 1, 0)
    dlo = mag - table[lo]
    dhi = table[hi] - mag
    pick_hi = (dhi < dlo) | ((dhi == dlo) & (hi % 2 == 0))
    idx = np.where(pick_hi, hi, lo)
    idx = np.where(mag >= table[-1], len(table) - 1, idx)
    return idx


def e4m3_encode(values) -> np.ndarray:
    """E4M3 bytes of float32 values: round to nearest, ties to even, finite
    values beyond 448 saturate to +-448 (the ``satfinite`` reading of the
    unprinted ``pack_fp8``). The sign of zero is kept."""
    v = np.asarray(values, dtype=np.float32).astype(np.float64)
    idx = _nearest_code(np.abs(v), _E4M3_POS).astype(np.uint8)
    return np.where(np.signbit(v), idx | 0x80, idx).astype(np.uint8)


# --------------------------------------------------------------------------- E2M1
def e2m1_value(nibble: int) -> float:
    """Value of one E2M1 nibble: bit 3 sign, bits 2..0 magnitude ("nvfp4-megamoe-
    kernel README.md" §2: sign-magnitude 4-bit). Exponent bits 2..1 (bias 1),
    mantissa bit 0; exponent 0 is subnormal (m * 0.5)."""
    nibble = int(nibble) & 0xF
    sign = -1.0 if nibble & 0x8 else 1.0
    e = (nibble >> 1) & 0x3
    m = nibble & 0x1
    if e == 0:
        return sign * m * 0.5
    return sign * (1.0 + m / 2.0) * 2.0 ** (e - 1)


_E2M1_TABLE = np.array([e2m1_value(c) for c in range(16)], dtype=np.float64)
_E2M1_POS = _E2M1_TABLE[:8].copy()


def e2m1_decode(nibbles) -> np.ndarray:
    return _E2M1_TABLE[np.asarray(nibbles, dtype=np.uint8) & 0xF]


def e2m1_encode(values) -> np.ndarray:
    """E2M1 nibbles of float32 values: nearest, ties to even code, saturating
    at +-6 (reading of "nearest-neighbor E2M1 quantization", nvfp4 README §2)."""
    v = np.asarray(values, dtype=np.float32).astype(np.float64)
    idx = _nearest_code(np.abs(v), _E2M1_POS).astype(np.uint8)
    return np.where(np.signbit(v), idx | 0x8, idx).astype(np.uint8)


def fp4_unpack(packed, k: int) -> np.ndarray:
    """Nibbles [..., k] from packed E2M1 bytes [..., k/2]: element 2i in the low
    nibble, 2i+1 in the high nibble ("Data Formats": 2 FP4 values per byte,
    K-major; the page does not fix the nibble order, so this one is a reading)."""
    p = np.asarray(packed, dtype=np.uint8)
    out = np.empty(p.shape[:-1] + (k,), dtype=np.uint8)
    out[..., 0::2] = p & 0xF
    out[..., 1::2] = p >> 4
    return out


# --------------------------------------------------------------------------- UE8M0
def ue8m0_round_up(scale) -> np.ndarray:
    """Smallest power of two >= max(scale, 1e-10) for positive float32 scales:
    the UE8M0 rounding of "mega_moe" x-quant and "shared_expert"
    ``_group_scale`` (when ue8m0). Written as 2^ceil(log2 s) via frexp."""
    s = np.maximum(np.asarray(scale, dtype=np.float32), np.float32(1e-10)).astype(np.float64)
    m, e = np.frexp(s)  # s = m * 2^e, m in [0.5, 1)
    e = np.where(m == 0.5, e - 1, e)
    return np.ldexp(1.0, e).astype(np.float32)


# --------------------------------------------------------------------------- BF16
def bf16_round(values) -> np.ndarray:
    """Round float64/float32 values to the nearest BF16 (ties to even), via
    float32 first; returned as float32 holding the BF16 value."""
    f = np.ascontiguousarray(np.asarray(values, dtype=np.float64).astype(np.float32))
    bits = f.view(np.uint32).astype(np.uint64)
    lsb = (bits >> 16) & 1
    rounded = ((bits + 0x7FFF + lsb) >> 16) << 16
    out = rounded.astype(np.uint32).view(np.float32)
    return np.where(np.isnan(f), f, out)


def bf16_bits(values) -> np.ndarray:
    """uint16 BF16 bit patterns of values already representable in BF16."""
    f = np.ascontiguousarray(np.asarray(values, dtype=np.float32))
    return (f.view(np.uint32) >> 16).astype(np.uint16)


def bf16_from_bits(bits) -> np.ndarray:
    b = np.ascontiguousarray(np.asarray(bits, dtype=np.uint16)).astype(np.uint32)
    return (b << 16).view(np.float32)
