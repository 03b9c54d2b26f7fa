"""Seeded synthetic inputs for the routed-expert MoE decode layer.

This module serves both sides of every parity check (the CPU oracle and the
CUDA library) and holds none of the method's arithmetic: it only draws bytes
and floats with the distributions the workloads state.

Randomness is counter-based so any expert, row or column can be regenerated on
the host bit-identically to a device-side fill of the whole tensor:

    base   = mix64(seed << 32 | tensor << 24 | expert)
    word_i = mix64(base + (i + 1) * GAMMA) >> 32      (i = element index)

``mix64`` and ``GAMMA`` are the SplitMix64 output function and increment
(Steele, Lea and Flood, "Fast splittable pseudorandom number generators",
OOPSLA 2014), so ``word_i`` is output number i of a SplitMix64 stream seeded
at ``base``. A byte code is drawn from a 256-entry table of cumulative
thresholds over 2^32: code = the first c with word < T[c]. The CUDA fill in
``synth/csrc/synth.cu`` implements the same definition.
"""

import math

import numpy as np

GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

# Tensor ids of the counter streams.
T_W13, T_W2, T_S13, T_S2, T_SW13, T_SW2 = 1, 2, 3, 4, 5, 6


def mix64(z):
    z = np.asarray(z, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def stream_base(seed: int, tensor: int, expert: int) -> np.uint64:
    key = ((int(seed) & 0xFFFFFFFF) << 32) | ((int(tensor) & 0xFF) << 24) | (int(expert) & 0xFFFFFF)
    return mix64(np.array([key], dtype=np.uint64))[0]


def words(seed: int, tensor: int, expert: int, index) -> np.ndarray:
    """uint32 word for each element index (any shape) of one expert's tensor."""
    base = stream_base(seed, tensor, expert)
    i = np.asarray(index, dtype=np.uint64)
    with np.errstate(over="ignore"):
        state = base + (i + np.uint64(1)) * GAMMA
    return (mix64(state) >> np.uint64(32)).astype(np.uint32)


def codes_from_words(w, table) -> np.ndarray:
    """Byte codes: first c with w < table[c] (table: uint64 cumulative, T[255] = 2^32)."""
    return np.searchsorted(np.asarray(table, dtype=np.uint64), np.asarray(w, dtype=np.uint64),
                           side="right").astype(np.uint8)


# --------------------------------------------------------------------------- tables
def _fp8_values() -> np.ndarray:
    """Values of the 256 FP8 E4M3 bytes, read through torch's float8 dtype (a
    library decoder, so this module carries no format arithmetic of its own)."""
    import torch

    return torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn) \
        .to(torch.float64).numpy()


def _cumulative(p: np.ndarray) -> np.ndarray:
    p = np.asarray(p, dtype=np.float64)
    p = p / p.sum()
    c = np.cumsum(p)
    t = np.round(c * 2.0**32).astype(np.uint64)
    # The last code with non-zero probability takes the rounding remainder, so
    # zero-probability codes (the NaN bytes) can never be drawn.
    last = int(np.nonzero(p)[0][-1])
    t[last:] = np.uint64(1) << np.uint64(32)
    return np.maximum.accumulate(t)


def _rounding_intervals():
    """Per non-negative finite E4M3 code 0x00..0x7E, the [lo, hi) interval of
    magnitudes that round to it (midpoints; the top code takes everything
    above, as a saturating conversion does)."""
    v = _fp8_values()[:0x7F]
    lo = np.concatenate([[0.0], (v[:-1] + v[1:]) / 2])
    hi = np.concatenate([(v[:-1] + v[1:]) / 2, [np.inf]])
    return lo, hi


def e4m3_normal_table() -> np.ndarray:
    """Thresholds for E4M3 bytes distributed as N(0,1) rounded to E4M3 and
    clamped to +-448 (the FP8 weight distribution of the workloads)."""
    lo, hi = _rounding_intervals()
    phi = lambda z: 0.5 * (1.0 + math.erf(z / math.sqrt(2.0))) if np.isfinite(z) else 1.0
    pos = np.array([phi(h) - phi(l) for l, h in zip(lo, hi)])
    p = np.zeros(256)
    p[:0x7F] = pos
    p[0x80:0xFF] = pos
    return _cumulative(p)


def e4m3_loguniform_table(lo_exp: float, hi_exp: float) -> np.ndarray:
    """Thresholds for E4M3 bytes of 2^U(lo_exp, hi_exp) rounded to E4M3 (the
    UE4M3 group-16 scale distribution of the NVFP4 workload)."""
    lo, hi = _rounding_intervals()
    with np.errstate(divide="ignore"):
        a = np.clip(np.log2(np.maximum(lo, 1e-300)), lo_exp, hi_exp)
        b = np.clip(np.log2(np.minimum(hi, 1e300)), lo_exp, hi_exp)
    p = np.zeros(256)
    p[:0x7F] = np.maximum(b - a, 0.0)
    return _cumulative(p)


def uniform_byte_table() -> np.ndarray:
    """Thresholds for uniformly distributed bytes (packed E2M1 pairs: every
    nibble uniform over the 16 codes)."""
    return _cumulative(np.ones(256))


# --------------------------------------------------------------------------- host draws
def expert_bytes(seed, tensor, expert, rows, cols, table, row_idx=None) -> np.ndarray:
    """[len(row_idx) or rows, cols] uint8 codes of one expert's tensor."""
    r = np.arange(rows) if row_idx is None else np.asarray(row_idx)
    index = r[:, None].astype(np.uint64) * np.uint64(cols) + np.arange(cols, dtype=np.uint64)[None, :]
    return codes_from_words(words(seed, tensor, expert, index), table)


def loguniform_f32(seed, tensor, shape, lo_exp, hi_exp) -> np.ndarray:
    """float32 2^U(lo_exp, hi_exp) array (FP32 block scales), counter-based."""
    n = int(np.prod(shape))
    w = words(seed, tensor, 0xFFFFFF, np.arange(n)).astype(np.float64)
    u = (w + 0.5) / 2.0**32
    return np.exp2(lo_exp + (hi_exp - lo_exp) * u).astype(np.float32).reshape(shape)


def pow2_ceil_f32(values) -> np.ndarray:
    """Round positive float32 scales up to powers of two (UE8M0 weight scales
    of the ue8m0 workload); an input transform, done with frexp."""
    m, e = np.frexp(np.asarray(values, dtype=np.float64))
    e = np.where(m == 0.5, e - 1, e)
    return np.ldexp(1.0, e).astype(np.float32)


def normal_f32(seed, stream, shape, std=1.0) -> np.ndarray:
    rng = np.random.default_rng([int(seed), int(stream)])
    return (rng.standard_normal(size=shape) * std).astype(np.float32)


def to_bf16_values(v) -> np.ndarray:
    """float32 values rounded to BF16 by torch (library cast), as float32."""
    import torch

    return torch.from_numpy(np.ascontiguousarray(v, dtype=np.float32)).to(torch.bfloat16) \
        .to(torch.float32).numpy()


# --------------------------------------------------------------------------- device fill
_HERE = __import__("os").path.dirname(__import__("os").path.abspath(__file__))
SYNTH_LIB = __import__("os").path.join(_HERE, "libfme_synth.so")
_synth = None


def build_device_lib(force=False):
    """Compile synth/csrc/synth.cu -> synth/libfme_synth.so (sm_103a)."""
    import os
    import subprocess

    src = os.path.join(_HERE, "csrc", "synth.cu")
    if not force and os.path.exists(SYNTH_LIB) and os.path.getmtime(SYNTH_LIB) >= os.path.getmtime(src):
        return SYNTH_LIB
    cmd = [os.environ.get("NVCC", "nvcc"), "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-shared",
           "-Xcompiler", "-fPIC", "-o", SYNTH_LIB + ".tmp", src]
    subprocess.run(cmd, check=True, capture_output=True)
    os.replace(SYNTH_LIB + ".tmp", SYNTH_LIB)
    return SYNTH_LIB


def _lib():
    global _synth
    if _synth is None:
        import ctypes

        build_device_lib()
        _synth = ctypes.CDLL(SYNTH_LIB)
        _synth.fme_synth_fill_codes.restype = ctypes.c_int
        _synth.fme_synth_fill_codes.argtypes = [ctypes.c_void_p, ctypes.c_longlong, ctypes.c_longlong,
                                                ctypes.c_uint, ctypes.c_int, ctypes.c_void_p, ctypes.c_int,
                                                ctypes.c_void_p]
    return _synth


def fill_codes_device(out, seed, tensor, table, expert0=0):
    """Fill a CUDA uint8 tensor [E, ...] in place: expert e (the first dim,
    offset by expert0) gets exactly ``expert_bytes(seed, tensor, e + expert0, ...)``."""
    import ctypes

    import torch

    assert out.dtype == torch.uint8 and out.is_cuda and out.is_contiguous()
    t = torch.as_tensor(np.asarray(table, dtype=np.uint64).view(np.int64), device=out.device)
    n_experts = out.shape[0]
    per = out.numel() // n_experts
    rc = _lib().fme_synth_fill_codes(ctypes.c_void_p(out.data_ptr()), n_experts, per, int(seed) & 0xFFFFFFFF,
                                     int(tensor), ctypes.c_void_p(t.data_ptr()), int(expert0),
                                     ctypes.c_void_p(torch.cuda.current_stream(out.device).cuda_stream))
    if rc != 0:
        raise RuntimeError(f"synth fill failed: cuda error {rc}")
    return out
