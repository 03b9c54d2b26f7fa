"""The workloads the layer is measured and checked on, and their seeded inputs.

Shapes and distributions follow the stated workload list (tiny routed FP8;
DeepSeek-V3-shaped routed FP8, plain and UE8M0 with the shared expert;
latent-MoE-shaped routed FP8 with a skewed bias; NVFP4 slot MoE over 48 local
experts of a 384-expert router). Nothing here computes any part of the layer.
"""

import dataclasses
from functools import lru_cache

import numpy as np

from . import (T_S13, T_S2, T_SW13, T_SW2, T_W13, T_W2, e4m3_loguniform_table, e4m3_normal_table,
               expert_bytes, fill_codes_device, loguniform_f32, normal_f32, pow2_ceil_f32, to_bf16_values,
               uniform_byte_table)

# Streams of the small host-drawn tensors.
S_X, S_LOGITS, S_BIAS = 11, 12, 13


@dataclasses.dataclass(frozen=True)
class Fp8Config:
    name: str
    H: int
    I: int
    E: int
    top_k: int
    limit: float
    scale: float
    ue8m0: bool
    logits_bf16: bool
    bias_std: float
    scale_lo: float  # log2 bounds of the FP32 block scales
    scale_hi: float
    Ms: tuple


TINY = Fp8Config("tiny_fp8", 512, 256, 8, 2, 7.0, 2.5, False, False, 0.1, -10, -6, (1,))
DSV3 = Fp8Config("dsv3_fp8", 7168, 2048, 256, 8, 7.0, 2.5, False, True, 0.05, -12, -6, (1, 2, 4, 8))
DSV3_UE8M0 = dataclasses.replace(DSV3, name="dsv3_fp8_ue8m0", ue8m0=True)
LATENT = Fp8Config("latent_fp8", 3584, 2048, 896, 16, 7.0, 2.5, False, False, 0.5, -12, -6, (1, 5, 16, 32))
# Extra parity shapes: several tiles, ragged expert count (E % 32 != 0), odd I/128.
RAGGED = Fp8Config("ragged_fp8", 1024, 384, 40, 3, 7.0, 1.5, False, False, 0.1, -10, -6, (5,))
FP8_CONFIGS = {c.name: c for c in (TINY, DSV3, DSV3_UE8M0, LATENT, RAGGED)}


@dataclasses.dataclass(frozen=True)
class SharedConfig:
    name: str
    H: int
    I: int
    limit: float
    ue8m0: bool


SHARED = SharedConfig("dsv3_shared_ue8m0", 7168, 2048, 7.0, True)


@dataclasses.dataclass(frozen=True)
class Nvfp4Config:
    name: str
    H: int
    N: int
    L: int
    E: int  # experts of the router
    e0: int
    top_k: int
    limit: float
    Ms: tuple


NVFP4 = Nvfp4Config("nvfp4_local48", 7168, 3072, 48, 384, 0, 6, float("inf"), (1, 8, 32, 64))


# --------------------------------------------------------------------------- FP8 routed
class HostExperts:
    """Lazy host view of a generated [E, rows, cols] byte tensor: expert e is
    regenerated on demand (and cached) from the counter-based stream."""

    def __init__(self, seed, tensor, rows, cols, table, n=None):
        self.seed, self.tensor, self.rows, self.cols, self.table = seed, tensor, rows, cols, table
        self.n = n
        self._get = lru_cache(maxsize=4)(self._make)

    def _make(self, e):
        return expert_bytes(self.seed, self.tensor, e, self.rows, self.cols, self.table)

    def __getitem__(self, e):
        return self._get(int(e))

    def rows_of(self, e, row_idx):
        return expert_bytes(self.seed, self.tensor, int(e), self.rows, self.cols, self.table, row_idx=row_idx)

    def full(self):
        return np.stack([self[e] for e in range(self.n)])


def fp8_weight_scales(cfg: Fp8Config, seed: int):
    s13 = loguniform_f32(seed, T_S13, (cfg.E, 2 * cfg.I // 128, cfg.H // 128), cfg.scale_lo, cfg.scale_hi)
    s2 = loguniform_f32(seed, T_S2, (cfg.E, cfg.H // 128, cfg.I // 128), cfg.scale_lo, cfg.scale_hi)
    if cfg.ue8m0:
        s13, s2 = pow2_ceil_f32(s13), pow2_ceil_f32(s2)
    return s13, s2


def fp8_weights_host(cfg: Fp8Config, seed: int):
    t = e4m3_normal_table()
    w13 = HostExperts(seed, T_W13, 2 * cfg.I, cfg.H, t, cfg.E)
    w2 = HostExperts(seed, T_W2, cfg.H, cfg.I, t, cfg.E)
    return w13, w2


def fp8_activations(cfg: Fp8Config, M: int, seed: int, step: int = 0):
    """x [M, H] (BF16 values as float32), logits [M, E] (BF16 values when the
    workload's logits are BF16) and bias [E]; `step` varies x and logits."""
    x = to_bf16_values(normal_f32(seed, S_X * 1000003 + step, (M, cfg.H)))
    logits = normal_f32(seed, S_LOGITS * 1000003 + step, (M, cfg.E))
    if cfg.logits_bf16:
        logits = to_bf16_values(logits)
    bias = normal_f32(seed, S_BIAS, (cfg.E,), cfg.bias_std)
    return x, logits, bias


def fp8_weights_device(cfg: Fp8Config, seed: int, device):
    """W13, S13, W2, S2 as CUDA tensors (weights filled on the device)."""
    import torch

    t = e4m3_normal_table()
    w13 = torch.empty(cfg.E, 2 * cfg.I, cfg.H, dtype=torch.uint8, device=device)
    w2 = torch.empty(cfg.E, cfg.H, cfg.I, dtype=torch.uint8, device=device)
    fill_codes_device(w13, seed, T_W13, t)
    fill_codes_device(w2, seed, T_W2, t)
    s13, s2 = fp8_weight_scales(cfg, seed)
    return w13, torch.from_numpy(s13).to(device), w2, torch.from_numpy(s2).to(device)


def shared_weights_host(cfg: SharedConfig, seed: int):
    """Shared-expert gate_up [2I, H] / down [H, I] E4M3 bytes and FP32 block
    scales (UE8M0 powers of two when the workload says so)."""
    t = e4m3_normal_table()
    w13 = expert_bytes(seed, T_W13, 0x7FFF, 2 * cfg.I, cfg.H, t)
    w2 = expert_bytes(seed, T_W2, 0x7FFF, cfg.H, cfg.I, t)
    s13 = loguniform_f32(seed + 77, T_S13, (2 * cfg.I // 128, cfg.H // 128), -12, -6)
    s2 = loguniform_f32(seed + 77, T_S2, (cfg.H // 128, cfg.I // 128), -12, -6)
    if cfg.ue8m0:
        s13, s2 = pow2_ceil_f32(s13), pow2_ceil_f32(s2)
    return w13, s13, w2, s2


# --------------------------------------------------------------------------- NVFP4
def nvfp4_weights_host(cfg: Nvfp4Config, seed: int):
    ub = uniform_byte_table()
    st = e4m3_loguniform_table(-8, 0)
    w13 = HostExperts(seed, T_W13, 2 * cfg.N, cfg.H // 2, ub, cfg.L)
    s13 = HostExperts(seed, T_SW13, 2 * cfg.N, cfg.H // 16, st, cfg.L)
    w2 = HostExperts(seed, T_W2, cfg.H, cfg.N // 2, ub, cfg.L)
    s2 = HostExperts(seed, T_SW2, cfg.H, cfg.N // 16, st, cfg.L)
    return w13, s13, w2, s2


def nvfp4_weights_device(cfg: Nvfp4Config, seed: int, device):
    import torch

    ub = uniform_byte_table()
    st = e4m3_loguniform_table(-8, 0)
    out = []
    for tensor, rows, cols, table in ((T_W13, 2 * cfg.N, cfg.H // 2, ub), (T_SW13, 2 * cfg.N, cfg.H // 16, st),
                                      (T_W2, cfg.H, cfg.N // 2, ub), (T_SW2, cfg.H, cfg.N // 16, st)):
        buf = torch.empty(cfg.L, rows, cols, dtype=torch.uint8, device=device)
        fill_codes_device(buf, seed, tensor, table)
        out.append(buf)
    return tuple(out)


def nvfp4_activations(cfg: Nvfp4Config, M: int, seed: int, step: int = 0):
    """x [M, H] BF16 values and router logits [M, E] / bias [E] (the tests derive
    topk ids and weights from these with the oracle's routing; the bench lets
    the fused-routing entry pick them)."""
    x = to_bf16_values(normal_f32(seed, S_X * 1000003 + step, (M, cfg.H)))
    logits = normal_f32(seed, S_LOGITS * 1000003 + step, (M, cfg.E))
    bias = normal_f32(seed, S_BIAS, (cfg.E,), 0.05)
    return x, logits, bias
