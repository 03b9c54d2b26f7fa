"""Python binding of libfme.so (include/fme.h): the routed-expert MoE decode
layer (FP8 and NVFP4) and the FP8 shared expert on sm_103a.

Argument marshalling only: torch supplies device memory and the current
stream; every step of the computation runs in the library's CUDA kernels.
Importing this package loads libfme.so and raises if it is missing (build it
with ``python -m fp4_moe_expert_gb300.build`` or ``__graft_entry__.build()``).
"""

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libfme.so")

FME_OK = 0
FME_F32 = 0
FME_BF16 = 1

# Every symbol include/fme.h declares, with its ctypes signature.
_c_int, _c_size, _vp, _c_float = ctypes.c_int, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_float
SIGNATURES = {
    "fme_last_error": (ctypes.c_char_p, []),
    "fme_version": (_c_int, []),
    "fme_moe_routed_fp8": (_c_int, [_vp, _vp, _c_int, _vp, _vp, _vp, _vp, _vp, _c_int, _c_int, _c_int, _c_int,
                                    _c_int, _c_float, _c_float, _c_int, _vp, _vp, _vp, _vp, _c_size, _vp]),
    "fme_moe_routed_fp8_workspace": (_c_size, [_c_int] * 5),
    "fme_moe_routed_fp8_mx": (_c_int, [_vp, _vp, _vp, _c_int, _vp, _vp, _vp, _vp, _vp, _c_int, _c_int, _c_int, _c_int,
                                       _c_int, _c_float, _c_float, _c_int, _vp, _vp, _vp, _vp, _c_size, _vp]),
    "fme_moe_routed_fp8_noalloc": (_c_int, [_vp, _vp, _c_int, _vp, _vp, _vp, _vp, _vp, _c_int, _c_int, _c_int,
                                            _c_int, _c_int, _c_float, _c_float, _c_int, _vp, _vp, _vp, _vp]),
    "fme_moe_routed_fp8_noalloc_error": (_c_int, [_vp, _vp]),
    "fme_shared_expert_fp8": (_c_int, [_vp, _vp, _vp, _vp, _vp, _c_int, _c_int, _c_int, _c_float, _c_int, _vp,
                                       _vp, _vp, _c_size, _vp]),
    "fme_shared_expert_fp8_workspace": (_c_size, [_c_int] * 3),
    "fme_moe_layer_fp8": (_c_int, [_vp, _vp, _c_int, _vp, _vp, _vp, _vp, _vp, _c_int, _c_int, _c_int, _c_int,
                                   _c_int, _c_float, _c_float, _c_int, _vp, _vp, _vp, _vp, _c_float, _c_int,
                                   _vp, _vp, _vp, _vp, _vp, _c_size, _vp]),
    "fme_moe_layer_fp8_workspace": (_c_size, [_c_int] * 5),
    "fme_ue8m0_unpack": (_c_int, [_vp, _c_int, _c_int, _vp, _c_int, _vp, _vp]),
    "fme_moe_routed_nvfp4": (_c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _c_int, _c_int, _c_int, _c_int, _c_int,
                                      _c_int, _c_float, _vp, _vp, _c_size, _vp]),
    "fme_moe_routed_nvfp4_workspace": (_c_size, [_c_int] * 5),
    "fme_moe_finalize": (_c_int, [_vp, _vp, _vp, _c_int, _c_int, _c_int, _vp, _vp]),
    "fme_mxfp8_quantize": (_c_int, [_vp, _c_int, _c_int, _vp, _vp, _vp]),
    "fme_combine_rmsnorm": (_c_int, [_vp, _c_int, _c_int, _c_int, _vp, _c_float, _vp, _vp, _vp]),
    "fme_moe_layer_nvfp4": (_c_int, [_vp, _vp, _c_int, _vp, _vp, _vp, _vp, _vp, _c_int, _c_int, _c_int, _c_int,
                                     _c_int, _c_int, _c_int, _c_float, _c_float, _vp, _vp, _vp, _vp, _c_size, _vp]),
    "fme_workspace_clear": (_c_int, [_vp, _c_size, _vp]),
    "fme_selftest_wait_timeout": (_c_int, [_vp, _c_size, _c_int, _vp]),
    "fme_workspace_error": (_c_int, [_vp, ctypes.POINTER(_c_int), _vp]),
    "fme_sm_count": (_c_int, []),
}


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libfme.so not built at {LIB_PATH}; run fp4_moe_expert_gb300/build.py")
    lib = ctypes.CDLL(LIB_PATH)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


lib = _load()


class FmeError(RuntimeError):
    def __init__(self, status, message):
        super().__init__(f"fme status {status}: {message}")
        self.status = status


def _check(status):
    if status != FME_OK:
        raise FmeError(status, lib.fme_last_error().decode())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device):
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _need(t, dtype, shape, name):
    if t.dtype != dtype or tuple(t.shape) != tuple(shape) or not t.is_contiguous() or not t.is_cuda:
        raise ValueError(f"{name}: expected contiguous CUDA {dtype} {tuple(shape)}, got {t.dtype} "
                         f"{tuple(t.shape)} contiguous={t.is_contiguous()} cuda={t.is_cuda}")


class Workspace:
    """Caller-owned device scratch for one stream: zero-filled once at creation;
    every successful call leaves it zeroed again."""

    def __init__(self, nbytes, device):
        self.nbytes = int(nbytes)
        self.buf = torch.zeros(max(self.nbytes, 256), dtype=torch.uint8, device=device)

    def ptr(self):
        return ctypes.c_void_p(self.buf.data_ptr())

    def clear(self):
        _check(lib.fme_workspace_clear(self.ptr(), self.nbytes, _stream(self.buf.device)))

    def error(self):
        """Device error word (0 = none); reading it synchronises the stream and clears it."""
        code = ctypes.c_int(0)
        lib.fme_workspace_error(self.ptr(), ctypes.byref(code), _stream(self.buf.device))
        return code.value


_ws_cache = {}


def _workspace(nbytes, device, workspace):
    if workspace is not None:
        if workspace.nbytes < nbytes:
            raise ValueError(f"workspace of {workspace.nbytes} bytes, {nbytes} needed")
        return workspace
    key = (device.index if device.index is not None else torch.cuda.current_device(), nbytes)
    ws = _ws_cache.get(key)
    if ws is None:
        ws = Workspace(nbytes, device)
        _ws_cache[key] = ws
    return ws


def moe_routed_fp8_workspace(M, H, I, E, top_k):
    return lib.fme_moe_routed_fp8_workspace(M, H, I, E, top_k)


def moe_routed_fp8(x, logits, bias, w13, s13, w2, s2, top_k, limit, scale, ue8m0,
                   out=None, ids=None, weights=None, workspace=None):
    """Routed FP8 experts of M tokens (fme_moe_routed_fp8).

    x [M, H] bf16; logits [M, E] bf16 or float32; bias [E] float32;
    w13 [E, 2I, H] uint8 (E4M3, up rows then gate rows); s13 [E, 2I/128, H/128] f32;
    w2 [E, H, I] uint8; s2 [E, H/128, I/128] f32.
    Returns out [M*top_k, H] bf16 (unweighted route rows), ids [M, top_k] int32,
    weights [M, top_k] float32.
    """
    M, H = x.shape
    E, n2, _ = w13.shape
    I = n2 // 2
    dev = x.device
    _need(x, torch.bfloat16, (M, H), "x")
    if logits.dtype not in (torch.float32, torch.bfloat16):
        raise ValueError("logits must be float32 or bfloat16")
    _need(logits, logits.dtype, (M, E), "logits")
    _need(bias, torch.float32, (E,), "bias")
    _need(w13, torch.uint8, (E, 2 * I, H), "w13")
    _need(s13, torch.float32, (E, 2 * I // 128, H // 128), "s13")
    _need(w2, torch.uint8, (E, H, I), "w2")
    _need(s2, torch.float32, (E, H // 128, I // 128), "s2")
    if out is None:
        out = torch.empty(M * top_k, H, dtype=torch.bfloat16, device=dev)
    if ids is None:
        ids = torch.empty(M, top_k, dtype=torch.int32, device=dev)
    if weights is None:
        weights = torch.empty(M, top_k, dtype=torch.float32, device=dev)
    need = moe_routed_fp8_workspace(M, H, I, E, top_k)
    ws = _workspace(need, dev, workspace)
    ldt = FME_F32 if logits.dtype == torch.float32 else FME_BF16
    _check(lib.fme_moe_routed_fp8(_ptr(x), _ptr(logits), ldt, _ptr(bias), _ptr(w13), _ptr(s13), _ptr(w2),
                                  _ptr(s2), M, H, I, E, top_k, float(limit), float(scale), int(bool(ue8m0)),
                                  _ptr(out), _ptr(ids), _ptr(weights), ws.ptr(), ws.nbytes, _stream(dev)))
    return out, ids, weights


def moe_routed_fp8_mx(xq, xscales, logits, bias, w13, s13, w2, s2, top_k, limit, scale, ue8m0,
                      out=None, ids=None, weights=None, workspace=None):
    """moe_routed_fp8 with MXFP8 activations (fme_moe_routed_fp8_mx): xq [M, H] uint8
    E4M3 and xscales [M, H/32] uint8 E8M0 (as mxfp8_quantize returns). Returns
    (out [M*top_k, H] bf16, ids [M, top_k] int32, weights [M, top_k] float32)."""
    M, H = xq.shape
    E = logits.shape[1]
    I = w2.shape[2]
    dev = xq.device
    _need(xq, torch.uint8, (M, H), "xq")
    _need(xscales, torch.uint8, (M, H // 32), "xscales")
    if logits.dtype == torch.float32:
        dt = FME_F32
    elif logits.dtype == torch.bfloat16:
        dt = FME_BF16
    else:
        raise ValueError("logits must be float32 or bfloat16")
    _need(logits, logits.dtype, (M, E), "logits")
    _need(bias, torch.float32, (E,), "bias")
    _need(w13, torch.uint8, (E, 2 * I, H), "w13")
    _need(s13, torch.float32, (E, 2 * I // 128, H // 128), "s13")
    _need(w2, torch.uint8, (E, H, I), "w2")
    _need(s2, torch.float32, (E, H // 128, I // 128), "s2")
    if out is None:
        out = torch.empty(M * top_k, H, dtype=torch.bfloat16, device=dev)
    if ids is None:
        ids = torch.empty(M, top_k, dtype=torch.int32, device=dev)
    if weights is None:
        weights = torch.empty(M, top_k, dtype=torch.float32, device=dev)
    need = moe_routed_fp8_workspace(M, H, I, E, top_k)
    ws = _workspace(need, dev, workspace)
    _check(lib.fme_moe_routed_fp8_mx(_ptr(xq), _ptr(xscales), _ptr(logits), dt, _ptr(bias), _ptr(w13), _ptr(s13),
                                     _ptr(w2), _ptr(s2), M, H, I, E, top_k, float(limit), float(scale), int(ue8m0),
                                     _ptr(out), _ptr(ids), _ptr(weights), ws.ptr(), ws.nbytes, _stream(dev)))
    return out, ids, weights


def shared_expert_fp8_workspace(M, H, I):
    return lib.fme_shared_expert_fp8_workspace(M, H, I)


def shared_expert_fp8(x, w13, s13, w2, s2, limit, ue8m0, out=None, gate_up=None, want_gate_up=False,
                      workspace=None):
    """FP8 shared expert (fme_shared_expert_fp8). w13 [2I, H] (gate rows first),
    s13 [2I/128, H/128] f32, w2 [H, I], s2 [H/128, I/128] f32. Returns out [M, H]
    bf16 (and gate_up [M, 2I] bf16 when want_gate_up)."""
    M, H = x.shape
    n2 = w13.shape[0]
    I = n2 // 2
    dev = x.device
    _need(x, torch.bfloat16, (M, H), "x")
    _need(w13, torch.uint8, (2 * I, H), "w13")
    _need(s13, torch.float32, (2 * I // 128, H // 128), "s13")
    _need(w2, torch.uint8, (H, I), "w2")
    _need(s2, torch.float32, (H // 128, I // 128), "s2")
    if out is None:
        out = torch.empty(M, H, dtype=torch.bfloat16, device=dev)
    if want_gate_up and gate_up is None:
        gate_up = torch.empty(M, 2 * I, dtype=torch.bfloat16, device=dev)
    need = shared_expert_fp8_workspace(M, H, I)
    ws = _workspace(need, dev, workspace)
    _check(lib.fme_shared_expert_fp8(_ptr(x), _ptr(w13), _ptr(s13), _ptr(w2), _ptr(s2), M, H, I, float(limit),
                                     int(bool(ue8m0)), _ptr(gate_up), _ptr(out), ws.ptr(), ws.nbytes,
                                     _stream(dev)))
    return (out, gate_up) if want_gate_up else out


def moe_layer_fp8_workspace(M, H, I, E, top_k):
    return lib.fme_moe_layer_fp8_workspace(M, H, I, E, top_k)


def moe_layer_fp8(x, logits, bias, w13, s13, w2, s2, top_k, limit, scale, ue8m0,
                  shared_w13, shared_s13, shared_w2, shared_s2, shared_limit, shared_ue8m0,
                  out=None, ids=None, weights=None, shared_out=None, workspace=None):
    """Routed experts and shared expert in one launch (fme_moe_layer_fp8).

    Routed arguments as moe_routed_fp8; shared_* as shared_expert_fp8 (same H, I).
    Returns (out [M*top_k, H], ids, weights, shared_out [M, H]).
    """
    M, H = x.shape
    E, n2, _ = w13.shape
    I = n2 // 2
    dev = x.device
    _need(x, torch.bfloat16, (M, H), "x")
    if logits.dtype not in (torch.float32, torch.bfloat16):
        raise ValueError("logits must be float32 or bfloat16")
    _need(logits, logits.dtype, (M, E), "logits")
    _need(bias, torch.float32, (E,), "bias")
    _need(w13, torch.uint8, (E, 2 * I, H), "w13")
    _need(s13, torch.float32, (E, 2 * I // 128, H // 128), "s13")
    _need(w2, torch.uint8, (E, H, I), "w2")
    _need(s2, torch.float32, (E, H // 128, I // 128), "s2")
    _need(shared_w13, torch.uint8, (2 * I, H), "shared_w13")
    _need(shared_s13, torch.float32, (2 * I // 128, H // 128), "shared_s13")
    _need(shared_w2, torch.uint8, (H, I), "shared_w2")
    _need(shared_s2, torch.float32, (H // 128, I // 128), "shared_s2")
    if out is None:
        out = torch.empty(M * top_k, H, dtype=torch.bfloat16, device=dev)
    if ids is None:
        ids = torch.empty(M, top_k, dtype=torch.int32, device=dev)
    if weights is None:
        weights = torch.empty(M, top_k, dtype=torch.float32, device=dev)
    if shared_out is None:
        shared_out = torch.empty(M, H, dtype=torch.bfloat16, device=dev)
    need = moe_layer_fp8_workspace(M, H, I, E, top_k)
    ws = _workspace(need, dev, workspace)
    ldt = FME_F32 if logits.dtype == torch.float32 else FME_BF16
    _check(lib.fme_moe_layer_fp8(_ptr(x), _ptr(logits), ldt, _ptr(bias), _ptr(w13), _ptr(s13), _ptr(w2),
                                 _ptr(s2), M, H, I, E, top_k, float(limit), float(scale), int(bool(ue8m0)),
                                 _ptr(shared_w13), _ptr(shared_s13), _ptr(shared_w2), _ptr(shared_s2),
                                 float(shared_limit), int(bool(shared_ue8m0)), _ptr(out), _ptr(ids),
                                 _ptr(weights), _ptr(shared_out), ws.ptr(), ws.nbytes, _stream(dev)))
    return out, ids, weights, shared_out


def moe_finalize(out, weights, shared_out=None, y=None):
    """y [M, H] BF16 = bf16(sum over r of weights[t, r] * out[t * top_k + r] (+ shared_out[t]))
    (fme_moe_finalize): out [M * top_k, H] BF16 unweighted expert rows as the routed
    call returns them, weights [M, top_k] FP32, shared_out [M, H] BF16 or None."""
    dev = out.device
    M, top_k = weights.shape
    H = out.shape[1]
    _need(out, torch.bfloat16, (M * top_k, H), "out")
    _need(weights, torch.float32, (M, top_k), "weights")
    if shared_out is not None:
        _need(shared_out, torch.bfloat16, (M, H), "shared_out")
    if y is None:
        y = torch.empty(M, H, dtype=torch.bfloat16, device=dev)
    _need(y, torch.bfloat16, (M, H), "y")
    _check(lib.fme_moe_finalize(_ptr(out), _ptr(weights), _ptr(shared_out), M, H, top_k, _ptr(y), _stream(dev)))
    return y


def mxfp8_quantize(x):
    """(q [T, H] uint8 E4M3, scales [T, H/32] uint8 E8M0) of x [T, H] BF16 (fme_mxfp8_quantize)."""
    T, H = x.shape
    dev = x.device
    _need(x, torch.bfloat16, (T, H), "x")
    q = torch.empty(T, H, dtype=torch.uint8, device=dev)
    sc = torch.empty(T, H // 32, dtype=torch.uint8, device=dev)
    _check(lib.fme_mxfp8_quantize(_ptr(x), T, H, _ptr(q), _ptr(sc), _stream(dev)))
    return q, sc


def combine_rmsnorm(partials, gamma, eps=1e-5):
    """(latent [T, H], normed [T, H]) BF16 of partials [T, N, H] BF16 and gamma [H] BF16
    (fme_combine_rmsnorm)."""
    T, N, H = partials.shape
    dev = partials.device
    _need(partials, torch.bfloat16, (T, N, H), "partials")
    _need(gamma, torch.bfloat16, (H,), "gamma")
    latent = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
    normed = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
    _check(lib.fme_combine_rmsnorm(_ptr(partials), T, N, H, _ptr(gamma), float(eps), _ptr(latent), _ptr(normed),
                                   _stream(dev)))
    return latent, normed


def ue8m0_unpack(packed, n, k, check=True):
    """FP32 [n/128, k/128] block scales from packed UE8M0 int32 [n, k/512]
    (fme_ue8m0_unpack). With check, raises ValueError when a 128-row block is
    not uniform (this reads a device flag, so it synchronises)."""
    dev = packed.device
    _need(packed, torch.int32, (n, k // 512), "packed")
    dst = torch.empty(n // 128, k // 128, dtype=torch.float32, device=dev)
    flag = torch.zeros(4, dtype=torch.int32, device=dev) if check else None
    _check(lib.fme_ue8m0_unpack(_ptr(packed), n, k, _ptr(dst), int(check), _ptr(flag), _stream(dev)))
    if check and int(flag[0].item()) != 0:
        raise ValueError("scales vary inside a 128-row block")
    return dst


def moe_routed_nvfp4_workspace(M, H, N, L, top_k):
    return lib.fme_moe_routed_nvfp4_workspace(M, H, N, L, top_k)


def moe_routed_nvfp4(x, topk_ids, topk_weights, w13, s13, w2, s2, e0, limit=float("inf"), y=None,
                     workspace=None):
    """NVFP4 slot MoE over local experts [e0, e0 + L) (fme_moe_routed_nvfp4).
    w13 [L, 2N, H/2] uint8 packed E2M1 (gate rows then up rows), s13 [L, 2N, H/16]
    uint8 UE4M3, w2 [L, H, N/2], s2 [L, H, N/16]. Returns y [M, H] bf16."""
    M, H = x.shape
    L, n2, _ = w13.shape
    N = n2 // 2
    top_k = topk_ids.shape[1]
    dev = x.device
    _need(x, torch.bfloat16, (M, H), "x")
    _need(topk_ids, torch.int32, (M, top_k), "topk_ids")
    _need(topk_weights, torch.float32, (M, top_k), "topk_weights")
    _need(w13, torch.uint8, (L, 2 * N, H // 2), "w13")
    _need(s13, torch.uint8, (L, 2 * N, H // 16), "s13")
    _need(w2, torch.uint8, (L, H, N // 2), "w2")
    _need(s2, torch.uint8, (L, H, N // 16), "s2")
    if y is None:
        y = torch.empty(M, H, dtype=torch.bfloat16, device=dev)
    need = moe_routed_nvfp4_workspace(M, H, N, L, top_k)
    ws = _workspace(need, dev, workspace)
    _check(lib.fme_moe_routed_nvfp4(_ptr(x), _ptr(topk_ids), _ptr(topk_weights), _ptr(w13), _ptr(s13), _ptr(w2),
                                    _ptr(s2), M, H, N, L, int(e0), top_k, float(limit), _ptr(y), ws.ptr(),
                                    ws.nbytes, _stream(dev)))
    return y


def moe_layer_nvfp4(x, logits, bias, w13, s13, w2, s2, e0, top_k, scale=1.0, limit=float("inf"), y=None,
                    workspace=None):
    """NVFP4 slot MoE with the routing fused in (fme_moe_layer_nvfp4): logits [M, E]
    FP32 or BF16 and bias [E] FP32 pick top_k of E experts per token; the slots of the
    local experts [e0, e0 + L) run as in moe_routed_nvfp4. Returns (y, ids, weights)."""
    M, H = x.shape
    E = logits.shape[1]
    L, n2, _ = w13.shape
    N = n2 // 2
    dev = x.device
    _need(x, torch.bfloat16, (M, H), "x")
    if logits.dtype == torch.float32:
        dt = FME_F32
    elif logits.dtype == torch.bfloat16:
        dt = FME_BF16
    else:
        raise ValueError("logits must be float32 or bfloat16")
    _need(logits, logits.dtype, (M, E), "logits")
    _need(bias, torch.float32, (E,), "bias")
    _need(w13, torch.uint8, (L, 2 * N, H // 2), "w13")
    _need(s13, torch.uint8, (L, 2 * N, H // 16), "s13")
    _need(w2, torch.uint8, (L, H, N // 2), "w2")
    _need(s2, torch.uint8, (L, H, N // 16), "s2")
    if y is None:
        y = torch.empty(M, H, dtype=torch.bfloat16, device=dev)
    ids = torch.empty(M, top_k, dtype=torch.int32, device=dev)
    weights = torch.empty(M, top_k, dtype=torch.float32, device=dev)
    need = moe_routed_nvfp4_workspace(M, H, N, L, top_k)
    ws = _workspace(need, dev, workspace)
    _check(lib.fme_moe_layer_nvfp4(_ptr(x), _ptr(logits), dt, _ptr(bias), _ptr(w13), _ptr(s13), _ptr(w2), _ptr(s2),
                                   M, H, N, L, E, int(e0), int(top_k), float(scale), float(limit), _ptr(y),
                                   _ptr(ids), _ptr(weights), ws.ptr(), ws.nbytes, _stream(dev)))
    return y, ids, weights


def sm_count():
    return lib.fme_sm_count()
