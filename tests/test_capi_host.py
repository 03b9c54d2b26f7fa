"""CPU-only checks of the C ABI: libfme.so loads, exports every entry point
include/fme.h declares, and its host-side argument checks reject bad calls
before touching the GPU."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fme.h")


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(fme_[a-z0-9_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def fme():
    import __graft_entry__
    __graft_entry__.build()
    import fp4_moe_expert_gb300 as m
    return m


def test_every_declared_symbol_is_exported(fme):
    names = _declared()
    assert "fme_moe_routed_fp8" in names and "fme_moe_routed_nvfp4" in names
    for n in names:
        assert hasattr(fme.lib, n), n
        assert n in fme.SIGNATURES, f"binding lacks {n}"
    # and the binding exposes nothing the header does not declare
    assert set(fme.SIGNATURES) == set(names)


def test_version_and_workspace_sizes(fme):
    assert fme.lib.fme_version() >= 100
    assert fme.moe_routed_fp8_workspace(8, 7168, 2048, 256, 8) > 64 * 2048 * 4
    assert fme.moe_routed_fp8_workspace(0, 7168, 2048, 256, 8) == 0
    assert fme.moe_routed_fp8_workspace(1, 7168, 2000, 256, 8) == 0
    assert fme.moe_routed_fp8_workspace(1, 7168, 2048, 256, 300) == 0
    assert fme.moe_routed_nvfp4_workspace(64, 7168, 3072, 48, 6) > 0


def _routed(fme, **kw):
    vp = ctypes.c_void_p
    args = dict(x=vp(16), logits=vp(16), dt=0, bias=vp(16), w13=vp(16), s13=vp(16), w2=vp(16), s2=vp(16),
                M=1, H=512, I=256, E=8, k=2, limit=7.0, scale=1.0, ue=0, out=vp(16), ids=vp(16),
                weights=vp(16), ws=vp(16), wsb=1 << 20, st=None)
    args.update(kw)
    return fme.lib.fme_moe_routed_fp8(*args.values())


def test_host_validation_rejects_bad_calls(fme):
    assert _routed(fme, x=None) == -1                 # null pointer
    assert _routed(fme, M=0) == -2                    # M outside [1, 64]
    assert _routed(fme, M=65) == -2
    assert _routed(fme, H=500) == -1                  # not a multiple of 128
    assert _routed(fme, I=100) == -1
    assert _routed(fme, k=9) == -1                    # top_k > E
    assert _routed(fme, E=2000) == -2
    assert _routed(fme, limit=0.0) == -1
    assert _routed(fme, dt=7) == -1
    assert _routed(fme, scale=float("inf")) == -1
    assert _routed(fme, w13=ctypes.c_void_p(17)) == -3  # misaligned
    msg = fme.lib.fme_last_error().decode()
    assert "aligned" in msg


def _routed_mx(fme, **kw):
    vp = ctypes.c_void_p
    args = dict(xq=vp(16), xs=vp(3), logits=vp(16), dt=0, bias=vp(16), w13=vp(16), s13=vp(16), w2=vp(16),
                s2=vp(16), M=1, H=512, I=256, E=8, k=2, limit=7.0, scale=1.0, ue=0, out=vp(16), ids=vp(16),
                weights=vp(16), ws=vp(16), wsb=1 << 20, st=None)
    args.update(kw)
    return fme.lib.fme_moe_routed_fp8_mx(*args.values())


def test_mx_input_validation(fme):
    assert _routed_mx(fme, xq=None) == -1
    assert _routed_mx(fme, xs=None) == -1
    assert _routed_mx(fme, M=65) == -2
    assert _routed_mx(fme, H=480) == -1
    assert _routed_mx(fme, dt=3) == -1
    assert _routed_mx(fme, xq=ctypes.c_void_p(8)) == -3


def test_nvfp4_and_unpack_validation(fme):
    vp = ctypes.c_void_p
    rc = fme.lib.fme_moe_routed_nvfp4(vp(16), vp(16), vp(16), vp(16), vp(16), vp(16), vp(16), 1, 7168, 3000,
                                      48, 0, 6, float("inf"), vp(16), vp(16), 1 << 20, None)
    assert rc == -1
    assert fme.lib.fme_ue8m0_unpack(vp(16), 100, 512, vp(16), 0, None, None) == -1
    assert fme.lib.fme_ue8m0_unpack(None, 128, 512, vp(16), 0, None, None) == -1


def test_finalize_validation(fme):
    vp = ctypes.c_void_p
    fin = fme.lib.fme_moe_finalize
    assert fin(vp(16), vp(16), None, 1, 7168, 8, None, None) == -1       # y missing
    assert fin(vp(16), vp(16), None, 0, 7168, 8, vp(16), None) == -1     # M
    assert fin(vp(16), vp(16), None, 2, 7164, 8, vp(16), None) == -1     # H not a multiple of 8
    assert fin(vp(16), vp(16), None, 2, 7168, 33, vp(16), None) == -1    # top_k
    assert fin(vp(24), vp(16), None, 2, 7168, 8, vp(16), None) == -3     # out misaligned
    assert fin(vp(16), vp(18), None, 2, 7168, 8, vp(16), None) == -3     # weights misaligned
    assert fin(vp(16), vp(16), vp(8), 2, 7168, 8, vp(16), None) == -3    # shared_out misaligned


def test_fused_nvfp4_validation(fme):
    vp = ctypes.c_void_p

    def call(**kw):
        a = dict(x=vp(16), lg=vp(16), dt=0, bias=vp(16), w13=vp(16), s13=vp(16), w2=vp(16), s2=vp(16), M=4,
                 H=7168, N=3072, L=48, E=384, e0=0, k=6, scale=1.0, limit=float("inf"), y=vp(16), ids=vp(16),
                 w=vp(16), ws=vp(16), wsb=1 << 30, st=None)
        a.update(kw)
        return fme.lib.fme_moe_layer_nvfp4(*a.values())

    assert call(lg=None) == -1
    assert call(e0=340) == -1          # local range past E
    assert call(E=1025) == -2
    assert call(k=33) == -1
    assert call(dt=7) == -1
    assert call(scale=float("nan")) == -1
    assert call(M=65) == -2
    assert call(ids=vp(20)) == -3


def test_ep_local_validation(fme):
    vp = ctypes.c_void_p
    assert fme.lib.fme_mxfp8_quantize(vp(16), 2, 48, vp(16), vp(16), None) == -1     # H % 32
    assert fme.lib.fme_mxfp8_quantize(vp(16), 0, 64, vp(16), vp(16), None) == -1
    assert fme.lib.fme_mxfp8_quantize(vp(8), 2, 64, vp(16), vp(16), None) == -3
    comb = fme.lib.fme_combine_rmsnorm
    assert comb(vp(16), 2, 4, 8200, vp(16), 1e-5, vp(16), vp(16), None) == -1       # H > 8192
    assert comb(vp(16), 2, 0, 3584, vp(16), 1e-5, vp(16), vp(16), None) == -1
    assert comb(vp(16), 2, 4, 3584, vp(16), -1.0, vp(16), vp(16), None) == -1
    assert comb(vp(16), 2, 4, 3584, vp(24), 1e-5, vp(16), vp(16), None) == -3


def test_binding_exposes_a_wrapper_per_entry_point(fme):
    for name in ("moe_routed_fp8", "moe_routed_fp8_workspace", "moe_layer_fp8", "moe_layer_fp8_workspace",
                 "shared_expert_fp8", "shared_expert_fp8_workspace", "moe_routed_nvfp4",
                 "moe_routed_nvfp4_workspace", "ue8m0_unpack", "moe_finalize", "moe_layer_nvfp4", "mxfp8_quantize", "combine_rmsnorm", "moe_routed_fp8_mx"):
        assert callable(getattr(fme, name)), name


def _layer(fme, **kw):
    vp = ctypes.c_void_p
    args = dict(x=vp(16), logits=vp(16), dt=0, bias=vp(16), w13=vp(16), s13=vp(16), w2=vp(16), s2=vp(16),
                M=1, H=512, I=256, E=8, k=2, limit=7.0, scale=1.0, ue=0, sw13=vp(16), ss13=vp(16), sw2=vp(16),
                ss2=vp(16), slimit=7.0, sue=1, out=vp(16), ids=vp(16), weights=vp(16), sout=vp(16), ws=vp(16),
                wsb=1 << 20, st=None)
    args.update(kw)
    return fme.lib.fme_moe_layer_fp8(*args.values())


def test_layer_validation_and_workspace(fme):
    assert _layer(fme, sw13=None) == -1               # the shared expert is required
    assert _layer(fme, sout=None) == -1
    assert _layer(fme, slimit=0.0) == -1
    assert _layer(fme, M=65) == -2
    assert _layer(fme, k=9) == -1
    assert _layer(fme, ss2=ctypes.c_void_p(20)) == -3
    # the one-launch layer needs the routed call's bytes plus M hidden rows
    routed = fme.moe_routed_fp8_workspace(8, 7168, 2048, 256, 8)
    layer = fme.moe_layer_fp8_workspace(8, 7168, 2048, 256, 8)
    assert layer >= routed + 8 * 2048 * 4 - 256
    assert fme.moe_layer_fp8_workspace(0, 7168, 2048, 256, 8) == 0
    # a workspace too small for the call is refused before any launch
    assert _layer(fme, wsb=64) in (-6, -4)


def test_workspace_sizes_grow_with_tokens_and_fit_the_documented_limits(fme):
    """A workspace sized for M serves every smaller token count, the layer's
    holds the routed call's, and the no-allocation variant's 64 MiB scratch
    covers what its header says: DeepSeek-V3 up to 63 tokens, Latent up to 32."""
    for H, I, E, k in ((7168, 2048, 256, 8), (3584, 2048, 896, 16), (1024, 384, 40, 3)):
        prev = 0
        for M in range(1, 65):
            routed = fme.moe_routed_fp8_workspace(M, H, I, E, k)
            assert routed >= prev
            assert fme.moe_layer_fp8_workspace(M, H, I, E, k) >= routed
            prev = routed
    limit = 64 << 20
    assert fme.moe_routed_fp8_workspace(63, 7168, 2048, 256, 8) <= limit
    assert fme.moe_routed_fp8_workspace(64, 7168, 2048, 256, 8) > limit
    assert fme.moe_routed_fp8_workspace(32, 3584, 2048, 896, 16) <= limit
    assert fme.moe_routed_fp8_workspace(64, 3584, 2048, 896, 16) > limit


def test_noalloc_checks_arguments_before_touching_its_scratch(fme):
    """The allocation-free variant runs fme_moe_routed_fp8's host checks before
    any CUDA call, so these rejections need no GPU."""
    vp = ctypes.c_void_p
    null = vp(16)
    rc = fme.lib.fme_moe_routed_fp8_noalloc(None, null, 0, null, null, null, null, null, 1, 256, 128, 8, 2, 7.0,
                                            1.0, 0, null, null, null, None)
    assert rc == -1 and "null" in fme.lib.fme_last_error().decode()
    rc = fme.lib.fme_moe_routed_fp8_noalloc(null, null, 0, null, null, null, null, null, 1, 256, 100, 8, 2, 7.0,
                                            1.0, 0, null, null, null, None)
    assert rc == -1  # I not a multiple of 128
    rc = fme.lib.fme_moe_routed_fp8_noalloc(vp(24), null, 0, null, null, null, null, null, 1, 256, 128, 8, 2, 7.0,
                                            1.0, 0, null, null, null, None)
    assert rc == -3  # misaligned x
    assert fme.lib.fme_moe_routed_fp8_noalloc_error(None, None) == -1
