"""The C-ABI library loads, exports every declared symbol, and validates
arguments on the host (CPU only: no compute call reaches a GPU here)."""
import ctypes
import os
import re

import pytest

from conftest import ROOT

HEADER = os.path.join(ROOT, "include", "fp8dl.h")


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    import fp8_delayed_scaling_gb300 as fd
    return fd


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b([a-z_][a-z0-9_]*)\s*\(", src)) - {"if", "sizeof"})


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("fp8_update_scale", "fp8_cast_amax_transpose", "fp8_gemm", "mxfp8_quantize", "mxfp8_gemm"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    so = ctypes.CDLL(lib.LIB_PATH)
    missing = [n for n in declared_functions() if not hasattr(so, n)]
    assert not missing, missing


def test_binding_has_the_same_names(lib):
    for n in declared_functions():
        assert hasattr(lib, n), n


def test_state_layout_sizes(lib):
    assert lib.fp8dl_slot_stride(1) == 48
    assert lib.fp8dl_slot_stride(16) == 96
    assert lib.fp8dl_slot_stride(1024) == 32 + 4096
    assert lib.fp8dl_scaling_state_bytes(16, 9) == 9 * 96
    assert lib.fp8dl_slot_stride(0) == 0
    assert lib.fp8_cast_workspace_size(2048, 3072) == 16 * 3072 * 4
    assert lib.fp8_cast_workspace_size(144, 32) == 2 * 32 * 4


def _raw(lib):
    return lib._lib


def test_host_validation_without_gpu(lib):
    L = _raw(lib)
    a16 = 1 << 20  # a fake, 16-byte aligned address: validation fails before any use
    # NULL input
    assert L.fp8_cast_amax_transpose(None, 1, 32, 32, 0, a16, a16, None, None, None, None, None, 0, None) == lib.ERR_INVALID_ARG
    # empty inputs: rejected before any launch (every dimension must be a positive multiple of 16)
    assert L.fp8_cast_amax_transpose(a16, 1, 0, 32, 0, a16, a16, None, None, None, None, None, 0, None) == lib.ERR_SHAPE
    assert L.fp8_cast_amax_transpose(a16, 1, 32, 0, 0, a16, a16, None, None, None, None, None, 0, None) == lib.ERR_SHAPE
    assert L.fp8_gemm(a16, 0, a16, 0, 0, 16, 16, a16, a16, None, 1, a16, 1, None, None) == lib.ERR_SHAPE
    assert L.fp8_gemm(a16, 0, a16, 0, 16, 16, 0, a16, a16, None, 1, a16, 1, None, None) == lib.ERR_SHAPE
    assert L.mxfp8_quantize(a16, 1, 0, 32, a16, a16, None, None, None, None, 0, None) == lib.ERR_SHAPE
    assert L.mxfp8_gemm(a16, a16, a16, a16, 32, 0, 32, None, 1, a16, 1, None, None) == lib.ERR_SHAPE
    # dimension not a multiple of 16
    assert L.fp8_cast_amax_transpose(a16, 1, 33, 32, 0, a16, a16, None, None, None, None, None, 0, None) == lib.ERR_SHAPE
    assert L.fp8_gemm(a16, 0, a16, 0, 16, 24, 16, a16, a16, None, 1, a16, 1, None, None) == lib.ERR_SHAPE
    # misaligned pointer
    assert L.fp8_cast_amax_transpose(a16 + 8, 1, 32, 32, 0, a16, a16, None, None, None, None, None, 0, None) == lib.ERR_ALIGN
    # dbias without workspace
    assert L.fp8_cast_amax_transpose(a16, 1, 32, 32, 0, a16, a16, None, None, None, a16, None, 0, None) == lib.ERR_WORKSPACE
    # a decode-factor output without a scale
    assert L.fp8_cast_amax_transpose(a16, 1, 32, 32, 0, None, None, None, a16, a16, None, None, 0, None) == lib.ERR_INVALID_ARG
    # bad dtype enums
    assert L.fp8_gemm(a16, 2, a16, 0, 16, 16, 16, a16, a16, None, 1, a16, 1, None, None) == lib.ERR_INVALID_ARG
    assert L.mxfp8_quantize(a16, 1, 48, 32, a16, a16, None, None, None, None, 0, None) == lib.ERR_SHAPE
    # grouped cast: item count out of range, a ragged item (checked before any launch)
    items = (lib.fp8dl_cast_item * 2)(lib.fp8dl_cast_item(a16, 32, 32, a16, a16, None, None, None),
                                      lib.fp8dl_cast_item(a16, 40, 32, a16, a16, None, None, None))
    assert L.fp8_cast_amax_transpose_multi(0, items, 1, 0, None) == lib.ERR_INVALID_ARG
    assert L.fp8_cast_amax_transpose_multi(9, items, 1, 0, None) == lib.ERR_INVALID_ARG
    assert L.fp8_cast_amax_transpose_multi(2, items, 1, 0, None) == lib.ERR_SHAPE
    # MX bias gradient without workspace
    assert L.mxfp8_quantize(a16, 1, 64, 32, a16, a16, None, None, a16, None, 0, None) == lib.ERR_WORKSPACE
    assert L.mxfp8_gemm(a16, a16, a16, a16, 32, 32, 48, None, 1, a16, 1, None, None) == lib.ERR_SHAPE
    # clock probe: NULL output, CTA count out of range, misaligned output
    assert L.fp8dl_clock_probe(None, 4, None) == lib.ERR_INVALID_ARG
    assert L.fp8dl_clock_probe(a16, 0, None) == lib.ERR_INVALID_ARG
    assert L.fp8dl_clock_probe(a16 + 8, 4, None) == lib.ERR_ALIGN
    r = lib.fp8dl_recipe(0, 0, 1, 16, 0)  # interval 0 is invalid
    assert L.fp8_update_scale(ctypes.byref(r), 3, a16, 0, None) == lib.ERR_INVALID_ARG
    r = lib.fp8dl_recipe(-1, 1, 1, 16, 0)
    assert L.fp8_update_scale(ctypes.byref(r), 3, a16, 0, None) == lib.ERR_INVALID_ARG
    r = lib.fp8dl_recipe(0, 1, 1, 16, 1)  # only "max" is defined
    assert L.fp8_update_scale(ctypes.byref(r), 3, a16, 0, None) == lib.ERR_INVALID_ARG
    assert lib.fp8dl_last_error() != ""


def test_layernorm_mlp_entry_validation_without_gpu(lib):
    """The LayerNormMLP entry points (LayerNorm forward/backward, GELU/dGELU casts, the fused
    GELU/dGELU GEMMs) reject bad arguments on the host, with the status the header names."""
    L = _raw(lib)
    a = 1 << 20  # a fake, 16-byte aligned address: validation fails before any use
    E4, E5, BF = lib.E4M3, lib.E5M2, lib.BF16
    ln = lambda x=a, rows=32, cols=64, g=a, b=a, eps=1e-5, fmt=E4, sc=a, out=a, mu=a: L.fp8_layernorm_cast(  # noqa: E731
        x, rows, cols, g, b, eps, fmt, sc, out, None, None, mu, a, None, None)
    assert ln(x=None) == lib.ERR_INVALID_ARG
    assert ln(mu=None) == lib.ERR_INVALID_ARG
    assert ln(fmt=2) == lib.ERR_INVALID_ARG
    assert ln(sc=None) == lib.ERR_INVALID_ARG  # an FP8 output needs its scale
    assert ln(eps=-1.0) == lib.ERR_INVALID_ARG
    assert ln(rows=0) == lib.ERR_SHAPE
    assert ln(cols=24) == lib.ERR_SHAPE
    assert ln(cols=8192 + 16) == lib.ERR_SHAPE  # widest row: 8192
    assert ln(g=a + 8) == lib.ERR_ALIGN
    assert ln(out=a + 4) == lib.ERR_ALIGN
    ws_ln = lib.fp8_layernorm_bwd_workspace_size(32, 64)
    assert ws_ln > 0 and lib.fp8_layernorm_bwd_workspace_size(0, 64) == 0
    lnb = lambda dx=a, rows=32, ws=a, wsb=ws_ln: L.fp8_layernorm_bwd(a, a, a, a, a, rows, 64, dx, a, a, ws, wsb,  # noqa: E731
                                                                     None)
    assert lnb(dx=None) == lib.ERR_INVALID_ARG
    assert lnb(rows=33) == lib.ERR_SHAPE
    assert lnb(dx=a + 2) == lib.ERR_ALIGN
    assert lnb(ws=a + 8) == lib.ERR_ALIGN
    assert lnb(ws=None) == lib.ERR_WORKSPACE
    assert lnb(wsb=ws_ln - 1) == lib.ERR_WORKSPACE
    # GELU / dGELU casts
    assert L.fp8_gelu_cast(a, 32, 64, E4, a, None, None, None, None, None) == lib.ERR_INVALID_ARG  # nothing to do
    assert L.fp8_gelu_cast(a, 32, 64, E4, None, a, None, None, None, None) == lib.ERR_INVALID_ARG  # no scale
    assert L.fp8_gelu_cast(a, 32, 40, E4, a, a, None, None, None, None) == lib.ERR_SHAPE
    assert L.fp8_gelu_cast(a, 32, 64, E4, a, a + 8, None, None, None, None) == lib.ERR_ALIGN
    assert L.fp8_dgelu_cast(a, None, 32, 64, E5, a, a, None, None, None, None, 0, None, None) == lib.ERR_INVALID_ARG
    ws_c = lib.fp8_cast_workspace_size(32, 64)
    assert L.fp8_dgelu_cast(a, a, 32, 64, E5, a, a, None, None, a, None, 0, None, None) == lib.ERR_WORKSPACE
    assert L.fp8_dgelu_cast(a, a, 32, 64, E5, a, a, None, None, a, a, ws_c - 1, None, None) == lib.ERR_WORKSPACE
    assert L.fp8_dgelu_cast(a, a, 32, 64, E5, a, a, None, None, a, a + 8, ws_c, None, None) == lib.ERR_ALIGN
    # fused GELU GEMM: the GEMM's own checks, then the cast's
    gg = lambda N=64, q=a, qt=a, qfmt=E4, qs=a, H=a: L.fp8_gemm_gelu_cast(  # noqa: E731
        a, E4, a, E4, 32, N, 64, a, a, None, BF, H, qfmt, qs, q, qt, None, None, None, None)
    assert gg(N=24) == lib.ERR_SHAPE
    assert gg(H=None) == lib.ERR_INVALID_ARG
    assert gg(qfmt=3) == lib.ERR_INVALID_ARG
    assert gg(q=None) == lib.ERR_INVALID_ARG
    assert gg(qs=None) == lib.ERR_INVALID_ARG
    assert gg(qt=a + 8) == lib.ERR_ALIGN
    # fused dGELU GEMM (its dg output is optional); the bias gradient needs its workspace
    ws_d = lib.fp8_gemm_dgelu_workspace_size(32, 64)
    assert ws_d == 1 * 64 * 4 and lib.fp8_gemm_dgelu_workspace_size(33, 64) == 2 * 64 * 4
    dgg = lambda h=a, db=None, ws=None, wsb=0, q=a, dh=None: L.fp8_gemm_dgelu_cast(  # noqa: E731
        a, E5, a, E4, 32, 64, 64, a, a, h, None, E5, a, q, a, None, db, ws, wsb, dh, None, None)
    assert dgg(h=None) == lib.ERR_INVALID_ARG
    assert dgg(q=None) == lib.ERR_INVALID_ARG
    assert dgg(dh=a + 8) == lib.ERR_ALIGN
    assert dgg(db=a) == lib.ERR_WORKSPACE
    assert dgg(db=a, ws=a, wsb=ws_d - 1) == lib.ERR_WORKSPACE
    assert dgg(db=a, ws=a + 8, wsb=ws_d) == lib.ERR_ALIGN
    assert lib.fp8dl_last_error() != ""


def test_valid_call_without_gpu_fails_loudly(lib):
    """No GPU: a well-formed call must fail (no CPU fallback), never compute."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    L = _raw(lib)
    a16 = 1 << 20
    st = L.fp8_cast_amax_transpose(a16, 1, 32, 32, 0, a16, a16, None, None, None, None, None, 0, None)
    assert st in (lib.ERR_CUDA, lib.ERR_UNSUPPORTED_DEVICE)
    assert lib.fp8dl_device_supported(0) is False


def test_weight_cache_reuse_without_a_cast_raises_before_any_launch(lib):
    """is_first_microbatch=False with nothing cached is a host-side error (no launch)."""
    import torch
    from fp8_delayed_scaling_gb300.linear import Fp8Linear, WeightCache
    wc = WeightCache(torch.empty((32, 16), dtype=torch.uint8), None)
    wc.check(None)
    wc.check(True)
    with pytest.raises(RuntimeError):
        wc.check(False)
    import types
    recipe = lib.Recipe(margin=0, interval=1, fp8_format=lib.FORMAT_HYBRID, amax_history_len=4)
    state = types.SimpleNamespace(recipe=recipe)  # never touched: the check comes first
    lin = Fp8Linear(state, 0, torch.zeros((32, 16), dtype=torch.bfloat16), None, 16)
    with pytest.raises(RuntimeError):
        lin.forward(torch.zeros((16, 16), dtype=torch.bfloat16), is_first_microbatch=False)
