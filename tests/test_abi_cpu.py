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
