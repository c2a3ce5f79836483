"""Python binding of libfp8dl — the GB300 (sm_103a) FP8 delayed-scaling linear layer.

Argument marshalling only: every function here forwards device pointers and
sizes to the C ABI declared in ``include/fp8dl.h`` (same names), and every step
of the computation runs in the library's CUDA kernels.  There is no CPU
fallback: if ``libfp8dl.so`` is missing the import fails, and on a machine
without an sm_103 GPU the calls return FP8DL_ERR_UNSUPPORTED_DEVICE.

PyTorch is used for device memory and streams only.  Pointer arguments accept a
``torch.Tensor`` (its ``data_ptr()``), a plain integer device address, or None.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libfp8dl.so")

if not os.path.exists(LIB_PATH):
    raise ImportError("libfp8dl.so is not built (%s); run `python -c 'import __graft_entry__ as g; g.build()'`"
                      % LIB_PATH)
_lib = ctypes.CDLL(LIB_PATH)

# enums (include/fp8dl.h)
OK, ERR_INVALID_ARG, ERR_SHAPE, ERR_ALIGN, ERR_UNSUPPORTED_DEVICE, ERR_CUDA, ERR_TIMEOUT, ERR_WORKSPACE = range(8)
E4M3, E5M2 = 0, 1
F32, BF16 = 0, 1
FORMAT_E4M3, FORMAT_HYBRID = 0, 1
FP8_MAX = {E4M3: 448.0, E5M2: 57344.0}

_vp, _i32, _i64, _sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t


class fp8dl_recipe(ctypes.Structure):
    _fields_ = [("margin", _i32), ("interval", _i32), ("fp8_format", _i32), ("amax_history_len", _i32),
                ("amax_compute_algo", _i32)]


class fp8dl_cast_item(ctypes.Structure):
    """One tensor of fp8_cast_amax_transpose_multi (include/fp8dl.h)."""
    _fields_ = [("x", ctypes.c_void_p), ("rows", ctypes.c_int64), ("cols", ctypes.c_int64),
                ("scale", ctypes.c_void_p), ("out", ctypes.c_void_p), ("out_t", ctypes.c_void_p),
                ("amax", ctypes.c_void_p), ("scale_inv_out", ctypes.c_void_p)]


_SIGS = {
    "fp8dl_slot_stride": (_sz, [_i32]),
    "fp8dl_scaling_state_bytes": (_sz, [_i32, _i32]),
    "fp8_scaling_state_init": (_i32, [ctypes.POINTER(fp8dl_recipe), _i32, _vp, _vp, _vp]),
    "fp8_update_scale": (_i32, [ctypes.POINTER(fp8dl_recipe), _i32, _vp, _i64, _vp]),
    "fp8_seed_amax_history": (_i32, [ctypes.POINTER(fp8dl_recipe), _i32, _vp, _vp]),
    "fp8_cast_workspace_size": (_sz, [_i64, _i64]),
    "fp8_cast_amax_transpose": (_i32, [_vp, _i32, _i64, _i64, _i32, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp]),
    "fp8_cast_amax_transpose_noalloc": (_i32, [_vp, _i32, _i64, _i64, _i32, _vp, _vp, _vp, _vp, _vp, _vp]),
    "fp8_cast_amax_transpose_multi": (_i32, [_i32, ctypes.POINTER(fp8dl_cast_item), _i32, _i32, _vp]),
    "fp8_gemm": (_i32, [_vp, _i32, _vp, _i32, _i64, _i64, _i64, _vp, _vp, _vp, _i32, _vp, _i32, _vp, _vp]),
    "fp8_gemm_gelu_cast": (_i32, [_vp, _i32, _vp, _i32, _i64, _i64, _i64, _vp, _vp, _vp, _i32, _vp, _i32, _vp, _vp,
                                  _vp, _vp, _vp, _vp, _vp]),
    "fp8_gemm_dgelu_workspace_size": (_sz, [_i64, _i64]),
    "fp8_gemm_dgelu_cast": (_i32, [_vp, _i32, _vp, _i32, _i64, _i64, _i64, _vp, _vp, _vp, _vp, _i32, _vp, _vp, _vp,
                                   _vp, _vp, _vp, _sz, _vp, _vp, _vp]),
    "mxfp8_scale_bytes": (_sz, [_i64, _i64]),
    "mxfp8_quantize": (_i32, [_vp, _i32, _i64, _i64, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp]),
    "mxfp8_gemm": (_i32, [_vp, _vp, _vp, _vp, _i64, _i64, _i64, _vp, _i32, _vp, _i32, _vp, _vp]),
    "fp8_layernorm_cast": (_i32, [_vp, _i64, _i64, _vp, _vp, ctypes.c_float, _i32, _vp, _vp, _vp, _vp, _vp, _vp,
                                  _vp, _vp]),
    "fp8_gelu_cast": (_i32, [_vp, _i64, _i64, _i32, _vp, _vp, _vp, _vp, _vp, _vp]),
    "fp8_dgelu_cast": (_i32, [_vp, _vp, _i64, _i64, _i32, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp, _vp]),
    "fp8_layernorm_bwd_workspace_size": (_sz, [_i64, _i64]),
    "fp8_layernorm_bwd": (_i32, [_vp, _vp, _vp, _vp, _vp, _i64, _i64, _vp, _vp, _vp, _vp, _sz, _vp]),
    "fp8dl_wait_selftest": (_i32, [_i64, _i32, _vp, _vp]),
    "fp8dl_device_supported": (_i32, [_i32]),
    "fp8dl_clock_probe": (_i32, [_vp, _i32, _vp]),
    "fp8dl_last_error": (ctypes.c_char_p, []),
    "fp8dl_version": (_i32, []),
    "fp8dl_kernel_launches": (ctypes.c_uint64, []),
}
for _name, (_res, _args) in _SIGS.items():
    _f = getattr(_lib, _name)
    _f.restype = _res
    _f.argtypes = _args


class FP8DLError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__("%s failed with status %d: %s" % (where, status, fp8dl_last_error()))


def _check(status: int, where: str) -> None:
    if status != OK:
        raise FP8DLError(status, where)


def _p(x):
    if x is None:
        return None
    if isinstance(x, torch.Tensor):
        return x.data_ptr()
    return int(x)


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream if torch.cuda.is_available() else None
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _hp(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return F32
    if t.dtype == torch.bfloat16:
        return BF16
    raise TypeError("expected float32 or bfloat16, got %s" % t.dtype)


# --------------------------------------------------------------------------
# library state
# --------------------------------------------------------------------------
def fp8dl_last_error() -> str:
    return _lib.fp8dl_last_error().decode()


def fp8dl_version() -> int:
    return _lib.fp8dl_version()


def fp8dl_kernel_launches() -> int:
    """Kernels the library has enqueued in this process (graph replays not included)."""
    return _lib.fp8dl_kernel_launches()


def fp8dl_device_supported(device: int = 0) -> bool:
    return bool(_lib.fp8dl_device_supported(device))


def fp8dl_clock_probe(out, n_ctas: int, stream=None) -> None:
    """out: uint64 device tensor of 3 * n_ctas entries (SM id, cycle counter, ns timer per CTA)."""
    _check(_lib.fp8dl_clock_probe(_p(out), int(n_ctas), _stream(stream)), "fp8dl_clock_probe")


def fp8dl_wait_selftest(budget_cycles: int, arrive_first: bool, dev_status, stream=None) -> None:
    """Run the bounded-wait self-test; the outcome is written to dev_status (device int32)."""
    _check(_lib.fp8dl_wait_selftest(int(budget_cycles), 1 if arrive_first else 0, _p(dev_status), _stream(stream)),
           "fp8dl_wait_selftest")


def fp8dl_slot_stride(amax_history_len: int) -> int:
    return _lib.fp8dl_slot_stride(amax_history_len)


def fp8dl_scaling_state_bytes(amax_history_len: int, n_slots: int) -> int:
    return _lib.fp8dl_scaling_state_bytes(amax_history_len, n_slots)


def fp8_cast_workspace_size(rows: int, cols: int) -> int:
    return _lib.fp8_cast_workspace_size(rows, cols)


# --------------------------------------------------------------------------
# recipe + scaling state
# --------------------------------------------------------------------------
@dataclass
class Recipe:
    """DelayedScaling recipe: margin, interval, fp8_format, amax_history_len, "max"."""
    margin: int = 0
    interval: int = 1
    fp8_format: int = FORMAT_HYBRID
    amax_history_len: int = 16
    amax_compute_algo: int = 0

    def c(self) -> fp8dl_recipe:
        return fp8dl_recipe(self.margin, self.interval, self.fp8_format, self.amax_history_len,
                            self.amax_compute_algo)

    def fwd_dtype(self) -> int:
        return E4M3

    def bwd_dtype(self) -> int:
        return E5M2 if self.fp8_format == FORMAT_HYBRID else E4M3


def fp8_scaling_state_init(recipe: Recipe, slot_fp8_dtype, state, stream=None) -> None:
    n = len(slot_fp8_dtype)
    arr = (ctypes.c_int32 * n)(*[int(d) for d in slot_fp8_dtype])
    r = recipe.c()
    _check(_lib.fp8_scaling_state_init(ctypes.byref(r), n, ctypes.cast(arr, _vp), _p(state), _stream(stream)),
           "fp8_scaling_state_init")


def fp8_update_scale(recipe: Recipe, n_slots: int, state, step: int, stream=None) -> None:
    r = recipe.c()
    _check(_lib.fp8_update_scale(ctypes.byref(r), n_slots, _p(state), int(step), _stream(stream)),
           "fp8_update_scale")


def fp8_seed_amax_history(recipe: Recipe, n_slots: int, state, stream=None) -> None:
    r = recipe.c()
    _check(_lib.fp8_seed_amax_history(ctypes.byref(r), n_slots, _p(state), _stream(stream)),
           "fp8_seed_amax_history")


class ScalingState:
    """Device block holding the delayed-scaling state of `len(slot_fp8_dtype)` tensors."""

    def __init__(self, recipe: Recipe, slot_fp8_dtype, device="cuda", stream=None):
        self.recipe = recipe
        self.slot_fp8_dtype = [int(d) for d in slot_fp8_dtype]
        self.n_slots = len(self.slot_fp8_dtype)
        self.stride = fp8dl_slot_stride(recipe.amax_history_len)
        self.buf = torch.empty(fp8dl_scaling_state_bytes(recipe.amax_history_len, self.n_slots),
                               dtype=torch.uint8, device=device)
        fp8_scaling_state_init(recipe, self.slot_fp8_dtype, self.buf, stream)

    def _addr(self, slot: int, off: int) -> int:
        assert 0 <= slot < self.n_slots
        return self.buf.data_ptr() + slot * self.stride + off

    def scale(self, slot: int) -> int:
        return self._addr(slot, 0)

    def scale_inv(self, slot: int) -> int:
        return self._addr(slot, 4)

    def amax(self, slot: int) -> int:
        return self._addr(slot, 8)

    def update(self, step: int, stream=None) -> None:
        fp8_update_scale(self.recipe, self.n_slots, self.buf, step, stream)

    def seed(self, stream=None) -> None:
        fp8_seed_amax_history(self.recipe, self.n_slots, self.buf, stream)

    def read(self) -> dict:
        """Host copy of every slot's fields (synchronises)."""
        raw = self.buf.cpu()
        L = self.recipe.amax_history_len
        rows = raw.view(self.n_slots, self.stride)
        hdr = rows[:, :32].contiguous()
        f = hdr.view(torch.float32)
        i = hdr.view(torch.int32)
        hist = rows[:, 32:32 + 4 * L].contiguous().view(torch.float32)
        return {"scale": f[:, 0].numpy().copy(), "scale_inv": f[:, 1].numpy().copy(),
                "amax": f[:, 2].numpy().copy(), "pos": i[:, 3].numpy().copy(),
                "fp8_dtype": i[:, 4].numpy().copy(), "hist": hist.numpy().copy()}


# --------------------------------------------------------------------------
# kernels
# --------------------------------------------------------------------------
def fp8_cast_amax_transpose(x: torch.Tensor, out_dtype: int, scale, out=None, out_t=None, amax=None, dbias=None,
                            workspace=None, scale_inv_out=None, stream=None) -> None:
    assert x.dim() == 2 and x.is_contiguous()
    rows, cols = x.shape
    ws_bytes = workspace.numel() * workspace.element_size() if isinstance(workspace, torch.Tensor) else 0
    _check(_lib.fp8_cast_amax_transpose(_p(x), _hp(x), rows, cols, out_dtype, _p(scale), _p(out), _p(out_t),
                                        _p(amax), _p(scale_inv_out), _p(dbias), _p(workspace), ws_bytes,
                                        _stream(stream)),
           "fp8_cast_amax_transpose")


def fp8_cast_amax_transpose_multi(items, out_dtype: int, stream=None) -> None:
    """Grouped cast: items is a list of dicts with keys x, scale, and any of out, out_t, amax,
    scale_inv_out (as for fp8_cast_amax_transpose, without dbias); one launch for all."""
    n = len(items)
    arr = (fp8dl_cast_item * n)()
    x_dtype = None
    for k, it in enumerate(items):
        x = it["x"]
        assert x.dim() == 2 and x.is_contiguous()
        if x_dtype is None:
            x_dtype = _hp(x)
        assert _hp(x) == x_dtype, "all items share one input dtype"
        arr[k] = fp8dl_cast_item(_p(x), x.shape[0], x.shape[1], _p(it.get("scale")), _p(it.get("out")),
                                 _p(it.get("out_t")), _p(it.get("amax")), _p(it.get("scale_inv_out")))
    _check(_lib.fp8_cast_amax_transpose_multi(n, arr, x_dtype if x_dtype is not None else BF16, out_dtype,
                                              _stream(stream)), "fp8_cast_amax_transpose_multi")


def fp8_cast_amax_transpose_noalloc(x: torch.Tensor, out_dtype: int, scale, out=None, out_t=None, amax=None,
                                    dbias=None, stream=None) -> None:
    """fp8_cast_amax_transpose for callers that cannot allocate device memory:
    the bias-gradient scratch is the library's own 4 MiB static device array
    (ceil(rows/128) * cols * 4 bytes must fit).  Calls on one device share
    that array, so concurrent calls must be ordered on one stream."""
    assert x.dim() == 2 and x.is_contiguous()
    rows, cols = x.shape
    _check(_lib.fp8_cast_amax_transpose_noalloc(_p(x), _hp(x), rows, cols, out_dtype, _p(scale), _p(out),
                                                _p(out_t), _p(amax), _p(dbias), _stream(stream)),
           "fp8_cast_amax_transpose_noalloc")


def fp8_gemm(A: torch.Tensor, a_dtype: int, B: torch.Tensor, b_dtype: int, a_scale_inv, b_scale_inv, D: torch.Tensor,
             bias: torch.Tensor | None = None, dev_status=None, stream=None) -> None:
    """D[M,N] = (A[M,K] * B[N,K]^T) * a_scale_inv * b_scale_inv + bias."""
    M, K = A.shape
    N, K2 = B.shape
    assert K == K2 and tuple(D.shape) == (M, N)
    _check(_lib.fp8_gemm(_p(A), a_dtype, _p(B), b_dtype, M, N, K, _p(a_scale_inv), _p(b_scale_inv), _p(bias),
                         _hp(bias) if bias is not None else BF16, _p(D), _hp(D), _p(dev_status), _stream(stream)),
           "fp8_gemm")


def fp8_gemm_gelu_cast(A: torch.Tensor, a_dtype: int, B: torch.Tensor, b_dtype: int, a_scale_inv, b_scale_inv,
                       H: torch.Tensor, q_dtype: int, q_scale, q: torch.Tensor, q_t: torch.Tensor, q_amax=None,
                       bias: torch.Tensor | None = None, g=None, dev_status=None, stream=None) -> None:
    """H = A*B^T*sa_inv*sb_inv + bias (bf16); q, q^T = FP8 codes of GELU(H) at q_scale; amax of GELU(H)."""
    M, K = A.shape
    N, K2 = B.shape
    assert K == K2 and tuple(H.shape) == (M, N) and H.dtype == torch.bfloat16
    _check(_lib.fp8_gemm_gelu_cast(_p(A), a_dtype, _p(B), b_dtype, M, N, K, _p(a_scale_inv), _p(b_scale_inv), _p(bias),
                                   _hp(bias) if bias is not None else BF16, _p(H), q_dtype, _p(q_scale), _p(q), _p(q_t),
                                   _p(q_amax), _p(g), _p(dev_status), _stream(stream)), "fp8_gemm_gelu_cast")


def fp8_gemm_dgelu_workspace_size(M: int, N: int) -> int:
    return _lib.fp8_gemm_dgelu_workspace_size(M, N)


def fp8_gemm_dgelu_cast(A: torch.Tensor, a_dtype: int, B: torch.Tensor, b_dtype: int, a_scale_inv, b_scale_inv,
                        h: torch.Tensor, q_dtype: int, q_scale, q: torch.Tensor, q_t: torch.Tensor, q_amax=None,
                        dbias=None, workspace=None, dg=None, dh=None, dev_status=None, stream=None) -> None:
    """dg = A*B^T*sa_inv*sb_inv (bf16, not stored unless dg is given); q, q^T = FP8 codes of
    dh = bf16(dg * GELU'(h)) at q_scale; amax |dh|; dbias = column sums of dh."""
    M, K = A.shape
    N, K2 = B.shape
    assert K == K2 and tuple(h.shape) == (M, N) and h.dtype == torch.bfloat16
    ws_bytes = workspace.numel() * workspace.element_size() if isinstance(workspace, torch.Tensor) else 0
    _check(_lib.fp8_gemm_dgelu_cast(_p(A), a_dtype, _p(B), b_dtype, M, N, K, _p(a_scale_inv), _p(b_scale_inv), _p(h),
                                    _p(dg), q_dtype, _p(q_scale), _p(q), _p(q_t), _p(q_amax), _p(dbias),
                                    _p(workspace), ws_bytes, _p(dh), _p(dev_status), _stream(stream)),
           "fp8_gemm_dgelu_cast")


def mxfp8_scale_bytes(rows: int, cols: int) -> int:
    """Bytes of the tiled E8M0 scale buffer of an MXFP8 [rows x cols] matrix (blocks along cols)."""
    return _lib.mxfp8_scale_bytes(rows, cols)


def mxfp8_quantize(x: torch.Tensor, row_q=None, row_s=None, col_q=None, col_s=None, dbias=None, workspace=None,
                   stream=None) -> None:
    """Row- and/or column-wise MXFP8 codes and tiled E8M0 scales of x; dbias (fp32 [cols])
    receives the column sums of x in the same pass (workspace: fp8_cast_workspace_size bytes)."""
    assert x.dim() == 2 and x.is_contiguous()
    rows, cols = x.shape
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(_lib.mxfp8_quantize(_p(x), _hp(x), rows, cols, _p(row_q), _p(row_s), _p(col_q), _p(col_s), _p(dbias),
                               _p(workspace), ws_bytes, _stream(stream)), "mxfp8_quantize")


def mxfp8_gemm(A, A_s, B, B_s, D: torch.Tensor, bias: torch.Tensor | None = None, dev_status=None,
               stream=None) -> None:
    """D[M,N] = sum over 32-blocks of 2^(ea+eb) * (A_blk * B_blk^T) + bias."""
    M, K = A.shape
    N, K2 = B.shape
    assert K == K2 and tuple(D.shape) == (M, N)
    _check(_lib.mxfp8_gemm(_p(A), _p(A_s), _p(B), _p(B_s), M, N, K, _p(bias),
                           _hp(bias) if bias is not None else BF16, _p(D), _hp(D), _p(dev_status), _stream(stream)),
           "mxfp8_gemm")


# --------------------------------------------------------------------------
# LayerNormMLP pieces (bf16 tensors)
# --------------------------------------------------------------------------
def _nbytes(t):
    return t.numel() * t.element_size() if isinstance(t, torch.Tensor) else 0


def fp8_layernorm_cast(x: torch.Tensor, gamma: torch.Tensor, beta: torch.Tensor, eps: float, out_dtype: int, scale,
                       mu: torch.Tensor, rsigma: torch.Tensor, out=None, out_t=None, amax=None, y=None,
                       stream=None) -> None:
    assert x.dtype == torch.bfloat16 and x.dim() == 2 and x.is_contiguous()
    rows, cols = x.shape
    _check(_lib.fp8_layernorm_cast(_p(x), rows, cols, _p(gamma), _p(beta), float(eps), out_dtype, _p(scale),
                                   _p(out), _p(out_t), _p(amax), _p(mu), _p(rsigma), _p(y), _stream(stream)),
           "fp8_layernorm_cast")


def fp8_gelu_cast(h: torch.Tensor, out_dtype: int, scale, out=None, out_t=None, amax=None, g=None,
                  stream=None) -> None:
    assert h.dtype == torch.bfloat16 and h.dim() == 2 and h.is_contiguous()
    rows, cols = h.shape
    _check(_lib.fp8_gelu_cast(_p(h), rows, cols, out_dtype, _p(scale), _p(out), _p(out_t), _p(amax), _p(g),
                              _stream(stream)), "fp8_gelu_cast")


def fp8_dgelu_cast(dg: torch.Tensor, h: torch.Tensor, out_dtype: int, scale, out=None, out_t=None, amax=None,
                   dbias=None, workspace=None, dh=None, stream=None) -> None:
    assert dg.dtype == torch.bfloat16 and h.dtype == torch.bfloat16 and dg.shape == h.shape
    rows, cols = h.shape
    _check(_lib.fp8_dgelu_cast(_p(dg), _p(h), rows, cols, out_dtype, _p(scale), _p(out), _p(out_t), _p(amax),
                               _p(dbias), _p(workspace), _nbytes(workspace), _p(dh), _stream(stream)),
           "fp8_dgelu_cast")


def fp8_layernorm_bwd_workspace_size(rows: int, cols: int) -> int:
    return _lib.fp8_layernorm_bwd_workspace_size(rows, cols)


def fp8_layernorm_bwd(dy: torch.Tensor, x: torch.Tensor, gamma: torch.Tensor, mu, rsigma, dx: torch.Tensor,
                      dgamma: torch.Tensor, dbeta: torch.Tensor, workspace: torch.Tensor, stream=None) -> None:
    rows, cols = x.shape
    _check(_lib.fp8_layernorm_bwd(_p(dy), _p(x), _p(gamma), _p(mu), _p(rsigma), rows, cols, _p(dx), _p(dgamma),
                                  _p(dbeta), _p(workspace), _nbytes(workspace), _stream(stream)),
           "fp8_layernorm_bwd")


from .autocast import fp8_autocast  # noqa: E402  (the step region; see autocast.py)
