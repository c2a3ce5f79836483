"""The oracle: a plain CPU statement of the FP8 delayed-scaling linear layer.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import this package.  It shares no
code with the CUDA path (``fp8_delayed_scaling_gb300``) and imports nothing
from it.  The arithmetic lives in ``fp8_oracle.c`` (plain C, built with no FMA
contraction); this module only marshals numpy arrays into it and holds the
per-tensor scaling state as plain numpy arrays.

Sources are cited by page title and section, see ``fp8_oracle.c``.

Inputs are numpy arrays: ``float32`` for fp32 tensors, ``uint16`` holding the
bit patterns of bf16 tensors.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

E4M3 = 0
E5M2 = 1

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fp8_oracle.c")
_SO = os.path.join(_HERE, "liborc.so")
_lib = None
_lock = threading.Lock()

_i64 = ctypes.c_int64
_f32 = ctypes.c_float
_vp = ctypes.c_void_p


def build(force: bool = False) -> str:
    """Compile fp8_oracle.c into liborc.so (gcc, no FMA contraction)."""
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-std=c99", "-ffp-contract=off", "-fno-fast-math",
                               "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _SO)
    return _SO


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_SO)
            L.orc_fp8_decode.restype = ctypes.c_double
            L.orc_fp8_decode.argtypes = [ctypes.c_int, ctypes.c_uint8]
            L.orc_fp8_max.restype = ctypes.c_double
            L.orc_fp8_max.argtypes = [ctypes.c_int]
            L.orc_fp8_encode.restype = ctypes.c_uint8
            L.orc_fp8_encode.argtypes = [ctypes.c_int, ctypes.c_float]
            L.orc_quantize.restype = None
            L.orc_quantize.argtypes = [ctypes.c_int, _vp, ctypes.c_int, _i64, _f32, _vp]
            L.orc_amax.restype = ctypes.c_float
            L.orc_amax.argtypes = [_vp, ctypes.c_int, _i64]
            L.orc_colsum.restype = None
            L.orc_colsum.argtypes = [_vp, ctypes.c_int, _i64, _i64, _vp, _vp]
            L.orc_update_scale.restype = None
            L.orc_update_scale.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, _i64,
                                           _vp, _vp, _vp, _vp, _vp]
            L.orc_seed_history.restype = None
            L.orc_seed_history.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, _vp, _vp, _vp, _vp, _vp]
            L.orc_gemm_elems.restype = None
            L.orc_gemm_elems.argtypes = [_vp, ctypes.c_int, _vp, ctypes.c_int, _i64, _i64, _i64, _f32, _f32,
                                         _vp, ctypes.c_int, _i64, _vp, _vp, _vp, _vp]
            L.orc_e8m0_exponent.restype = ctypes.c_int
            L.orc_e8m0_exponent.argtypes = [ctypes.c_float]
            L.orc_mx_quantize_rows.restype = None
            L.orc_mx_quantize_rows.argtypes = [_vp, ctypes.c_int, _i64, _i64, _vp, _vp]
            L.orc_mx_gemm_elems.restype = None
            L.orc_mx_gemm_elems.argtypes = [_vp, _vp, _vp, _vp, _i64, _i64, _i64, _vp, ctypes.c_int,
                                            _i64, _vp, _vp, _vp, _vp]
            _lib = L
    return _lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


def _kind(x: np.ndarray) -> int:
    if x.dtype == np.float32:
        return 0
    if x.dtype == np.uint16:
        return 1
    raise TypeError("oracle inputs are float32 or uint16 (bf16 bits), got %s" % x.dtype)


def _threads(n_items: int, threads: int | None) -> int:
    t = threads if threads is not None else (os.cpu_count() or 1)
    return max(1, min(t, n_items // (1 << 16) + 1))


# --------------------------------------------------------------------------
# formats
# --------------------------------------------------------------------------
def fp8_max(fmt: int) -> float:
    return lib().orc_fp8_max(fmt)


def decode_table(fmt: int) -> np.ndarray:
    """Value of every one of the 256 codes (fp64; NaN for NaN codes)."""
    L = lib()
    return np.array([L.orc_fp8_decode(fmt, c) for c in range(256)], dtype=np.float64)


def encode(fmt: int, v: np.ndarray, threads: int | None = None) -> np.ndarray:
    """Encode fp32 values (no scaling)."""
    v = np.ascontiguousarray(v, dtype=np.float32)
    return quantize(fmt, v, 1.0, threads=threads)


# --------------------------------------------------------------------------
# per-tensor cast and amax
# --------------------------------------------------------------------------
def quantize(fmt: int, x: np.ndarray, scale: float, threads: int | None = None) -> np.ndarray:
    """q = enc(fl32(x * scale)) elementwise; same shape as x, uint8."""
    x = np.ascontiguousarray(x)
    k = _kind(x)
    flat = x.reshape(-1)
    out = np.empty(flat.shape, dtype=np.uint8)
    n = flat.size
    t = _threads(n, threads)
    L = lib()
    bounds = [n * i // t for i in range(t + 1)]

    def run(i):
        lo, hi = bounds[i], bounds[i + 1]
        if hi > lo:
            L.orc_quantize(fmt, flat.ctypes.data + lo * flat.itemsize, k, hi - lo, float(np.float32(scale)),
                           out.ctypes.data + lo)

    if t == 1:
        run(0)
    else:
        with ThreadPoolExecutor(t) as ex:
            list(ex.map(run, range(t)))
    return out.reshape(x.shape)


def amax(x: np.ndarray, threads: int | None = None) -> np.float32:
    """max |x| over all elements (fp32)."""
    x = np.ascontiguousarray(x)
    k = _kind(x)
    flat = x.reshape(-1)
    n = flat.size
    t = _threads(n, threads)
    L = lib()
    bounds = [n * i // t for i in range(t + 1)]

    def run(i):
        lo, hi = bounds[i], bounds[i + 1]
        return L.orc_amax(flat.ctypes.data + lo * flat.itemsize, k, hi - lo) if hi > lo else 0.0

    if t == 1:
        parts = [run(0)]
    else:
        with ThreadPoolExecutor(t) as ex:
            parts = list(ex.map(run, range(t)))
    return np.float32(max(parts))


def colsum(x: np.ndarray):
    """Column sums of a 2-D tensor in fp64, and the sums of |x| (for bounds)."""
    x = np.ascontiguousarray(x)
    rows, cols = x.shape
    s = np.empty(cols, np.float64)
    a = np.empty(cols, np.float64)
    lib().orc_colsum(_ptr(x), _kind(x), rows, cols, _ptr(s), _ptr(a))
    return s, a


# --------------------------------------------------------------------------
# delayed scaling state
# --------------------------------------------------------------------------
class ScalingState:
    """Per-tensor delayed-scaling state, one slot per scaled tensor.

    Holds scale, scale_inv, the amax recorded during the current step, and an
    amax history ring (length L) with its write position.
    """

    def __init__(self, slot_formats, hist_len: int, margin: int = 0, interval: int = 1):
        self.fmt = [int(f) for f in slot_formats]
        n = len(self.fmt)
        self.L = int(hist_len)
        self.margin = int(margin)
        self.interval = int(interval)
        self.scale = np.ones(n, np.float32)
        self.scale_inv = np.ones(n, np.float32)
        self.amax_cur = np.zeros(n, np.float32)
        self.pos = np.zeros(n, np.int32)
        self.hist = np.zeros((n, self.L), np.float32)

    @property
    def n_slots(self) -> int:
        return len(self.fmt)

    def record_amax(self, slot: int, value) -> None:
        """What a cast does to its slot: amax_cur = max(amax_cur, value)."""
        self.amax_cur[slot] = max(self.amax_cur[slot], np.float32(value))

    def _slot_ptrs(self, i):
        base = lambda a, it: a.ctypes.data + i * it  # noqa: E731
        return (self.hist.ctypes.data + i * self.L * 4, base(self.pos, 4), base(self.amax_cur, 4),
                base(self.scale, 4), base(self.scale_inv, 4))

    def update(self, step: int) -> None:
        L = lib()
        for i in range(self.n_slots):
            h, p, a, s, si = self._slot_ptrs(i)
            L.orc_update_scale(self.fmt[i], self.margin, self.interval, self.L, int(step), h, p, a, s, si)

    def seed(self) -> None:
        L = lib()
        for i in range(self.n_slots):
            h, p, a, s, si = self._slot_ptrs(i)
            L.orc_seed_history(self.fmt[i], self.margin, self.L, h, p, a, s, si)

    def window_max(self) -> np.ndarray:
        return self.hist.max(axis=1)


# --------------------------------------------------------------------------
# GEMMs
# --------------------------------------------------------------------------
def _bias_args(bias):
    if bias is None:
        return None, 0
    bias = np.ascontiguousarray(bias)
    return bias, _kind(bias)


def gemm_elems(A, afmt, B, bfmt, sa_inv, sb_inv, bias, ms, ns, threads: int | None = None):
    """Reference values of D = A * B^T at the listed (m, n) elements.

    Returns (ref, abs_ref), fp64: ref is the exact sum times fl32(sa_inv*sb_inv)
    plus bias; abs_ref the same sum over |products| (for the error bound).
    """
    A = np.ascontiguousarray(A, dtype=np.uint8)
    B = np.ascontiguousarray(B, dtype=np.uint8)
    M, K = A.shape
    N, K2 = B.shape
    assert K == K2
    ms = np.ascontiguousarray(ms, dtype=np.int64)
    ns = np.ascontiguousarray(ns, dtype=np.int64)
    n = ms.size
    ref = np.empty(n, np.float64)
    absr = np.empty(n, np.float64)
    bias, bk = _bias_args(bias)
    L = lib()
    t = max(1, min(threads or os.cpu_count() or 1, n))
    bounds = [n * i // t for i in range(t + 1)]

    def run(i):
        lo, hi = bounds[i], bounds[i + 1]
        if hi > lo:
            L.orc_gemm_elems(_ptr(A), afmt, _ptr(B), bfmt, M, N, K, float(np.float32(sa_inv)),
                             float(np.float32(sb_inv)), None if bias is None else _ptr(bias), bk, hi - lo,
                             ms.ctypes.data + 8 * lo, ns.ctypes.data + 8 * lo,
                             ref.ctypes.data + 8 * lo, absr.ctypes.data + 8 * lo)

    with ThreadPoolExecutor(t) as ex:
        list(ex.map(run, range(t)))
    return ref, absr


def e8m0_exponent(amax_b: float) -> int:
    return lib().orc_e8m0_exponent(float(np.float32(amax_b)))


def mx_quantize_rows(x: np.ndarray, threads: int | None = None):
    """Row-wise MXFP8 quantisation: (q [R x C] uint8, s [R x C/32] uint8)."""
    x = np.ascontiguousarray(x)
    R, C = x.shape
    assert C % 32 == 0
    q = np.empty((R, C), np.uint8)
    s = np.empty((R, C // 32), np.uint8)
    k = _kind(x)
    L = lib()
    t = _threads(R * C, threads)
    bounds = [R * i // t for i in range(t + 1)]

    def run(i):
        lo, hi = bounds[i], bounds[i + 1]
        if hi > lo:
            L.orc_mx_quantize_rows(x.ctypes.data + lo * C * x.itemsize, k, hi - lo, C,
                                   q.ctypes.data + lo * C, s.ctypes.data + lo * (C // 32))

    with ThreadPoolExecutor(t) as ex:
        list(ex.map(run, range(t)))
    return q, s


def mx_quantize_cols(x: np.ndarray, threads: int | None = None):
    """Column-wise MXFP8 quantisation (blocks of 32 along the rows), stored
    transposed: (q [C x R], s [C x R/32]) — the row-wise rule on x^T."""
    return mx_quantize_rows(np.ascontiguousarray(x.T), threads=threads)


def mx_gemm_elems(A, As, B, Bs, bias, ms, ns, threads: int | None = None):
    """Reference values of the block-scaled D = A * B^T at the listed elements."""
    A = np.ascontiguousarray(A, dtype=np.uint8)
    B = np.ascontiguousarray(B, dtype=np.uint8)
    As = np.ascontiguousarray(As, dtype=np.uint8)
    Bs = np.ascontiguousarray(Bs, dtype=np.uint8)
    M, K = A.shape
    N, K2 = B.shape
    assert K == K2 and K % 32 == 0 and As.shape == (M, K // 32) and Bs.shape == (N, K // 32)
    ms = np.ascontiguousarray(ms, dtype=np.int64)
    ns = np.ascontiguousarray(ns, dtype=np.int64)
    n = ms.size
    ref = np.empty(n, np.float64)
    absr = np.empty(n, np.float64)
    bias, bk = _bias_args(bias)
    L = lib()
    t = max(1, min(threads or os.cpu_count() or 1, n))
    bounds = [n * i // t for i in range(t + 1)]

    def run(i):
        lo, hi = bounds[i], bounds[i + 1]
        if hi > lo:
            L.orc_mx_gemm_elems(_ptr(A), _ptr(As), _ptr(B), _ptr(Bs), M, N, K,
                                None if bias is None else _ptr(bias), bk, hi - lo,
                                ms.ctypes.data + 8 * lo, ns.ctypes.data + 8 * lo,
                                ref.ctypes.data + 8 * lo, absr.ctypes.data + 8 * lo)

    with ThreadPoolExecutor(t) as ex:
        list(ex.map(run, range(t)))
    return ref, absr


# --------------------------------------------------------------------------
# LayerNormMLP pieces (fp64)
# --------------------------------------------------------------------------
def _sig_lnmlp(L):
    if getattr(L, "_lnmlp", False):
        return
    L.orc_layernorm_fwd.restype = None
    L.orc_layernorm_fwd.argtypes = [_vp, ctypes.c_int, _i64, _i64, _vp, _vp, ctypes.c_int, ctypes.c_double,
                                    _vp, _vp, _vp]
    L.orc_gelu.restype = None
    L.orc_gelu.argtypes = [_vp, ctypes.c_int, _i64, _vp]
    L.orc_dgelu.restype = None
    L.orc_dgelu.argtypes = [_vp, _vp, ctypes.c_int, _i64, _vp]
    L.orc_layernorm_bwd.restype = None
    L.orc_layernorm_bwd.argtypes = [_vp, _vp, ctypes.c_int, _i64, _i64, _vp, ctypes.c_int, _vp, _vp, _vp, _vp,
                                    _vp, _vp, _vp, _vp]
    L._lnmlp = True


def layernorm_fwd(x: np.ndarray, gamma: np.ndarray, beta: np.ndarray, eps: float = 1e-5):
    """(y, mu, rsigma) in fp64 for a 2-D x (float32 or bf16 bits)."""
    L = lib()
    _sig_lnmlp(L)
    x = np.ascontiguousarray(x)
    gamma, beta = np.ascontiguousarray(gamma), np.ascontiguousarray(beta)
    assert _kind(gamma) == _kind(beta)
    R, C = x.shape
    y = np.empty((R, C), np.float64)
    mu = np.empty(R, np.float64)
    rs = np.empty(R, np.float64)
    t = _threads(R * C, None)
    bounds = [R * i // t for i in range(t + 1)]

    def run(i):
        lo, hi = bounds[i], bounds[i + 1]
        if hi > lo:
            L.orc_layernorm_fwd(x.ctypes.data + lo * C * x.itemsize, _kind(x), hi - lo, C, _ptr(gamma), _ptr(beta),
                                _kind(gamma), float(eps), y.ctypes.data + lo * C * 8, mu.ctypes.data + lo * 8,
                                rs.ctypes.data + lo * 8)

    with ThreadPoolExecutor(t) as ex:
        list(ex.map(run, range(t)))
    return y, mu, rs


def gelu(h: np.ndarray) -> np.ndarray:
    L = lib()
    _sig_lnmlp(L)
    h = np.ascontiguousarray(h)
    out = np.empty(h.shape, np.float64)
    L.orc_gelu(_ptr(h), _kind(h), h.size, _ptr(out))
    return out


def dgelu(dg: np.ndarray, h: np.ndarray) -> np.ndarray:
    L = lib()
    _sig_lnmlp(L)
    dg, h = np.ascontiguousarray(dg), np.ascontiguousarray(h)
    assert dg.shape == h.shape and _kind(dg) == _kind(h)
    out = np.empty(h.shape, np.float64)
    L.orc_dgelu(_ptr(dg), _ptr(h), _kind(h), h.size, _ptr(out))
    return out


def layernorm_bwd(dy: np.ndarray, x: np.ndarray, gamma: np.ndarray, mu: np.ndarray, rsigma: np.ndarray):
    """(dx, dgamma, dbeta, dx_abs, dgamma_abs, dbeta_abs) in fp64."""
    L = lib()
    _sig_lnmlp(L)
    dy, x, gamma = np.ascontiguousarray(dy), np.ascontiguousarray(x), np.ascontiguousarray(gamma)
    mu = np.ascontiguousarray(mu, dtype=np.float64)
    rsigma = np.ascontiguousarray(rsigma, dtype=np.float64)
    assert _kind(dy) == _kind(x)
    R, C = x.shape
    dx = np.empty((R, C), np.float64)
    dxa = np.empty((R, C), np.float64)
    dg = np.empty(C, np.float64)
    db = np.empty(C, np.float64)
    dga = np.empty(C, np.float64)
    dba = np.empty(C, np.float64)
    L.orc_layernorm_bwd(_ptr(dy), _ptr(x), _kind(x), R, C, _ptr(gamma), _kind(gamma), _ptr(mu), _ptr(rsigma),
                        _ptr(dx), _ptr(dg), _ptr(db), _ptr(dxa), _ptr(dga), _ptr(dba))
    return dx, dg, db, dxa, dga, dba
