"""Pins of the oracle against what the pages and mathematics fix (CPU only).

Each test checks the oracle against something other than itself: hand-derived
values (tests/golden/, each with its citation), an independent library routine
(torch's float8 conversions, numpy's matmul), closed forms, invariants, or
brute force on tiny inputs.
"""
import math
import struct

import numpy as np
import pytest
import torch

import oracle
from conftest import golden_lines

FMT = {"E4M3": oracle.E4M3, "E5M2": oracle.E5M2}
TORCH_FP8 = {oracle.E4M3: torch.float8_e4m3fn, oracle.E5M2: torch.float8_e5m2}


def f32_hex(x):
    return struct.unpack("<I", struct.pack("<f", float(x)))[0]


def hex_f32(h):
    return struct.unpack("<f", struct.pack("<I", int(h, 16)))[0]


# --------------------------------------------------------------------------
# formats
# --------------------------------------------------------------------------
def test_decode_golden():
    for fmt, code, val in golden_lines("fp8_codes.txt"):
        got = oracle.decode_table(FMT[fmt])[int(code, 16)]
        want = float(val)
        if math.isnan(want):
            assert math.isnan(got), (fmt, code)
        else:
            assert got == want and math.copysign(1, got) == math.copysign(1, want), (fmt, code, got, want)


@pytest.mark.parametrize("fmt", [oracle.E4M3, oracle.E5M2])
def test_decode_matches_torch_for_all_codes(fmt):
    mine = oracle.decode_table(fmt)
    lib = torch.arange(256, dtype=torch.uint8).view(TORCH_FP8[fmt]).to(torch.float64).numpy()
    nan = np.isnan(lib)
    assert np.array_equal(np.isnan(mine), nan)
    assert np.array_equal(mine[~nan], lib[~nan])
    assert np.array_equal(np.signbit(mine[~nan]), np.signbit(lib[~nan]))


def test_format_maxima_and_counts():
    # E4M3 max 448 (the page's range); E5M2 max 57344 (the page's 57334 garbled)
    assert oracle.fp8_max(oracle.E4M3) == 448.0
    assert oracle.fp8_max(oracle.E5M2) == 57344.0
    t4, t5 = oracle.decode_table(oracle.E4M3), oracle.decode_table(oracle.E5M2)
    assert np.isnan(t4).sum() == 2 and np.isinf(t4).sum() == 0
    assert np.isnan(t5).sum() == 6 and np.isinf(t5).sum() == 2
    assert np.nanmax(t4) == 448.0 and np.nanmax(t5[np.isfinite(t5)]) == 57344.0


@pytest.mark.parametrize("fmt", [oracle.E4M3, oracle.E5M2])
def test_roundtrip_all_codes(fmt):
    t = oracle.decode_table(fmt)
    codes = np.array([c for c in range(256) if np.isfinite(t[c])], dtype=np.uint8)
    got = oracle.encode(fmt, t[codes].astype(np.float32))
    assert np.array_equal(got, codes)


@pytest.mark.parametrize("fmt", [oracle.E4M3, oracle.E5M2])
def test_midpoints_tie_to_even(fmt):
    t = oracle.decode_table(fmt)
    top = 0x7E if fmt == oracle.E4M3 else 0x7B
    for c in range(top):
        lo, hi = t[c], t[c + 1]
        mid = np.float32((lo + hi) / 2)
        assert float(mid) == (lo + hi) / 2  # exact in fp32
        even = c if c % 2 == 0 else c + 1
        for sign in (1, -1):
            got = int(oracle.encode(fmt, np.array([sign * mid], np.float32))[0])
            assert got == (even | (0x80 if sign < 0 else 0)), (c, sign)


@pytest.mark.parametrize("fmt", [oracle.E4M3, oracle.E5M2])
def test_encode_matches_torch_in_range(fmt):
    """In range, torch's float8 conversion (round to nearest even) is an independent encoder."""
    rng = np.random.default_rng(7)
    mx = oracle.fp8_max(fmt)
    t = oracle.decode_table(fmt)
    fin = t[np.isfinite(t)]
    mids = ((np.sort(fin)[1:] + np.sort(fin)[:-1]) / 2).astype(np.float32)
    v = np.concatenate([
        rng.uniform(-mx, mx, 200000),
        rng.standard_normal(200000) * 10.0 ** rng.integers(-6, 3, 200000),
        mids, np.nextafter(mids, np.float32(np.inf)), np.nextafter(mids, np.float32(-np.inf)),
    ]).astype(np.float32)
    v = v[np.abs(v) <= mx]
    mine = oracle.encode(fmt, v)
    lib = torch.from_numpy(v).to(TORCH_FP8[fmt]).view(torch.uint8).numpy()
    bad = np.nonzero(mine != lib)[0]
    assert bad.size == 0, [(float(v[i]), int(mine[i]), int(lib[i])) for i in bad[:5]]


def test_encode_golden():
    for fmt, val, code in golden_lines("fp8_encode.txt"):
        got = int(oracle.encode(FMT[fmt], np.array([float(val)], np.float32))[0])
        assert got == int(code, 16), (fmt, val, hex(got))


@pytest.mark.parametrize("fmt", [oracle.E4M3, oracle.E5M2])
def test_encode_monotone_and_nan(fmt):
    v = np.sort(np.random.default_rng(3).uniform(-1e5, 1e5, 100000).astype(np.float32))
    dec = oracle.decode_table(fmt)[oracle.encode(fmt, v)]
    assert np.all(np.diff(dec) >= 0)
    q = oracle.encode(fmt, np.array([np.nan, -np.nan], np.float32))
    assert np.all(np.isnan(oracle.decode_table(fmt)[q]))


def test_quantize_rounds_product_to_fp32_first():
    """q = enc(fl32(x*scale)): find x, s whose exact product lies just off an
    E4M3 midpoint but whose fp32 product is the midpoint itself; the tie rule
    then decides, unlike an encoder fed the exact product."""
    rng = np.random.default_rng(11)
    t = oracle.decode_table(oracle.E4M3)
    fin = np.sort(t[np.isfinite(t) & (t > 0)])
    mids = (fin[1:] + fin[:-1]) / 2
    found = 0
    for _ in range(200000):
        m = mids[rng.integers(0, len(mids))]
        s = np.float32(rng.uniform(0.5, 2.0))
        x = np.float32(m / float(s))
        p32 = np.float32(x * s)
        exact = float(x) * float(s)
        if float(p32) == m and exact != m:
            q = int(oracle.quantize(oracle.E4M3, np.array([x], np.float32), float(s))[0])
            lo = int(np.searchsorted(fin, m)) - 1 + 1  # code index of the value below m (codes start at 0x00=0)
            below, above = lo, lo + 1
            even = below if below % 2 == 0 else above
            nearest = above if exact > m else below
            assert q == even
            found += 1 if even != nearest else 0
            if found >= 20:
                break
    assert found >= 20


def test_amax_hand():
    x = np.array([0.5, -3.25, 2.0, -0.0, np.nan, 1.0], np.float32)
    assert oracle.amax(x) == np.float32(3.25)
    assert oracle.amax(np.zeros(7, np.float32)) == 0.0
    b = torch.tensor([[1.5, -7.0], [2.0, 6.5]], dtype=torch.bfloat16)
    assert oracle.amax(b.view(torch.int16).numpy().view(np.uint16)) == 7.0


def test_quantize_bf16_input_matches_fp32_input():
    """bf16 inputs are widened exactly to fp32 before the product."""
    g = torch.Generator().manual_seed(5)
    x = torch.randn(4096, generator=g).to(torch.bfloat16)
    bits = x.view(torch.int16).numpy().view(np.uint16)
    a = oracle.quantize(oracle.E4M3, bits, 37.5)
    b = oracle.quantize(oracle.E4M3, x.float().numpy(), 37.5)
    assert np.array_equal(a, b)


def test_colsum_small():
    x = np.array([[1, 2, -3], [4, -5, 6]], np.float32)
    s, a = oracle.colsum(x)
    assert np.array_equal(s, [5, -3, 3]) and np.array_equal(a, [5, 7, 9])


# --------------------------------------------------------------------------
# delayed scaling
# --------------------------------------------------------------------------
def test_scale_closed_form():
    for fmt, amax, margin, want in golden_lines("scale_closed_form.txt"):
        st = oracle.ScalingState([FMT[fmt]], hist_len=4, margin=int(margin))
        st.record_amax(0, np.float32(float(amax)))
        st.update(0)
        assert f32_hex(st.scale[0]) == int(want, 16), (fmt, amax, margin, st.scale[0])
        assert st.scale_inv[0] == np.float32(1.0) / st.scale[0]


def test_history_window_sequence():
    st = oracle.ScalingState([oracle.E4M3], hist_len=4)
    for step, amax, wmax, want in golden_lines("history_window.txt"):
        st.record_amax(0, np.float32(float(amax)))
        st.update(int(step))
        assert st.window_max()[0] == np.float32(float(wmax)), step
        assert f32_hex(st.scale[0]) == int(want, 16), step
        assert st.amax_cur[0] == 0.0


def test_interval_updates_scale_every_n_steps():
    st = oracle.ScalingState([oracle.E4M3], hist_len=8, interval=3)
    scales = []
    for step, a in enumerate([1.0, 2.0, 4.0, 8.0, 16.0, 32.0, 64.0]):
        st.record_amax(0, a)
        st.update(step)
        scales.append(float(st.scale[0]))
    # recomputed at steps 0, 3, 6 from the window max so far: 1, 8, 64
    assert scales == [448.0, 448.0, 448.0, 56.0, 56.0, 56.0, 7.0]
    assert list(st.hist[0, :7]) == [1, 2, 4, 8, 16, 32, 64]


def test_zero_and_nonfinite_amax_keep_scale():
    st = oracle.ScalingState([oracle.E4M3], hist_len=1)
    st.record_amax(0, 2.0)
    st.update(0)
    assert st.scale[0] == 224.0
    for bad in (0.0, np.inf):
        st.record_amax(0, bad)
        st.update(1)
        assert st.scale[0] == 224.0 and st.scale_inv[0] == np.float32(1 / 224)
    # an amax so small that FP8_MAX/amax overflows fp32 also keeps the scale
    st.record_amax(0, np.float32(1e-38))
    st.update(2)
    assert st.scale[0] == 224.0


def test_margin_is_power_of_two_divisor():
    for m in range(0, 8):
        st = oracle.ScalingState([oracle.E5M2], hist_len=2, margin=m)
        st.record_amax(0, 3.0)
        st.update(0)
        assert st.scale[0] == np.float32(np.float32(57344.0) / np.float32(3.0)) / np.float32(2.0 ** m)


def test_seed_fills_history():
    st = oracle.ScalingState([oracle.E4M3, oracle.E5M2], hist_len=16)
    st.record_amax(0, 3.0)
    st.record_amax(1, 0.25)
    st.seed()
    assert np.all(st.hist[0] == 3.0) and np.all(st.hist[1] == 0.25)
    assert f32_hex(st.scale[0]) == 0x43155555 and st.scale[1] == 57344.0 * 4
    assert np.all(st.amax_cur == 0)


def test_resume_from_checkpoint_is_bit_identical():
    rng = np.random.default_rng(0)
    amaxes = rng.uniform(0.01, 10, (30, 3)).astype(np.float32)

    def run(st, lo, hi):
        for t in range(lo, hi):
            for s in range(3):
                st.record_amax(s, amaxes[t, s])
            st.update(t)

    a = oracle.ScalingState([0, 0, 1], hist_len=5, margin=1, interval=2)
    run(a, 0, 30)
    b = oracle.ScalingState([0, 0, 1], hist_len=5, margin=1, interval=2)
    run(b, 0, 13)
    c = oracle.ScalingState([0, 0, 1], hist_len=5, margin=1, interval=2)
    for k in ("scale", "scale_inv", "amax_cur", "pos", "hist"):
        setattr(c, k, getattr(b, k).copy())
    run(c, 13, 30)
    for k in ("scale", "scale_inv", "hist", "pos"):
        assert np.array_equal(getattr(a, k), getattr(c, k))


# --------------------------------------------------------------------------
# GEMM
# --------------------------------------------------------------------------
def test_gemm_hand_example():
    g = {row[0]: row[1:] for row in golden_lines("gemm_hand.txt")}
    A = np.array([int(c, 16) for c in g["A"]], np.uint8).reshape(2, 2)
    B = np.array([int(c, 16) for c in g["B"]], np.uint8).reshape(2, 2)
    bias = np.array([float(v) for v in g["bias"]], np.float32)
    ms, ns = np.meshgrid(np.arange(2), np.arange(2), indexing="ij")
    ref, _ = oracle.gemm_elems(A, 0, B, 0, float(g["sa_inv"][0]), float(g["sb_inv"][0]), bias,
                               ms.ravel(), ns.ravel())
    assert list(ref) == [float(v) for v in g["D"]]


def _finite_codes(rng, fmt, shape):
    t = oracle.decode_table(fmt)
    ok = np.array([c for c in range(256) if np.isfinite(t[c])], np.uint8)
    return ok[rng.integers(0, ok.size, shape)]


@pytest.mark.parametrize("afmt,bfmt", [(0, 0), (1, 0), (0, 1), (1, 1)])
def test_gemm_matches_numpy_matmul(afmt, bfmt):
    rng = np.random.default_rng(afmt * 2 + bfmt)
    M, N, K = 48, 32, 80  # non-square, distinct dims: catches a transposed operand
    A = _finite_codes(rng, afmt, (M, K))
    B = _finite_codes(rng, bfmt, (N, K))
    sa, sb = np.float32(0.37), np.float32(1.9)
    bias = rng.standard_normal(N).astype(np.float32)
    ms, ns = np.meshgrid(np.arange(M), np.arange(N), indexing="ij")
    ref, absr = oracle.gemm_elems(A, afmt, B, bfmt, sa, sb, bias, ms.ravel(), ns.ravel())
    DA = oracle.decode_table(afmt)[A]
    DB = oracle.decode_table(bfmt)[B]
    s = float(np.float32(sa * sb))
    want = (DA @ DB.T) * s + bias.astype(np.float64)[None, :]
    want_abs = (np.abs(DA) @ np.abs(DB).T) * s
    np.testing.assert_allclose(ref.reshape(M, N), want, rtol=1e-13, atol=1e-9 * np.abs(want).max())
    np.testing.assert_allclose(absr.reshape(M, N), want_abs, rtol=1e-13)


def test_gemm_one_hot_picks_entries():
    M, N, K = 16, 16, 32
    rng = np.random.default_rng(2)
    A = _finite_codes(rng, 0, (M, K))
    B = np.zeros((N, K), np.uint8)
    for n in range(N):
        B[n, (3 * n + 1) % K] = 0x38  # 1.0
    ms, ns = np.meshgrid(np.arange(M), np.arange(N), indexing="ij")
    ref, _ = oracle.gemm_elems(A, 0, B, 0, 1.0, 1.0, None, ms.ravel(), ns.ravel())
    dec = oracle.decode_table(0)
    for m in range(M):
        for n in range(N):
            assert ref[m * N + n] == dec[A[m, (3 * n + 1) % K]]


# --------------------------------------------------------------------------
# MXFP8
# --------------------------------------------------------------------------
def test_e8m0_golden():
    for amax, e in golden_lines("e8m0_cases.txt"):
        assert oracle.e8m0_exponent(float(amax)) == int(e), amax


def test_e8m0_is_the_smallest_non_saturating_power_of_two():
    rng = np.random.default_rng(4)
    a = (rng.uniform(1, 2, 20000) * 2.0 ** rng.integers(-100, 100, 20000)).astype(np.float32)
    a = np.concatenate([a, np.float32(448) * np.float32(2.0) ** np.arange(-60, 60, dtype=np.float32)])
    for v in a:
        e = oracle.e8m0_exponent(v)
        if -127 < e < 127:
            assert math.ldexp(float(v), -e) <= 448.0 < math.ldexp(float(v), -(e - 1)), v


def test_mx_quantize_rows_block_properties():
    g = torch.Generator().manual_seed(9)
    x = (torch.randn(64, 256, generator=g) * torch.logspace(-3, 2, 256)[None, :]).to(torch.bfloat16)
    bits = x.view(torch.int16).numpy().view(np.uint16)
    q, s = oracle.mx_quantize_rows(bits)
    xf = x.float().numpy().astype(np.float64)
    dec = oracle.decode_table(0)[q]
    e = s.astype(np.int64) - 127
    recon = dec * np.repeat(2.0 ** e, 32, axis=1)
    blk_amax = np.abs(xf).reshape(64, 8, 32).max(-1)
    # the block maximum never saturates, and one exponent less would saturate it
    assert np.all(blk_amax * 2.0 ** -e <= 448)
    assert np.all((blk_amax == 0) | (blk_amax * 2.0 ** -(e - 1) > 448))
    # elementwise: nearest-code error at most half an E4M3 step of the scaled value
    scaled = xf * np.repeat(2.0 ** -e, 32, axis=1)
    tab = np.sort(oracle.decode_table(0)[np.isfinite(oracle.decode_table(0))])
    idx = np.clip(np.searchsorted(tab, scaled), 1, len(tab) - 1)
    gap = tab[idx] - tab[idx - 1]
    assert np.all(np.abs(dec - scaled) <= gap / 2 + 1e-30)
    assert np.all(np.isfinite(recon))


def test_mx_cols_is_rows_of_transpose():
    g = torch.Generator().manual_seed(10)
    x = torch.randn(64, 96, generator=g).to(torch.bfloat16)
    bits = x.view(torch.int16).numpy().view(np.uint16)
    qc, sc = oracle.mx_quantize_cols(bits)
    assert qc.shape == (96, 64) and sc.shape == (96, 2)
    # column c, block b covers rows 32b..32b+31 of x
    xf = x.float().numpy()
    for c in (0, 17, 95):
        for b in range(2):
            amax_b = np.abs(xf[32 * b:32 * b + 32, c]).max()
            assert int(sc[c, b]) - 127 == oracle.e8m0_exponent(amax_b)


def test_mx_gemm_matches_numpy_and_uniform_case():
    rng = np.random.default_rng(12)
    M, N, K = 32, 48, 128
    A = _finite_codes(rng, 0, (M, K))
    B = _finite_codes(rng, 0, (N, K))
    As = rng.integers(120, 135, (M, K // 32)).astype(np.uint8)
    Bs = rng.integers(120, 135, (N, K // 32)).astype(np.uint8)
    ms, ns = np.meshgrid(np.arange(M), np.arange(N), indexing="ij")
    ref, _ = oracle.mx_gemm_elems(A, As, B, Bs, None, ms.ravel(), ns.ravel())
    dec = oracle.decode_table(0)
    DA = dec[A] * np.repeat(2.0 ** (As.astype(np.int64) - 127), 32, axis=1)
    DB = dec[B] * np.repeat(2.0 ** (Bs.astype(np.int64) - 127), 32, axis=1)
    np.testing.assert_allclose(ref.reshape(M, N), DA @ DB.T, rtol=1e-12, atol=1e-12 * np.abs(DA @ DB.T).max())
    # uniform block scales reduce to the per-tensor GEMM with power-of-two scale_inv
    As1 = np.full_like(As, 130)
    Bs1 = np.full_like(Bs, 125)
    r1, _ = oracle.mx_gemm_elems(A, As1, B, Bs1, None, ms.ravel(), ns.ravel())
    r2, _ = oracle.gemm_elems(A, 0, B, 0, 8.0, 0.25, None, ms.ravel(), ns.ravel())
    np.testing.assert_allclose(r1, r2, rtol=1e-14, atol=1e-12)
