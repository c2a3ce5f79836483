"""GPU parity of the scale update and the fused cast + amax + transpose
(+ bias gradient) against the oracle: bit-exact codes, amax and scales."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from helpers import gpu, host

pytestmark = pytest.mark.gpu


def _fd():
    import fp8_delayed_scaling_gb300 as fd
    return fd


def _run_cast(x, fmt, scale_val, transpose=True, dbias=False):
    fd = _fd()
    dev = x.device
    rows, cols = x.shape
    scale = torch.tensor([scale_val], dtype=torch.float32, device=dev)
    amax = torch.zeros(1, dtype=torch.float32, device=dev)
    out = torch.full((rows, cols), 0xAA, dtype=torch.uint8, device=dev)
    out_t = torch.full((cols, rows), 0xAA, dtype=torch.uint8, device=dev) if transpose else None
    db = torch.full((cols,), float("nan"), dtype=torch.float32, device=dev) if dbias else None
    ws = torch.empty(fd.fp8_cast_workspace_size(rows, cols), dtype=torch.uint8, device=dev) if dbias else None
    fd.fp8_cast_amax_transpose(x, fmt, scale, out=out, out_t=out_t, amax=amax, dbias=db, workspace=ws)
    torch.cuda.synchronize()
    return out, out_t, amax, db


SHAPES = [(16, 16), (48, 80), (128, 128), (144, 272), (256, 48), (2048, 768), (400, 1040)]


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("kind,fmt", [(torch.float32, 0), (torch.bfloat16, 0), (torch.bfloat16, 1),
                                      (torch.float32, 1)])
def test_cast_parity(shape, kind, fmt):
    dev = gpu()
    g = wl.generator(31, "cast/%s/%s/%d" % (shape, kind, fmt))
    x = wl.normal(shape, 1.0 if fmt == 0 else 1e-3, g, kind)
    if fmt == 1:
        x = wl.with_outliers(x, 0.001, 1000.0, g)
    xs = host(x)
    a = oracle.amax(xs)
    scale = np.float32(oracle.fp8_max(fmt)) / a / np.float32(2.0)  # some non-trivial fp32 scale
    out, out_t, amax, db = _run_cast(x.to(dev), fmt, float(scale), dbias=True)
    q = oracle.quantize(fmt, xs, float(scale))
    assert np.array_equal(out.cpu().numpy(), q)
    assert np.array_equal(out_t.cpu().numpy(), q.T)
    assert amax.item() == a
    s, sabs = oracle.colsum(xs)
    rows = shape[0]
    bound = rows * 2.0 ** -24 * sabs + 1e-30
    assert np.all(np.abs(db.cpu().numpy().astype(np.float64) - s) <= bound)


# Column sums for dbias: the running-sum variant with its grid cut to a multiple of the
# column-tile count (2048 x 6144: 48 column tiles, 768 tiles over 608 resident CTAs), and the
# per-tile variant, which only a row wider than the resident grid (640 column tiles) takes.
@pytest.mark.parametrize("shape", [(2048, 6144), (16, 81920)])
def test_cast_dbias_paths(shape):
    dev = gpu()
    g = wl.generator(33, "cast-dbias/%s" % (shape,))
    x = wl.with_outliers(wl.normal(shape, 1e-3, g, torch.bfloat16), 0.001, 1000.0, g)
    xs = host(x)
    scale = np.float32(oracle.fp8_max(1)) / oracle.amax(xs) / np.float32(2.0)
    out, out_t, amax, db = _run_cast(x.to(dev), 1, float(scale), dbias=True)
    q = oracle.quantize(1, xs, float(scale))
    assert np.array_equal(out.cpu().numpy(), q)
    assert np.array_equal(out_t.cpu().numpy(), q.T)
    assert amax.item() == oracle.amax(xs)
    s, sabs = oracle.colsum(xs)
    bound = shape[0] * 2.0 ** -24 * sabs + 1e-30
    assert np.all(np.abs(db.cpu().numpy().astype(np.float64) - s) <= bound)


@pytest.mark.parametrize("kind,fmt", [(torch.bfloat16, 0), (torch.float32, 1)])
def test_grouped_cast_parity(kind, fmt):
    """fp8_cast_amax_transpose_multi: several tensors of different (ragged) shapes and scales in
    one launch; each tensor's codes, transposed codes, amax and decode factor bit-exact against
    the oracle, and the outputs one item leaves out untouched."""
    fd = _fd()
    dev = gpu()
    shapes = [(2048, 768), (16, 16), (400, 1040), (144, 272), (4096, 4096), (48, 80)]
    items, ref = [], []
    for k, shape in enumerate(shapes):
        g = wl.generator(35, "multi/%d/%s/%d" % (k, kind, fmt))
        x = wl.normal(shape, 10.0 ** (k - 3), g, kind)
        xs = host(x)
        scale_val = float(np.float32(oracle.fp8_max(fmt)) / oracle.amax(xs) / np.float32(1 + k))
        rows, cols = shape
        it = dict(x=x.to(dev), scale=torch.tensor([scale_val], dtype=torch.float32, device=dev),
                  out=torch.full((rows, cols), 0xAA, dtype=torch.uint8, device=dev),
                  out_t=torch.full((cols, rows), 0xAA, dtype=torch.uint8, device=dev) if k != 1 else None,
                  amax=torch.zeros(1, dtype=torch.float32, device=dev) if k != 3 else None,
                  scale_inv_out=torch.full((1,), float("nan"), dtype=torch.float32, device=dev) if k % 2 else None)
        items.append(it)
        ref.append((xs, scale_val))
    fd.fp8_cast_amax_transpose_multi(items, fmt)
    torch.cuda.synchronize()
    for it, (xs, scale_val) in zip(items, ref):
        q = oracle.quantize(fmt, xs, scale_val)
        assert np.array_equal(it["out"].cpu().numpy(), q)
        if it["out_t"] is not None:
            assert np.array_equal(it["out_t"].cpu().numpy(), q.T)
        if it["amax"] is not None:
            assert it["amax"].item() == oracle.amax(xs)
        if it["scale_inv_out"] is not None:
            assert it["scale_inv_out"].item() == float(np.float32(1.0) / np.float32(scale_val))


def test_grouped_cast_matches_single_casts():
    """The grouped cast of two weights gives the bits of two separate casts (the LayerNormMLP
    forward uses it for W1 and W2)."""
    fd = _fd()
    dev = gpu()
    g = wl.generator(36, "multi-vs-single")
    ws = [wl.normal((1024, 512), 0.02, g, torch.bfloat16).to(dev), wl.normal((512, 1024), 0.02, g, torch.bfloat16).to(dev)]
    sc = [torch.tensor([4096.0], device=dev), torch.tensor([8192.0], device=dev)]
    res = []
    for grouped in (False, True):
        outs = [(torch.empty_like(w, dtype=torch.uint8), torch.empty(w.shape[::-1], dtype=torch.uint8, device=dev),
                 torch.zeros(1, device=dev), torch.empty(1, device=dev)) for w in ws]
        if grouped:
            fd.fp8_cast_amax_transpose_multi([dict(x=w, scale=s, out=o[0], out_t=o[1], amax=o[2], scale_inv_out=o[3])
                                              for w, s, o in zip(ws, sc, outs)], fd.E4M3)
        else:
            for w, s, o in zip(ws, sc, outs):
                fd.fp8_cast_amax_transpose(w, fd.E4M3, s, out=o[0], out_t=o[1], amax=o[2], scale_inv_out=o[3])
        torch.cuda.synchronize()
        res.append(outs)
    for a, b in zip(*res):
        for ta, tb in zip(a, b):
            assert torch.equal(ta, tb)


def test_cast_special_values():
    """NaN, infinities, overflow, fp32 subnormals and signed zeros through the hardware cvt."""
    dev = gpu()
    vals = np.array([0.0, -0.0, 1e-45, -1e-45, 1e-40, 2.0 ** -10, -2.0 ** -10, 447.9, 448.0, 464.0, 480.0, 1e30,
                     np.inf, -np.inf, np.nan, 57343.0, 57344.0, 61439.0, 61440.0, 1e38, 3.0e-5, 1.5e-5, -7.7e-6],
                    np.float32)
    x = np.resize(vals, 32 * 32).astype(np.float32).reshape(32, 32)
    for fmt in (0, 1):
        out, out_t, amax, _ = _run_cast(torch.from_numpy(x).to(dev), fmt, 1.0)
        q = oracle.quantize(fmt, x, 1.0)
        got = out.cpu().numpy()
        tab = oracle.decode_table(fmt)
        nan = np.isnan(x)
        assert np.all(np.isnan(tab[got[nan]]))
        assert np.array_equal(got[~nan], q[~nan]), (fmt, x[~nan][got[~nan] != q[~nan]])
        assert amax.item() == oracle.amax(x)  # inf


def _sweep_chunk(fmt, start, count, dev):
    fd = _fd()
    bits = torch.arange(start, start + count, dtype=torch.int64, device=dev).to(torch.int32)
    x = bits.view(torch.float32).reshape(count // 16384, 16384)
    scale = torch.ones(1, dtype=torch.float32, device=dev)
    out = torch.empty_like(x, dtype=torch.uint8)
    fd.fp8_cast_amax_transpose(x, fmt, scale, out=out)
    return out.reshape(-1).cpu().numpy()


@pytest.mark.parametrize("fmt", [0, 1])
def test_encoder_all_fp32_inputs(fmt):
    """Every one of the 2^32 fp32 bit patterns, scale 1: GPU codes == oracle codes
    (NaN inputs: any NaN code)."""
    dev = gpu()
    chunk = 1 << 27
    tab = oracle.decode_table(fmt)
    for start in range(0, 1 << 32, chunk):
        got = _sweep_chunk(fmt, start, chunk, dev)
        v = np.arange(start, start + chunk, dtype=np.uint64).astype(np.uint32).view(np.float32)
        want = oracle.encode(fmt, v)
        nan = np.isnan(v)
        if nan.any():
            assert np.all(np.isnan(tab[got[nan]]))
            got, want = got[~nan], want[~nan]
        bad = np.nonzero(got != want)[0]
        assert bad.size == 0, (hex(start), bad[:5], got[bad[:5]], want[bad[:5]])


def test_amax_only_pass_and_accumulation():
    fd = _fd()
    dev = gpu()
    g = wl.generator(5, "amax-only")
    x1 = wl.normal((512, 256), 2.0, g, torch.bfloat16)
    x2 = wl.normal((512, 256), 0.5, g, torch.bfloat16)
    amax = torch.zeros(1, dtype=torch.float32, device=dev)
    fd.fp8_cast_amax_transpose(x2.to(dev), 0, None, amax=amax)
    fd.fp8_cast_amax_transpose(x1.to(dev), 0, None, amax=amax)
    torch.cuda.synchronize()
    assert amax.item() == max(oracle.amax(host(x1)), oracle.amax(host(x2)))


def test_update_scale_parity_random_sequences():
    """fp8_update_scale vs the oracle over 40 steps: scale, scale_inv, history and
    position bit-exact, for several recipes and HYBRID slot formats."""
    fd = _fd()
    dev = gpu()
    rng = np.random.default_rng(17)
    for L, margin, interval in [(16, 0, 1), (4, 2, 3), (1024, 0, 1), (1, 5, 2), (7, 0, 4)]:
        recipe = fd.Recipe(margin=margin, interval=interval, fp8_format=fd.FORMAT_HYBRID, amax_history_len=L)
        fmts = [0, 0, 1, 0, 0, 1]
        st = fd.ScalingState(recipe, fmts, device=dev)
        ost = oracle.ScalingState(fmts, hist_len=L, margin=margin, interval=interval)
        view = st.buf.view(torch.float32).view(len(fmts), st.stride // 4)
        for step in range(40):
            a = (rng.uniform(0, 3, len(fmts)) * 10.0 ** rng.integers(-6, 4, len(fmts))).astype(np.float32)
            if step % 11 == 5:
                a[1] = 0.0
            if step % 13 == 7:
                a[4] = np.inf
            view[:, 2] = torch.from_numpy(a).to(dev)
            for i in range(len(fmts)):
                ost.record_amax(i, a[i])
            if step == 0:
                st.seed()
                ost.seed()
            else:
                st.update(step)
                ost.update(step)
            got = st.read()
            assert np.array_equal(got["scale"], ost.scale), (L, step)
            assert np.array_equal(got["scale_inv"], ost.scale_inv), (L, step)
            assert np.array_equal(got["hist"], ost.hist), (L, step)
            assert np.array_equal(got["pos"], ost.pos), (L, step)
            assert np.all(got["amax"] == 0)


@pytest.mark.parametrize("margin", [0, 7, 126])
def test_update_scale_degenerate_amaxes(margin):
    """Amaxes at the edges of fp32 against the oracle, bit for bit: subnormal and tiny
    amaxes (FP8_MAX/amax overflows: the scale is kept), a huge amax with a large margin (the
    scale underflows: kept), an amax whose scale_inv is subnormal, NaN (ignored by the window
    max) and infinity (kept)."""
    fd = _fd()
    dev = gpu()
    seq = [1.0, 1e-45, 1e-38, 3.0e38, 2e-36, float("nan"), 7.5, float("inf"), 0.0, 1e-37, 5e-3, 2.0 ** -126]
    for L in (1, 3):
        recipe = fd.Recipe(margin=margin, interval=1, fp8_format=fd.FORMAT_HYBRID, amax_history_len=L)
        fmts = [0, 1]
        st = fd.ScalingState(recipe, fmts, device=dev)
        ost = oracle.ScalingState(fmts, hist_len=L, margin=margin, interval=1)
        view = st.buf.view(torch.float32).view(len(fmts), st.stride // 4)
        for step, a0 in enumerate(seq):
            a = np.array([a0, a0], np.float32)
            # the amax fields are written directly on both sides (a cast's max would drop a NaN)
            view[:, 2] = torch.from_numpy(a).to(dev)
            ost.amax_cur[:] = a
            if step == 0:
                st.seed()
                ost.seed()
            else:
                st.update(step)
                ost.update(step)
            got = st.read()
            assert np.array_equal(got["scale"], ost.scale), (margin, L, step)
            assert np.array_equal(got["scale_inv"], ost.scale_inv), (margin, L, step)
            assert np.array_equal(got["hist"], ost.hist, equal_nan=True), (margin, L, step)
