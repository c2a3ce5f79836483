"""The allocation-free cast entry point (fp8_cast_amax_transpose_noalloc).

Some callers cannot allocate device memory: a plugin or custom-op interface
whose fixed signature passes only inputs and outputs, or a process whose
device memory belongs to another allocator.  They cannot pass the bias-gradient
workspace either, so this entry point keeps that scratch in a static device
array of the library.  These tests call it through the C ABI and compare it
with the workspace-taking entry point on the same inputs, twice in a row (the
second call must not see the first call's leftovers), and check that sizes
beyond the static array are refused before any launch.

Kept in a file that pytest collects last, so that a run stopping at the first
failure has already run every other test.
"""
import numpy as np
import pytest
import torch

import workloads as wl
from helpers import gpu

pytestmark = pytest.mark.gpu


def _both(fd, x, fmt, scale_val):
    dev = x.device
    rows, cols = x.shape
    scale = torch.tensor([scale_val], dtype=torch.float32, device=dev)
    res = []
    for noalloc in (False, True):
        amax = torch.zeros(1, dtype=torch.float32, device=dev)
        out = torch.full((rows, cols), 0xAA, dtype=torch.uint8, device=dev)
        out_t = torch.full((cols, rows), 0xAA, dtype=torch.uint8, device=dev)
        db = torch.full((cols,), float("nan"), dtype=torch.float32, device=dev)
        if noalloc:
            fd.fp8_cast_amax_transpose_noalloc(x, fmt, scale, out=out, out_t=out_t, amax=amax, dbias=db)
        else:
            ws = torch.empty(fd.fp8_cast_workspace_size(rows, cols), dtype=torch.uint8, device=dev)
            fd.fp8_cast_amax_transpose(x, fmt, scale, out=out, out_t=out_t, amax=amax, dbias=db, workspace=ws)
        torch.cuda.synchronize()
        res.append((out.cpu(), out_t.cpu(), amax.item(), db.cpu().numpy().astype(np.float64)))
    return res


def test_noalloc_matches_workspace_entry_point_on_two_calls():
    import fp8_delayed_scaling_gb300 as fd
    dev = gpu()
    g = wl.generator(77, "noalloc")
    cases = [  # (input, format, scale); the second call is smaller, so stale scratch from the first remains
        (wl.with_outliers(wl.normal((2048, 3072), 1e-3, g, torch.bfloat16), 0.001, 1000.0, g), fd.E5M2, 4096.0),
        (wl.normal((400, 784), 1.0, g, torch.float32), fd.E4M3, 97.25),
    ]
    for x, fmt, scale in cases:
        xd = x.to(dev)
        (o1, t1, a1, d1), (o2, t2, a2, d2) = _both(fd, xd, fmt, scale)
        assert torch.equal(o1, o2) and torch.equal(t1, t2)
        assert a1 == a2
        xs = x.float().numpy().astype(np.float64)
        bound = x.shape[0] * 2.0 ** -24 * np.abs(xs).sum(0) + 1e-30  # dbias tolerance of the cast tests
        assert np.all(np.abs(d2 - d1) <= bound)
        assert np.all(np.abs(d2 - xs.sum(0)) <= bound)


def test_noalloc_refuses_sizes_beyond_the_static_array():
    import fp8_delayed_scaling_gb300 as fd
    gpu()
    L = fd._lib
    a16 = 1 << 20  # never dereferenced: the size check fails before any launch
    # ceil(8192/128) * 32768 * 4 = 8 MiB > 4 MiB
    st = L.fp8_cast_amax_transpose_noalloc(a16, fd.BF16, 8192, 32768, fd.E4M3, a16, a16, None, None, a16, None)
    assert st == fd.ERR_WORKSPACE
    assert "static" in fd.fp8dl_last_error()
    # the largest size that fits: ceil(8192/128) * 16384 * 4 = 4 MiB exactly is accepted by the check
    assert fd.fp8_cast_workspace_size(8192, 16384) == 4 << 20


def test_noalloc_at_the_full_static_array():
    """A bias gradient whose scratch fills the 4 MiB array exactly (8192 x 16384 bf16:
    64 row tiles x 16384 columns x 4 bytes) matches the workspace entry point, twice in a
    row; one size step larger in either dimension is refused before any launch."""
    import fp8_delayed_scaling_gb300 as fd
    dev = gpu()
    rows, cols = 8192, 16384
    assert fd.fp8_cast_workspace_size(rows, cols) == 4 << 20
    g = wl.generator(78, "noalloc-full")
    x = wl.normal((rows, cols), 1e-2, g, torch.bfloat16).to(dev)
    scale = torch.tensor([2048.0], dtype=torch.float32, device=dev)
    ws = torch.empty(fd.fp8_cast_workspace_size(rows, cols), dtype=torch.uint8, device=dev)
    ref = [torch.empty((rows, cols), dtype=torch.uint8, device=dev), torch.empty((cols, rows), dtype=torch.uint8,
           device=dev), torch.zeros(1, dtype=torch.float32, device=dev), torch.empty(cols, dtype=torch.float32,
                                                                                       device=dev)]
    fd.fp8_cast_amax_transpose(x, fd.E4M3, scale, out=ref[0], out_t=ref[1], amax=ref[2], dbias=ref[3], workspace=ws)
    xs = x.float().cpu().numpy().astype(np.float64)
    bound = rows * 2.0 ** -24 * np.abs(xs).sum(0) + 1e-30
    for _ in range(2):
        out = torch.full((rows, cols), 0xAA, dtype=torch.uint8, device=dev)
        out_t = torch.full((cols, rows), 0xAA, dtype=torch.uint8, device=dev)
        amax = torch.zeros(1, dtype=torch.float32, device=dev)
        db = torch.full((cols,), float("nan"), dtype=torch.float32, device=dev)
        fd.fp8_cast_amax_transpose_noalloc(x, fd.E4M3, scale, out=out, out_t=out_t, amax=amax, dbias=db)
        torch.cuda.synchronize()
        assert torch.equal(out, ref[0]) and torch.equal(out_t, ref[1]) and torch.equal(amax, ref[2])
        d1, d2 = ref[3].cpu().numpy().astype(np.float64), db.cpu().numpy().astype(np.float64)
        assert np.all(np.abs(d2 - d1) <= bound) and np.all(np.abs(d2 - xs.sum(0)) <= bound)
    # one step of 16 beyond the array in rows (65 row tiles) or in columns: refused, outputs untouched
    for r, c in ((rows + 16, cols), (rows, cols + 16)):
        assert fd.fp8_cast_workspace_size(r, c) > 4 << 20
        xb = torch.zeros((r, c), dtype=torch.bfloat16, device=dev)
        db = torch.full((c,), 7.0, dtype=torch.float32, device=dev)
        with pytest.raises(fd.FP8DLError) as e:
            fd.fp8_cast_amax_transpose_noalloc(xb, fd.E4M3, scale, dbias=db)
        assert e.value.status == fd.ERR_WORKSPACE
        torch.cuda.synchronize()
        assert torch.all(db == 7.0)
