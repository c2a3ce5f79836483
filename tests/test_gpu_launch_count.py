"""fp8dl_kernel_launches counts the kernels each entry point enqueues: the figure
bench.py reports as gpu_launches comes from it."""
import pytest
import torch

import workloads as wl
from helpers import gpu

pytestmark = pytest.mark.gpu


def _count(fd, fn):
    n0 = fd.fp8dl_kernel_launches()
    fn()
    return fd.fp8dl_kernel_launches() - n0


def test_launch_counts_per_entry_point(monkeypatch):
    import fp8_delayed_scaling_gb300 as fd
    dev = gpu()
    monkeypatch.delenv("FP8DL_LN_VARIANT", raising=False)
    monkeypatch.delenv("FP8DL_LN_CLUSTERS", raising=False)
    g = wl.generator(90, "launches")
    R, C = 256, 4096
    x = wl.normal((R, C), 1.0, g, torch.bfloat16).to(dev)
    sc = torch.ones(1, device=dev)
    q = torch.empty((R, C), dtype=torch.uint8, device=dev)
    qt = torch.empty((C, R), dtype=torch.uint8, device=dev)
    am = torch.zeros(1, device=dev)
    db = torch.empty(C, device=dev)
    sinv = torch.empty(1, device=dev)
    ws = torch.empty(fd.fp8_cast_workspace_size(R, C), dtype=torch.uint8, device=dev)
    assert _count(fd, lambda: fd.fp8_cast_amax_transpose(x, fd.E4M3, sc, out=q, out_t=qt, amax=am)) == 1
    assert _count(fd, lambda: fd.fp8_cast_amax_transpose(x, fd.E4M3, sc, out=q, amax=am, dbias=db, workspace=ws,
                                                         scale_inv_out=sinv)) == 3  # cast, column sums, 1/scale
    w2 = torch.empty((C, R), dtype=torch.bfloat16, device=dev).fill_(0.5)
    q2 = torch.empty((C, R), dtype=torch.uint8, device=dev)
    grouped = [dict(x=x, scale=sc, out=q, out_t=qt, amax=am), dict(x=w2, scale=sc, out=q2, amax=am)]
    assert _count(fd, lambda: fd.fp8_cast_amax_transpose_multi(grouped, fd.E4M3)) == 1  # one grid for both
    grouped[1]["scale_inv_out"] = sinv
    assert _count(fd, lambda: fd.fp8_cast_amax_transpose_multi(grouped, fd.E4M3)) == 2  # + the decode factors
    gam = torch.ones(C, dtype=torch.bfloat16, device=dev)
    bet = torch.zeros(C, dtype=torch.bfloat16, device=dev)
    mu = torch.empty(R, device=dev)
    rs = torch.empty(R, device=dev)
    ln = lambda: fd.fp8_layernorm_cast(x, gam, bet, 1e-5, fd.E4M3, sc, mu, rs, out=q, out_t=qt, amax=am)  # noqa: E731
    assert _count(fd, ln) == 1  # 4096 columns: one cluster kernel
    dx = torch.empty_like(x)
    dg = torch.empty(C, device=dev)
    lw = torch.empty(fd.fp8_layernorm_bwd_workspace_size(R, C), dtype=torch.uint8, device=dev)
    lnb = lambda: fd.fp8_layernorm_bwd(x, x, gam, mu, rs, dx, dg, db, lw)  # noqa: E731
    assert _count(fd, lnb) == 2  # cluster kernel + column-partial reduction
    monkeypatch.setenv("FP8DL_LN_VARIANT", "tiles")
    assert _count(fd, ln) == 2  # statistics pass + tiled pass
    assert _count(fd, lnb) == 3  # row sums, tiles, reduction
    monkeypatch.delenv("FP8DL_LN_VARIANT")
    one = torch.ones(1, device=dev)
    D = torch.empty((R, R), dtype=torch.bfloat16, device=dev)
    assert _count(fd, lambda: fd.fp8_gemm(q, fd.E4M3, q[:R], fd.E4M3, one, one, D)) == 1
    torch.cuda.synchronize()
