"""GPU parity of the LayerNormMLP kernels against the oracle.

The activations are transcendental (erf, exp, rsqrt), so their bf16 values are
compared within a stated bound; the FP8 codes and amaxes that follow are
bit-exact, computed by the oracle from the GPU's own bf16 activation tensor
(both sides then take the same integer decision from the same input)."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from helpers import as_f64, gpu, host

pytestmark = pytest.mark.gpu


def _fd():
    import fp8_delayed_scaling_gb300 as fd
    return fd


# FP8DL_LN_VARIANT / FP8DL_LN_CLUSTERS select the implementation: widths that are a
# multiple of 512 (up to 8192) take the cluster path, the rest the tile path.
VARIANTS = {"default": {}, "tiles": {"FP8DL_LN_VARIANT": "tiles"}, "two-clusters": {"FP8DL_LN_CLUSTERS": "2"}}


def _variant(monkeypatch, name):
    for k in ("FP8DL_LN_VARIANT", "FP8DL_LN_CLUSTERS"):
        monkeypatch.delenv(k, raising=False)
    for k, v in VARIANTS[name].items():
        monkeypatch.setenv(k, v)


@pytest.mark.parametrize("shape", [(16, 64), (48, 768), (256, 4096), (32, 8192), (160, 1040), (64, 2000 // 16 * 16)])
def test_layernorm_cast_parity(shape):
    _layernorm_cast_check(shape, 0)


# cluster sizes 1, 3, 8, 16; a 16-row tail block; two clusters walking many blocks
@pytest.mark.parametrize("variant", list(VARIANTS))
@pytest.mark.parametrize("shape,fmt", [((16, 512), 0), ((208, 1536), 1), ((1040, 4096), 0), ((48, 8192), 1)])
def test_layernorm_cast_variants(shape, fmt, variant, monkeypatch):
    _variant(monkeypatch, variant)
    _layernorm_cast_check(shape, fmt)


def _layernorm_cast_check(shape, fmt):
    fd = _fd()
    dev = gpu()
    R, C = shape
    g = wl.generator(51, "ln/%s" % (shape,))
    x = (wl.normal((R, C), 1.0, g) * 2.0 + 0.5).to(torch.bfloat16)
    gamma = (1.0 + wl.normal((C,), 0.1, g)).to(torch.bfloat16)
    beta = wl.normal((C,), 0.1, g, torch.bfloat16)
    scale = 37.0
    xd, gd, bd = x.to(dev), gamma.to(dev), beta.to(dev)
    q = torch.full((R, C), 0xAA, dtype=torch.uint8, device=dev)
    qt = torch.full((C, R), 0xAA, dtype=torch.uint8, device=dev)
    amax = torch.zeros(1, dtype=torch.float32, device=dev)
    mu = torch.empty(R, dtype=torch.float32, device=dev)
    rs = torch.empty(R, dtype=torch.float32, device=dev)
    y = torch.empty((R, C), dtype=torch.bfloat16, device=dev)
    sc = torch.tensor([scale], dtype=torch.float32, device=dev)
    fd.fp8_layernorm_cast(xd, gd, bd, 1e-5, fmt, sc, mu, rs, out=q, out_t=qt, amax=amax, y=y)
    torch.cuda.synchronize()
    yr, mur, rsr = oracle.layernorm_fwd(host(x), host(gamma), host(beta), 1e-5)
    yg = as_f64(y)
    assert np.all(np.abs(yg - yr) <= 2.0 ** -7 * np.abs(yr) + 2.0 ** -14)
    assert np.all(np.abs(mu.cpu().numpy() - mur) <= 2.0 ** -20 * np.abs(host_f(x)).max())
    assert np.all(np.abs(rs.cpu().numpy() - rsr) <= 2.0 ** -18 * rsr)
    yb = host(y)
    qo = oracle.quantize(fmt, yb, scale)
    assert np.array_equal(q.cpu().numpy(), qo)
    assert np.array_equal(qt.cpu().numpy(), qo.T)
    assert amax.item() == oracle.amax(yb)


def host_f(t):
    return t.float().numpy()


@pytest.mark.parametrize("variant", ["default", "tiles"])
def test_layernorm_cast_offset_rows(variant, monkeypatch):
    """Rows whose mean is far from zero (64 +- 0.5): the statistics are merged from two-pass
    partials, so no cancellation of sum(x^2) - n mean^2 spoils rsigma."""
    _variant(monkeypatch, variant)
    fd = _fd()
    dev = gpu()
    R, C = 256, 4096
    g = wl.generator(55, "ln-offset")
    x = (wl.normal((R, C), 0.5, g) + 64.0).to(torch.bfloat16)
    gamma = torch.ones(C, dtype=torch.bfloat16)
    beta = torch.zeros(C, dtype=torch.bfloat16)
    mu = torch.empty(R, dtype=torch.float32, device=dev)
    rs = torch.empty(R, dtype=torch.float32, device=dev)
    q = torch.empty((R, C), dtype=torch.uint8, device=dev)
    sc = torch.tensor([16.0], dtype=torch.float32, device=dev)
    fd.fp8_layernorm_cast(x.to(dev), gamma.to(dev), beta.to(dev), 1e-5, 0, sc, mu, rs, out=q)
    torch.cuda.synchronize()
    _, mur, rsr = oracle.layernorm_fwd(host(x), host(gamma), host(beta), 1e-5)
    assert np.all(np.abs(mu.cpu().numpy() - mur) <= 2.0 ** -20 * np.abs(host_f(x)).max())
    assert np.all(np.abs(rs.cpu().numpy() - rsr) <= 2.0 ** -18 * rsr)


def test_layernorm_cast_without_outputs_records_amax_and_stats():
    fd = _fd()
    dev = gpu()
    R, C = 64, 1024
    g = wl.generator(52, "ln-amax")
    x = wl.normal((R, C), 1.0, g, torch.bfloat16).to(dev)
    gamma = torch.ones(C, dtype=torch.bfloat16, device=dev)
    beta = torch.zeros(C, dtype=torch.bfloat16, device=dev)
    amax = torch.zeros(1, dtype=torch.float32, device=dev)
    mu = torch.empty(R, dtype=torch.float32, device=dev)
    rs = torch.empty(R, dtype=torch.float32, device=dev)
    y = torch.empty((R, C), dtype=torch.bfloat16, device=dev)
    fd.fp8_layernorm_cast(x, gamma, beta, 1e-5, fd.E4M3, None, mu, rs, amax=amax, y=y)
    torch.cuda.synchronize()
    assert amax.item() == oracle.amax(host(y))


@pytest.mark.parametrize("shape", [(128, 128), (48, 80), (256, 1040)])
@pytest.mark.parametrize("fmt", [0, 1])
def test_gelu_cast_parity(shape, fmt):
    fd = _fd()
    dev = gpu()
    R, C = shape
    h = wl.normal(shape, 3.0, wl.generator(53, "gelu/%s" % (shape,)), torch.bfloat16)
    sc = torch.tensor([11.5], dtype=torch.float32, device=dev)
    q = torch.full((R, C), 0xAA, dtype=torch.uint8, device=dev)
    qt = torch.full((C, R), 0xAA, dtype=torch.uint8, device=dev)
    amax = torch.zeros(1, dtype=torch.float32, device=dev)
    gout = torch.empty((R, C), dtype=torch.bfloat16, device=dev)
    fd.fp8_gelu_cast(h.to(dev), fmt, sc, out=q, out_t=qt, amax=amax, g=gout)
    torch.cuda.synchronize()
    ref = oracle.gelu(host(h))
    got = as_f64(gout)
    hf = np.abs(host_f(h).astype(np.float64))
    assert np.all(np.abs(got - ref) <= 2.0 ** -7 * np.abs(ref) + 2.0 ** -21 * hf)
    gb = host(gout)
    qo = oracle.quantize(fmt, gb, 11.5)
    assert np.array_equal(q.cpu().numpy(), qo)
    assert np.array_equal(qt.cpu().numpy(), qo.T)
    assert amax.item() == oracle.amax(gb)


@pytest.mark.parametrize("shape", [(128, 128), (48, 80), (384, 1040)])
def test_dgelu_cast_parity(shape):
    fd = _fd()
    dev = gpu()
    R, C = shape
    g = wl.generator(54, "dgelu/%s" % (shape,))
    h = wl.normal(shape, 3.0, g, torch.bfloat16)
    dg = wl.normal(shape, 1e-3, g, torch.bfloat16)
    sc = torch.tensor([2.0 ** 14], dtype=torch.float32, device=dev)
    q = torch.full((R, C), 0xAA, dtype=torch.uint8, device=dev)
    qt = torch.full((C, R), 0xAA, dtype=torch.uint8, device=dev)
    amax = torch.zeros(1, dtype=torch.float32, device=dev)
    dh = torch.empty((R, C), dtype=torch.bfloat16, device=dev)
    db = torch.empty(C, dtype=torch.float32, device=dev)
    ws = torch.empty(fd.fp8_cast_workspace_size(R, C), dtype=torch.uint8, device=dev)
    fd.fp8_dgelu_cast(dg.to(dev), h.to(dev), fd.E5M2, sc, out=q, out_t=qt, amax=amax, dbias=db, workspace=ws, dh=dh)
    torch.cuda.synchronize()
    ref = oracle.dgelu(host(dg), host(h))
    got = as_f64(dh)
    assert np.all(np.abs(got - ref) <= 2.0 ** -7 * np.abs(ref) + 2.0 ** -21 * np.abs(host_f(dg).astype(np.float64)))
    dhb = host(dh)
    qo = oracle.quantize(fd.E5M2, dhb, 2.0 ** 14)
    assert np.array_equal(q.cpu().numpy(), qo)
    assert np.array_equal(qt.cpu().numpy(), qo.T)
    assert amax.item() == oracle.amax(dhb)
    s, sabs = oracle.colsum(dhb)
    assert np.all(np.abs(db.cpu().numpy().astype(np.float64) - s) <= R * 2.0 ** -24 * sabs + 1e-30)


@pytest.mark.parametrize("shape", [(16, 64), (48, 768), (256, 4096), (144, 1040)])
def test_layernorm_bwd_parity(shape):
    _layernorm_bwd_check(shape)


@pytest.mark.parametrize("variant", list(VARIANTS))
@pytest.mark.parametrize("shape", [(16, 512), (208, 1536), (1040, 4096), (48, 8192)])
def test_layernorm_bwd_variants(shape, variant, monkeypatch):
    _variant(monkeypatch, variant)
    _layernorm_bwd_check(shape)


def _layernorm_bwd_check(shape):
    fd = _fd()
    dev = gpu()
    R, C = shape
    g = wl.generator(55, "lnb/%s" % (shape,))
    x = (wl.normal((R, C), 1.0, g) * 1.5 - 0.25).to(torch.bfloat16)
    gamma = (1.0 + wl.normal((C,), 0.1, g)).to(torch.bfloat16)
    beta = torch.zeros(C, dtype=torch.bfloat16)
    dy = wl.normal((R, C), 1e-3, g, torch.bfloat16)
    xd, gd = x.to(dev), gamma.to(dev)
    mu = torch.empty(R, dtype=torch.float32, device=dev)
    rs = torch.empty(R, dtype=torch.float32, device=dev)
    fd.fp8_layernorm_cast(xd, gd, beta.to(dev), 1e-5, fd.E4M3, None, mu, rs,
                          amax=torch.zeros(1, dtype=torch.float32, device=dev))
    dx = torch.empty((R, C), dtype=torch.bfloat16, device=dev)
    dgam = torch.empty(C, dtype=torch.float32, device=dev)
    dbet = torch.empty(C, dtype=torch.float32, device=dev)
    ws = torch.empty(fd.fp8_layernorm_bwd_workspace_size(R, C), dtype=torch.uint8, device=dev)
    fd.fp8_layernorm_bwd(dy.to(dev), xd, gd, mu, rs, dx, dgam, dbet, ws)
    torch.cuda.synchronize()
    # the oracle takes the GPU's saved statistics as inputs (the backward's own inputs)
    rdx, rdg, rdb, adx, adg, adb = oracle.layernorm_bwd(host(dy), host(x), host(gamma),
                                                        mu.cpu().numpy().astype(np.float64),
                                                        rs.cpu().numpy().astype(np.float64))
    assert np.all(np.abs(as_f64(dx) - rdx) <= 2.0 ** -7 * np.abs(rdx) + 2.0 ** -16 * adx)
    assert np.all(np.abs(dgam.cpu().numpy().astype(np.float64) - rdg) <= (R + 8) * 2.0 ** -22 * adg + 1e-30)
    assert np.all(np.abs(dbet.cpu().numpy().astype(np.float64) - rdb) <= R * 2.0 ** -24 * adb + 1e-30)
