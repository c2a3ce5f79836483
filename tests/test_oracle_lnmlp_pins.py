"""Pins of the oracle's LayerNormMLP pieces (CPU only) against independent
library routines in float64 (torch's layer_norm and gelu and their autograd),
textbook identities and finite differences."""
import numpy as np
import torch
import torch.nn.functional as F

import oracle


def _bf16(t):
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_layernorm_matches_torch_float64():
    g = torch.Generator().manual_seed(0)
    x = torch.randn(37, 96, generator=g).to(torch.bfloat16)
    gamma = (1 + 0.1 * torch.randn(96, generator=g)).to(torch.bfloat16)
    beta = (0.3 * torch.randn(96, generator=g)).to(torch.bfloat16)
    y, mu, rs = oracle.layernorm_fwd(_bf16(x), _bf16(gamma), _bf16(beta), 1e-5)
    ref = F.layer_norm(x.double(), (96,), gamma.double(), beta.double(), 1e-5).numpy()
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(mu, x.double().mean(1).numpy(), rtol=1e-12, atol=1e-14)
    var = x.double().var(1, unbiased=False).numpy()
    np.testing.assert_allclose(rs, 1 / np.sqrt(var + 1e-5), rtol=1e-12)


def test_layernorm_normalises_rows():
    x = np.random.default_rng(1).standard_normal((8, 512)).astype(np.float32) * 5 + 3
    ones, zeros = np.ones(512, np.float32), np.zeros(512, np.float32)
    y, _, _ = oracle.layernorm_fwd(x, ones, zeros, 0.0)
    np.testing.assert_allclose(y.mean(1), 0, atol=1e-12)
    np.testing.assert_allclose(y.var(1), 1, rtol=1e-12)


def test_gelu_matches_torch_and_identities():
    h = torch.linspace(-12, 12, 4097, dtype=torch.float64).to(torch.bfloat16)
    got = oracle.gelu(_bf16(h))
    ref = F.gelu(h.double(), approximate="none").numpy()
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-15)
    assert oracle.gelu(_bf16(torch.zeros(4)))[0] == 0.0
    big = torch.tensor([10.0, 20.0], dtype=torch.bfloat16)
    np.testing.assert_allclose(oracle.gelu(_bf16(big)), [10.0, 20.0], rtol=1e-15)


def test_dgelu_matches_autograd_and_finite_differences():
    h = torch.linspace(-8, 8, 2049, dtype=torch.float64).to(torch.bfloat16)
    dg = torch.randn(2049, generator=torch.Generator().manual_seed(2), dtype=torch.float64).to(torch.bfloat16)
    got = oracle.dgelu(_bf16(dg), _bf16(h))
    hd = h.double().requires_grad_(True)
    F.gelu(hd, approximate="none").backward(dg.double())
    np.testing.assert_allclose(got, hd.grad.numpy(), rtol=1e-13, atol=1e-15)
    # central differences of the oracle's own gelu in fp64 (step 1e-6) on fp32 inputs
    v = np.linspace(-5, 5, 101).astype(np.float32)
    eps = 1e-3
    fd = (oracle.gelu((v + eps).astype(np.float32)) - oracle.gelu((v - eps).astype(np.float32))) / (
        (v + eps).astype(np.float32).astype(np.float64) - (v - eps).astype(np.float32).astype(np.float64))
    np.testing.assert_allclose(oracle.dgelu(np.ones_like(v), v), fd, atol=2e-6)


def test_layernorm_bwd_matches_autograd():
    g = torch.Generator().manual_seed(3)
    R, C = 24, 128
    x = torch.randn(R, C, generator=g).to(torch.bfloat16)
    gamma = (1 + 0.1 * torch.randn(C, generator=g)).to(torch.bfloat16)
    beta = torch.zeros(C).to(torch.bfloat16)
    dy = torch.randn(R, C, generator=g).to(torch.bfloat16)
    _, mu, rs = oracle.layernorm_fwd(_bf16(x), _bf16(gamma), _bf16(beta), 1e-5)
    dx, dgam, dbet, dxa, _, _ = oracle.layernorm_bwd(_bf16(dy), _bf16(x), _bf16(gamma), mu, rs)
    xd = x.double().requires_grad_(True)
    gd = gamma.double().requires_grad_(True)
    bd = beta.double().requires_grad_(True)
    F.layer_norm(xd, (C,), gd, bd, 1e-5).backward(dy.double())
    np.testing.assert_allclose(dx, xd.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dgam, gd.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dbet, bd.grad.numpy(), rtol=1e-12, atol=1e-12)
    assert np.all(dxa >= np.abs(dx) - 1e-12)
