"""Seeded synthetic inputs for the FP8 delayed-scaling linear workloads.

This module is the one thing the CUDA path's tests/benchmark and the oracle
share: it draws the input tensors (shapes, distributions, seeds) and holds
none of the method's arithmetic.  Every tensor is drawn on the CPU from a
``torch.Generator`` seeded by (workload seed, tensor id, step), so the same
bytes reach the GPU and the oracle.

Workloads (the shapes are the te.Linear example of the Transformer Engine
README, "示例 PyTorch": 2048 tokens, 768 -> 3072; Llama-7B-shaped projections;
an MXFP8 MLP; a LayerNormMLP):

  linear_fwd      X fp32 [2048 x 768] ~N(0,1), W fp32 [3072 x 768] ~N(0,0.02),
                  bias zeros; E4M3 recipe, margin 0, interval 1, history 16.
  linear_hybrid   same layer, fresh X and dY each step; dY bf16 ~N(0,1e-3)
                  with 0.1 % of the entries (seeded positions) x1000;
                  HYBRID recipe, history 16, 10 steps.
  llama_proj      tokens 8192, hidden 4096: QKV 4096->12288, out 4096->4096,
                  up 4096->11008, down 11008->4096; X bf16 Student-t(3) x 0.5,
                  W bf16 ~N(0,0.02), dY bf16 ~N(0,1e-3); HYBRID, history 1024.
  mx_mlp          16384 tokens, 8192 -> 28672 -> 8192; X bf16 ~N(0,1) times a
                  per-input-channel factor log-uniform in [1e-3, 1e2]; W bf16
                  ~N(0,0.02); dY bf16 ~N(0,1); MXFP8 (1x32 E8M0 blocks).
  ln_mlp          x bf16 [16384 x 4096] ~N(0,1), gamma ~N(1,0.1), beta 0,
                  fc1 4096->16384, fc2 16384->4096, W ~N(0,0.02), dY ~N(0,1e-3);
                  HYBRID, history 16, 20 steps.
"""
from __future__ import annotations

import hashlib

import numpy as np
import torch

SEEDS = {"linear_fwd": 0, "linear_hybrid": 1, "llama_proj": 2, "mx_mlp": 3, "ln_mlp": 4}

LLAMA_PROJ = [  # (name, in_features K, out_features N); tokens M = 8192
    ("qkv", 4096, 12288),
    ("out", 4096, 4096),
    ("up", 4096, 11008),
    ("down", 11008, 4096),
]


def generator(seed: int, tensor: str, step: int = 0) -> torch.Generator:
    """A CPU generator for one (workload seed, tensor name, step) triple."""
    h = hashlib.sha256(f"{seed}/{tensor}/{step}".encode()).digest()
    g = torch.Generator(device="cpu")
    g.manual_seed(int.from_bytes(h[:8], "little") & ((1 << 63) - 1))
    return g


def normal(shape, std: float, g: torch.Generator, dtype=torch.float32) -> torch.Tensor:
    """N(0, std^2) drawn in fp32, then rounded (nearest even) to `dtype`."""
    return (torch.randn(shape, generator=g, dtype=torch.float32) * std).to(dtype)


def student_t3(shape, mult: float, g: torch.Generator, dtype=torch.bfloat16) -> torch.Tensor:
    """Student-t with 3 degrees of freedom times `mult`: Z / sqrt(chi2_3 / 3)."""
    z = torch.randn(shape, generator=g, dtype=torch.float32)
    c = torch.randn((3,) + tuple(shape), generator=g, dtype=torch.float32)
    chi2 = (c * c).sum(0)
    return (z / torch.sqrt(chi2 / 3.0) * mult).to(dtype)


def log_uniform(n: int, lo: float, hi: float, g: torch.Generator) -> torch.Tensor:
    """n values exp(U(ln lo, ln hi)), fp32."""
    u = torch.rand(n, generator=g, dtype=torch.float64)
    return torch.exp(np.log(lo) + u * (np.log(hi) - np.log(lo))).to(torch.float32)


def with_outliers(t: torch.Tensor, frac: float, factor: float, g: torch.Generator) -> torch.Tensor:
    """Multiply a seeded `frac` of the entries (distinct positions) by `factor`."""
    flat = t.reshape(-1).to(torch.float32)
    k = max(1, int(round(flat.numel() * frac)))
    idx = torch.randperm(flat.numel(), generator=g)[:k]
    flat = flat.clone()
    flat[idx] *= factor
    return flat.reshape(t.shape).to(t.dtype)


def channel_scaled_normal(rows: int, cols: int, g: torch.Generator) -> torch.Tensor:
    """bf16 [rows x cols] ~N(0,1) times a per-column factor log-uniform in [1e-3, 1e2]."""
    s = log_uniform(cols, 1e-3, 1e2, g)
    return (torch.randn((rows, cols), generator=g, dtype=torch.float32) * s[None, :]).to(torch.bfloat16)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """The bf16 tensor's bit patterns as a uint16 numpy array (CPU copy)."""
    assert t.dtype == torch.bfloat16
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def host_array(t: torch.Tensor) -> np.ndarray:
    """numpy view for the oracle: float32 stays float32, bf16 becomes uint16 bits."""
    if t.dtype == torch.bfloat16:
        return bf16_bits(t)
    if t.dtype == torch.float32:
        return t.detach().cpu().contiguous().numpy()
    if t.dtype == torch.uint8:
        return t.detach().cpu().contiguous().numpy()
    raise TypeError(t.dtype)
