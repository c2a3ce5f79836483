"""te.Linear under an MXFP8 block-scaling recipe, sequenced over the C ABI.

MXFP8 is named by the Transformer Engine README ("亮点": MXFP8 on Blackwell).
Every operand is quantised per 32-element block along its GEMM's reduction
axis with its own E8M0 scale, so there is no amax history and no delay:

  forward   X -> row-wise (blocks along K) + column-wise (blocks along M)
            W -> row-wise (blocks along K) + column-wise (blocks along N)
            Y[M,N]  = mx_gemm(X_row, W_row) + b
  backward  dY -> row-wise (blocks along N) + column-wise (blocks along M)
            dX[M,K] = mx_gemm(dY_row, W_col)     (reduction over N)
            dW[N,K] = mx_gemm(dY_col, X_col)     (reduction over M)
            db      = column sums of dY, in the same pass as dY's quantisation

Micro-batching (te modules' is_first_microbatch): forward(..., is_first_microbatch=True)
quantises the weight and keeps both copies; later micro-batches (False) reuse them and launch
no weight quantisation.  MXFP8 has no scaling state, so the cached codes and E8M0 scales stand
alone.  None (the default) quantises the weight at every forward.
"""
from __future__ import annotations

import torch

from . import fp8_cast_workspace_size, mxfp8_gemm, mxfp8_quantize, mxfp8_scale_bytes


class MXTensor:
    """Row- and column-wise MXFP8 copies of one [R x C] matrix."""

    def __init__(self, rows: int, cols: int, device):
        u8 = dict(dtype=torch.uint8, device=device)
        self.row_q = torch.empty((rows, cols), **u8)
        self.row_s = torch.empty(mxfp8_scale_bytes(rows, cols), **u8)
        self.col_q = torch.empty((cols, rows), **u8)
        self.col_s = torch.empty(mxfp8_scale_bytes(cols, rows), **u8)

    def quantize(self, x: torch.Tensor, rowwise=True, colwise=True, dbias=None, workspace=None, stream=None) -> None:
        mxfp8_quantize(x, self.row_q if rowwise else None, self.row_s if rowwise else None,
                       self.col_q if colwise else None, self.col_s if colwise else None, dbias=dbias,
                       workspace=workspace, stream=stream)


class MxLinear:
    def __init__(self, weight: torch.Tensor, bias: torch.Tensor | None, tokens: int, out_dtype=torch.bfloat16):
        self.w, self.b = weight, bias
        self.N, self.K = weight.shape
        self.M = tokens
        dev = weight.device
        M, N, K = self.M, self.N, self.K
        self.mx_x = MXTensor(M, K, dev)
        self.mx_w = MXTensor(N, K, dev)
        self.mx_dy = MXTensor(M, N, dev)
        self.y = torch.empty((M, N), dtype=out_dtype, device=dev)
        self.dx = torch.empty((M, K), dtype=torch.bfloat16, device=dev)
        self.dw = torch.empty((N, K), dtype=torch.bfloat16, device=dev)
        self.db = torch.empty(N, dtype=torch.float32, device=dev) if bias is not None else None
        self.ws = torch.empty(fp8_cast_workspace_size(M, N), dtype=torch.uint8, device=dev) if bias is not None else None
        self.w_cached = False  # mx_w holds the current weight's copies, kept for reuse

    def forward(self, x: torch.Tensor, stream=None, is_first_microbatch=None) -> torch.Tensor:
        if is_first_microbatch is False and not self.w_cached:
            raise RuntimeError("is_first_microbatch=False, but no MXFP8 copy of the weight is cached: "
                               "quantise it first with is_first_microbatch=True")
        self.mx_x.quantize(x, stream=stream)
        if is_first_microbatch is not False:
            self.mx_w.quantize(self.w, stream=stream)
            self.w_cached = bool(is_first_microbatch)
        mxfp8_gemm(self.mx_x.row_q, self.mx_x.row_s, self.mx_w.row_q, self.mx_w.row_s, self.y, bias=self.b,
                   stream=stream)
        return self.y

    def backward(self, dy: torch.Tensor, stream=None):
        self.mx_dy.quantize(dy, dbias=self.db, workspace=self.ws, stream=stream)
        mxfp8_gemm(self.mx_dy.row_q, self.mx_dy.row_s, self.mx_w.col_q, self.mx_w.col_s, self.dx, stream=stream)
        mxfp8_gemm(self.mx_dy.col_q, self.mx_dy.col_s, self.mx_x.col_q, self.mx_x.col_s, self.dw, stream=stream)
        return self.dx, self.dw, self.db
