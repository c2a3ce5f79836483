"""te.LayerNormMLP under a DelayedScaling recipe, sequenced over the C ABI.

"NVIDIA Transformer Engine 加速训练教程" uses te.LayerNormMLP: LayerNorm ->
fc1 -> GELU -> fc2.  Under delayed scaling ("FP8 低精度训练：Transformer
Engine 简析" §三.1, §三.3) every GEMM operand is an FP8 cast with a stored
scale, so each activation is fused with the cast of its output:

  forward   LN+cast(x)        -> q_ln, q_ln^T      (slot fc1.in)
            cast W1           -> qW1, qW1^T        (slot fc1.w; one grouped launch with
                                                    W2's cast after step 0)
            h  = fc1(q_ln, qW1) + b1               (bf16)
            GELU+cast(h)      -> q_g, q_g^T        (slot fc2.in; fused into
                                                    the fc1 epilogue after step 0)
            cast W2           -> qW2, qW2^T        (slot fc2.w)
            y  = fc2(q_g, qW2) + b2                (bf16)
  backward  cast dY (+db2)    -> qdY, qdY^T        (slot fc2.grad)
            dW2 = wgrad(qdY^T, q_g^T);  dg = dgrad(qdY, qW2^T)
            dGELU+cast(dg, h) (+db1) -> qdh, qdh^T (slot fc1.grad; fused into
                                                    the dgrad epilogue after step 0,
                                                    so dg never reaches HBM)
            dln = dgrad(qdh, qW1^T);  dW1 = wgrad(qdh^T, q_ln^T)
            LN backward(dln, x) -> dx, dgamma, dbeta
  update    all six slots, one launch.

On the first step every slot's history is seeded with that step's own amax
(an amax-only pass) before its cast; because each activation depends on the
previous GEMM, the seeding is interleaved with the forward and backward.

scaling="current" runs the just-in-time alternative the same page contrasts
with delayed scaling (§三.1): each tensor's scale comes from its own amax of
this step, so every cast needs that amax first.  The producing kernel writes
the bf16 tensor and its amax, the seed call turns the amax into the current
scale (a history of length 1), and a separate cast pass reads the tensor
again — the extra HBM round trip that delayed scaling avoids.

Under delayed scaling the two weights can be cached across micro-batches
(is_first_microbatch, as for te.Linear in linear.py).
"""
from __future__ import annotations

import torch

from . import (E4M3, E5M2, FORMAT_HYBRID, Recipe, ScalingState, fp8_cast_amax_transpose, fp8_cast_workspace_size,
               fp8_dgelu_cast, fp8_gelu_cast, fp8_gemm, fp8_gemm_dgelu_cast, fp8_gemm_dgelu_workspace_size,
               fp8_gemm_gelu_cast, fp8_layernorm_bwd,
               fp8_layernorm_bwd_workspace_size, fp8_layernorm_cast, fp8_seed_amax_history)
from .linear import WeightCache, cast_weights

FC1_IN, FC1_W, FC1_GRAD, FC2_IN, FC2_W, FC2_GRAD = range(6)
SLOTS = 6


def slot_dtypes(recipe: Recipe):
    g = E5M2 if recipe.fp8_format == FORMAT_HYBRID else E4M3
    return [E4M3, E4M3, g, E4M3, E4M3, g]


def make_state(recipe: Recipe, n_blocks: int = 1, device="cuda") -> ScalingState:
    return ScalingState(recipe, slot_dtypes(recipe) * n_blocks, device=device)


class Fp8LayerNormMLP:
    def __init__(self, state: ScalingState, block_index: int, gamma, beta, w1, b1, w2, b2, tokens: int,
                 eps: float = 1e-5, keep_activations: bool = False, scaling: str = "delayed", fused: bool = True):
        assert scaling in ("delayed", "current")
        self.scaling = scaling
        # GELU + cast inside the fc1 GEMM's epilogue and dGELU + cast (+ db1) inside the fc2
        # dgrad's (delayed scaling, after step 0)
        self.fused = fused
        self.state = state
        self.base = block_index * SLOTS
        self.recipe = state.recipe
        self.gamma, self.beta, self.w1, self.b1, self.w2, self.b2 = gamma, beta, w1, b1, w2, b2
        self.F, self.H = w1.shape
        self.M = tokens
        self.eps = eps
        self.gfmt = E5M2 if self.recipe.fp8_format == FORMAT_HYBRID else E4M3
        dev = w1.device
        M, F, H = self.M, self.F, self.H
        u8 = dict(dtype=torch.uint8, device=dev)
        bf = dict(dtype=torch.bfloat16, device=dev)
        f32 = dict(dtype=torch.float32, device=dev)
        self.q_ln, self.q_lnT = torch.empty((M, H), **u8), torch.empty((H, M), **u8)
        self.mu, self.rs = torch.empty(M, **f32), torch.empty(M, **f32)
        self.qw1, self.qw1T = torch.empty((F, H), **u8), torch.empty((H, F), **u8)
        self.h = torch.empty((M, F), **bf)
        self.q_g, self.q_gT = torch.empty((M, F), **u8), torch.empty((F, M), **u8)
        self.qw2, self.qw2T = torch.empty((H, F), **u8), torch.empty((F, H), **u8)
        self.y = torch.empty((M, H), **bf)
        self.qdy, self.qdyT = torch.empty((M, H), **u8), torch.empty((H, M), **u8)
        self.db2 = torch.empty(H, **f32)
        self.dg = torch.empty((M, F), **bf)
        self.dw2 = torch.empty((H, F), **bf)
        self.qdh, self.qdhT = torch.empty((M, F), **u8), torch.empty((F, M), **u8)
        self.db1 = torch.empty(F, **f32)
        self.dln = torch.empty((M, H), **bf)
        self.dw1 = torch.empty((F, H), **bf)
        self.dx = torch.empty((M, H), **bf)
        self.dgamma, self.dbeta = torch.empty(H, **f32), torch.empty(H, **f32)
        self.ws_cast = torch.empty(max(fp8_cast_workspace_size(M, H), fp8_cast_workspace_size(M, F)), **u8)
        self.ws_ln = torch.empty(fp8_layernorm_bwd_workspace_size(M, H), **u8)
        # fused dGELU epilogue: fc1 bias-gradient partials per 32-row group
        self.ws_dgelu = torch.empty(fp8_gemm_dgelu_workspace_size(M, F), **u8) if fused else None
        self.w1cache, self.w2cache = WeightCache(self.qw1, self.qw1T), WeightCache(self.qw2, self.qw2T)
        self.w1_sinv = self.w2_sinv = None  # the weights' decode factors used by this step's forward
        self.keep = keep_activations
        if keep_activations or scaling == "current":  # the bf16 tensors that are cast
            self.y_ln = torch.empty((M, H), **bf)
            self.g = torch.empty((M, F), **bf)
            self.dh = torch.empty((M, F), **bf)
        else:
            self.y_ln = self.g = self.dh = None

    def slot(self, k: int) -> int:
        return self.base + k

    def _seed(self, first: int, count: int, stream) -> None:
        fp8_seed_amax_history(self.recipe, count, self.state.buf.data_ptr() + self.slot(first) * self.state.stride,
                              stream=stream)

    def _current_cast(self, t: torch.Tensor, fmt: int, slot: int, out, out_t, stream, dbias=None) -> None:
        """Just-in-time cast: the slot's amax was recorded by the producer; turn it into
        this step's scale, then cast."""
        self._seed(slot - self.base, 1, stream)
        fp8_cast_amax_transpose(t, fmt, self.state.scale(slot), out=out, out_t=out_t, dbias=dbias,
                                workspace=self.ws_cast if dbias is not None else None, stream=stream)

    def forward(self, x: torch.Tensor, seed: bool = False, stream=None, is_first_microbatch=None) -> torch.Tensor:
        """is_first_microbatch: the FP8 weight cache of te modules (None: cast the
        weights every call; True: cast and keep them; False: reuse the kept codes)."""
        if self.scaling == "current":
            if is_first_microbatch is not None:
                raise ValueError("the FP8 weight cache is defined for delayed scaling only")
            return self._forward_current(x, stream)
        if seed and is_first_microbatch is False:
            raise ValueError("the seeding step casts the weights; it cannot reuse a cached copy")
        self.w1cache.check(is_first_microbatch)
        self.w2cache.check(is_first_microbatch)
        st = self.state
        s = self.slot
        if seed:
            fp8_layernorm_cast(x, self.gamma, self.beta, self.eps, E4M3, None, self.mu, self.rs,
                               amax=st.amax(s(FC1_IN)), stream=stream)
            fp8_cast_amax_transpose(self.w1, E4M3, None, amax=st.amax(s(FC1_W)), stream=stream)
            self._seed(FC1_IN, 2, stream)
        fp8_layernorm_cast(x, self.gamma, self.beta, self.eps, E4M3, st.scale(s(FC1_IN)), self.mu, self.rs,
                           out=self.q_ln, out_t=self.q_lnT, amax=st.amax(s(FC1_IN)), y=self.y_ln, stream=stream)
        if self.fused and not seed:
            # both weights in one grouped cast (their scales are this step's delayed ones)
            self.w1_sinv, self.w2_sinv = cast_weights([self.w1cache, self.w2cache], [self.w1, self.w2], st,
                                                      [s(FC1_W), s(FC2_W)], is_first_microbatch, stream)
            fp8_gemm_gelu_cast(self.q_ln, E4M3, self.qw1, E4M3, st.scale_inv(s(FC1_IN)), self.w1_sinv, self.h,
                               E4M3, st.scale(s(FC2_IN)), self.q_g, self.q_gT, q_amax=st.amax(s(FC2_IN)),
                               bias=self.b1, g=self.g, stream=stream)
            fp8_gemm(self.q_g, E4M3, self.qw2, E4M3, st.scale_inv(s(FC2_IN)), self.w2_sinv, self.y,
                     bias=self.b2, stream=stream)
            return self.y
        self.w1_sinv = self.w1cache.cast(self.w1, st, s(FC1_W), is_first_microbatch, stream)
        fp8_gemm(self.q_ln, E4M3, self.qw1, E4M3, st.scale_inv(s(FC1_IN)), self.w1_sinv, self.h,
                 bias=self.b1, stream=stream)
        if seed:
            fp8_gelu_cast(self.h, E4M3, None, amax=st.amax(s(FC2_IN)), g=None, stream=stream)
            fp8_cast_amax_transpose(self.w2, E4M3, None, amax=st.amax(s(FC2_W)), stream=stream)
            self._seed(FC2_IN, 2, stream)
        fp8_gelu_cast(self.h, E4M3, st.scale(s(FC2_IN)), out=self.q_g, out_t=self.q_gT, amax=st.amax(s(FC2_IN)),
                      g=self.g, stream=stream)
        self.w2_sinv = self.w2cache.cast(self.w2, st, s(FC2_W), is_first_microbatch, stream)
        fp8_gemm(self.q_g, E4M3, self.qw2, E4M3, st.scale_inv(s(FC2_IN)), self.w2_sinv, self.y,
                 bias=self.b2, stream=stream)
        return self.y

    def _forward_current(self, x, stream):
        st, s = self.state, self.slot
        fp8_layernorm_cast(x, self.gamma, self.beta, self.eps, E4M3, None, self.mu, self.rs, amax=st.amax(s(FC1_IN)),
                           y=self.y_ln, stream=stream)
        self._current_cast(self.y_ln, E4M3, s(FC1_IN), self.q_ln, self.q_lnT, stream)
        fp8_cast_amax_transpose(self.w1, E4M3, None, amax=st.amax(s(FC1_W)), stream=stream)
        self._current_cast(self.w1, E4M3, s(FC1_W), self.qw1, self.qw1T, stream)
        fp8_gemm(self.q_ln, E4M3, self.qw1, E4M3, st.scale_inv(s(FC1_IN)), st.scale_inv(s(FC1_W)), self.h,
                 bias=self.b1, stream=stream)
        fp8_gelu_cast(self.h, E4M3, None, amax=st.amax(s(FC2_IN)), g=self.g, stream=stream)
        self._current_cast(self.g, E4M3, s(FC2_IN), self.q_g, self.q_gT, stream)
        fp8_cast_amax_transpose(self.w2, E4M3, None, amax=st.amax(s(FC2_W)), stream=stream)
        self._current_cast(self.w2, E4M3, s(FC2_W), self.qw2, self.qw2T, stream)
        fp8_gemm(self.q_g, E4M3, self.qw2, E4M3, st.scale_inv(s(FC2_IN)), st.scale_inv(s(FC2_W)), self.y,
                 bias=self.b2, stream=stream)
        return self.y

    def _backward_current(self, x, dy, stream):
        st, s, g = self.state, self.slot, self.gfmt
        fp8_cast_amax_transpose(dy, g, None, amax=st.amax(s(FC2_GRAD)), stream=stream)
        self._current_cast(dy, g, s(FC2_GRAD), self.qdy, self.qdyT, stream, dbias=self.db2)
        fp8_gemm(self.qdy, g, self.qw2T, E4M3, st.scale_inv(s(FC2_GRAD)), st.scale_inv(s(FC2_W)), self.dg,
                 stream=stream)
        fp8_gemm(self.qdyT, g, self.q_gT, E4M3, st.scale_inv(s(FC2_GRAD)), st.scale_inv(s(FC2_IN)), self.dw2,
                 stream=stream)
        fp8_dgelu_cast(self.dg, self.h, g, None, amax=st.amax(s(FC1_GRAD)), dh=self.dh, stream=stream)
        self._current_cast(self.dh, g, s(FC1_GRAD), self.qdh, self.qdhT, stream, dbias=self.db1)
        fp8_gemm(self.qdh, g, self.qw1T, E4M3, st.scale_inv(s(FC1_GRAD)), st.scale_inv(s(FC1_W)), self.dln,
                 stream=stream)
        fp8_gemm(self.qdhT, g, self.q_lnT, E4M3, st.scale_inv(s(FC1_GRAD)), st.scale_inv(s(FC1_IN)), self.dw1,
                 stream=stream)
        fp8_layernorm_bwd(self.dln, x, self.gamma, self.mu, self.rs, self.dx, self.dgamma, self.dbeta, self.ws_ln,
                          stream=stream)
        return self.dx

    def backward(self, x: torch.Tensor, dy: torch.Tensor, seed: bool = False, stream=None):
        if self.scaling == "current":
            return self._backward_current(x, dy, stream)
        st = self.state
        s = self.slot
        g = self.gfmt
        if seed:
            fp8_cast_amax_transpose(dy, g, None, amax=st.amax(s(FC2_GRAD)), stream=stream)
            self._seed(FC2_GRAD, 1, stream)
        fp8_cast_amax_transpose(dy, g, st.scale(s(FC2_GRAD)), out=self.qdy, out_t=self.qdyT,
                                amax=st.amax(s(FC2_GRAD)), dbias=self.db2, workspace=self.ws_cast, stream=stream)
        fp8_gemm(self.qdyT, g, self.q_gT, E4M3, st.scale_inv(s(FC2_GRAD)), st.scale_inv(s(FC2_IN)), self.dw2,
                 stream=stream)
        if self.fused and not seed:  # dgrad with dGELU + cast + dbias in its epilogue; dg stays on chip
            fp8_gemm_dgelu_cast(self.qdy, g, self.qw2T, E4M3, st.scale_inv(s(FC2_GRAD)), self.w2_sinv, self.h, g,
                                st.scale(s(FC1_GRAD)), self.qdh, self.qdhT, q_amax=st.amax(s(FC1_GRAD)),
                                dbias=self.db1, workspace=self.ws_dgelu, dg=self.dg if self.keep else None,
                                dh=self.dh, stream=stream)
            return self._backward_fc1(x, stream)
        fp8_gemm(self.qdy, g, self.qw2T, E4M3, st.scale_inv(s(FC2_GRAD)), self.w2_sinv, self.dg, stream=stream)
        if seed:
            fp8_dgelu_cast(self.dg, self.h, g, None, amax=st.amax(s(FC1_GRAD)), stream=stream)
            self._seed(FC1_GRAD, 1, stream)
        fp8_dgelu_cast(self.dg, self.h, g, st.scale(s(FC1_GRAD)), out=self.qdh, out_t=self.qdhT,
                       amax=st.amax(s(FC1_GRAD)), dbias=self.db1, workspace=self.ws_cast, dh=self.dh, stream=stream)
        return self._backward_fc1(x, stream)

    def _backward_fc1(self, x: torch.Tensor, stream):
        """fc1 dgrad and wgrad from the dh codes, then the LayerNorm backward."""
        st, s, g = self.state, self.slot, self.gfmt
        fp8_gemm(self.qdh, g, self.qw1T, E4M3, st.scale_inv(s(FC1_GRAD)), self.w1_sinv, self.dln, stream=stream)
        fp8_gemm(self.qdhT, g, self.q_lnT, E4M3, st.scale_inv(s(FC1_GRAD)), st.scale_inv(s(FC1_IN)), self.dw1,
                 stream=stream)
        fp8_layernorm_bwd(self.dln, x, self.gamma, self.mu, self.rs, self.dx, self.dgamma, self.dbeta, self.ws_ln,
                          stream=stream)
        return self.dx
