"""te.Linear under a DelayedScaling recipe, sequenced over the C ABI.

"FP8 低精度训练：Transformer Engine 简析", §三.3 "FP8框架TE计算流程": inside
the FP8 autocast a TE module casts its input and weight to FP8 with the scales
stored in fp8_meta, records their amaxes, and calls fp8_gemm; the backward
casts grad_output (E5M2 in HYBRID, §三.1) and runs the gradient GEMMs; at
autocast exit the recorded amaxes update the history and the scales used by
the next step.

Slots of one layer in the shared ScalingState: base+0 input (E4M3),
base+1 weight (E4M3), base+2 grad_output (E5M2 in HYBRID, else E4M3).

Per step, for D = X W^T + b with X [M x K], W [N x K]:
  forward   cast X -> qX (+ qX^T for wgrad), cast W -> qW (+ qW^T for dgrad)
            (one grouped launch for both)
            Y[M,N]  = fp8_gemm(qX, qW)            * sx_inv * sw_inv + b
  backward  cast dY -> qdY, qdY^T (+ db = column sums of dY)
            dX[M,K] = fp8_gemm(qdY, qW^T)        * sdy_inv * sw_inv
            dW[N,K] = fp8_gemm(qdY^T, qX^T)      * sdy_inv * sx_inv
  update    fp8_update_scale over all slots (one launch)

FP8 weight cache (§三.3: the weight cast is skipped while a cached FP8 copy
exists).  forward(..., is_first_microbatch=True) casts the weight and keeps the
codes together with the decode factor they were cast at; later micro-batches
(is_first_microbatch=False) reuse both and launch no weight cast.  The decode
factor must travel with the codes: the scale update after each forward may
already have moved the slot's scale_inv on (a new weight amax entered the
history).  A skipped cast records no weight amax for that step.

scaling="current" runs the just-in-time alternative that §三.1 contrasts with
delayed scaling: each tensor's scale comes from its own amax of this step.  A
cast is then an amax-only pass over the tensor, the amax turned into the
slot's scale (fp8_seed_amax_history over one slot), and the cast: the tensor
is read twice, and no history is kept or updated.
"""
from __future__ import annotations

import torch

from . import (E4M3, E5M2, FORMAT_HYBRID, Recipe, ScalingState, fp8_cast_amax_transpose,
               fp8_cast_amax_transpose_multi, fp8_cast_workspace_size, fp8_gemm, fp8_seed_amax_history)

SLOTS_PER_LAYER = 3
IN, WEIGHT, GRAD = 0, 1, 2


class WeightCache:
    """The FP8 codes of one weight (row-major and transposed) and the scale_inv
    they decode with.  `valid` says the codes stand for the current weight."""

    def __init__(self, q: torch.Tensor, q_t: torch.Tensor | None):
        self.q, self.q_t = q, q_t
        self.scale_inv = torch.empty(1, dtype=torch.float32, device=q.device)
        self.valid = False

    def check(self, is_first_microbatch) -> None:
        """Raise before any launch when a reuse is asked for and nothing is cached."""
        if is_first_microbatch is False and not self.valid:
            raise RuntimeError("is_first_microbatch=False, but no FP8 copy of the weight is cached: "
                               "cast it first with is_first_microbatch=True")

    def cast(self, w: torch.Tensor, state: ScalingState, slot: int, is_first_microbatch, stream=None):
        """Cast w into the cache (or reuse it) and return the scale_inv to decode with:
        None -> cast, decode with the slot's scale_inv, nothing kept;
        True -> cast, keep the codes and their decode factor;
        False -> no launch, the kept codes and factor."""
        self.check(is_first_microbatch)
        if is_first_microbatch is False:
            return self.scale_inv
        keep = bool(is_first_microbatch)
        fp8_cast_amax_transpose(w, E4M3, state.scale(slot), out=self.q, out_t=self.q_t, amax=state.amax(slot),
                                scale_inv_out=self.scale_inv if keep else None, stream=stream)
        self.valid = keep
        return self.scale_inv if keep else state.scale_inv(slot)


def cast_weights(caches, weights, state: ScalingState, slots, is_first_microbatch, stream=None):
    """WeightCache.cast of several weights with one grouped launch (the same codes, amaxes and
    decode factors as one cast each); returns their decode factors."""
    for c in caches:
        c.check(is_first_microbatch)
    if is_first_microbatch is False:
        return [c.scale_inv for c in caches]
    keep = bool(is_first_microbatch)
    fp8_cast_amax_transpose_multi([dict(x=w, scale=state.scale(s), out=c.q, out_t=c.q_t, amax=state.amax(s),
                                        scale_inv_out=c.scale_inv if keep else None)
                                   for c, w, s in zip(caches, weights, slots)], E4M3, stream=stream)
    for c in caches:
        c.valid = keep
    return [c.scale_inv if keep else state.scale_inv(s) for c, s in zip(caches, slots)]


def layer_slot_dtypes(recipe: Recipe):
    return [E4M3, E4M3, E5M2 if recipe.fp8_format == FORMAT_HYBRID else E4M3]


def make_state(recipe: Recipe, n_layers: int, device="cuda") -> ScalingState:
    return ScalingState(recipe, layer_slot_dtypes(recipe) * n_layers, device=device)


class Fp8Linear:
    """One linear layer's FP8 buffers and step sequencing (no autograd)."""

    def __init__(self, state: ScalingState, layer_index: int, weight: torch.Tensor, bias: torch.Tensor | None,
                 tokens: int, out_dtype=torch.bfloat16, training: bool = True, scaling: str = "delayed"):
        assert scaling in ("delayed", "current")
        self.scaling = scaling
        self.state = state
        self.base = layer_index * SLOTS_PER_LAYER
        self.recipe = state.recipe
        self.w = weight
        self.b = bias
        self.N, self.K = weight.shape
        self.M = tokens
        dev = weight.device
        u8 = dict(dtype=torch.uint8, device=dev)
        M, N, K = self.M, self.N, self.K
        self.training = training
        self.qx = torch.empty((M, K), **u8)
        self.qw = torch.empty((N, K), **u8)
        self.y = torch.empty((M, N), dtype=out_dtype, device=dev)
        if training:
            self.qxT = torch.empty((K, M), **u8)
            self.qwT = torch.empty((K, N), **u8)
            self.qdy = torch.empty((M, N), **u8)
            self.qdyT = torch.empty((N, M), **u8)
            self.dx = torch.empty((M, K), dtype=torch.bfloat16, device=dev)
            self.dw = torch.empty((N, K), dtype=torch.bfloat16, device=dev)
            self.db = torch.empty((N,), dtype=torch.float32, device=dev) if bias is not None else None
            self.ws = torch.empty(fp8_cast_workspace_size(M, N), dtype=torch.uint8, device=dev)
        self.bwd_dtype = E5M2 if self.recipe.fp8_format == FORMAT_HYBRID else E4M3
        self.wcache = WeightCache(self.qw, self.qwT if training else None)
        self.w_sinv = None  # the weight's decode factor used by this step's forward

    def slot(self, k: int) -> int:
        return self.base + k

    def _state_at(self, k: int) -> int:
        return self.state.buf.data_ptr() + self.slot(k) * self.state.stride

    def seed_forward(self, x: torch.Tensor, stream=None) -> None:
        """First step: amax-only passes over input and weight, then seed their histories."""
        st = self.state
        fp8_cast_amax_transpose(x, E4M3, None, amax=st.amax(self.slot(IN)), stream=stream)
        fp8_cast_amax_transpose(self.w, E4M3, None, amax=st.amax(self.slot(WEIGHT)), stream=stream)
        fp8_seed_amax_history(self.recipe, 2, self._state_at(IN), stream=stream)

    def seed_backward(self, dy: torch.Tensor, stream=None) -> None:
        st = self.state
        fp8_cast_amax_transpose(dy, self.bwd_dtype, None, amax=st.amax(self.slot(GRAD)), stream=stream)
        fp8_seed_amax_history(self.recipe, 1, self._state_at(GRAD), stream=stream)

    def _current_cast(self, t: torch.Tensor, fmt: int, k: int, out, out_t, stream, dbias=None) -> None:
        """Just-in-time cast of t into slot k: amax-only pass, this step's scale, cast."""
        st = self.state
        fp8_cast_amax_transpose(t, fmt, None, amax=st.amax(self.slot(k)), stream=stream)
        fp8_seed_amax_history(self.recipe, 1, self._state_at(k), stream=stream)
        fp8_cast_amax_transpose(t, fmt, st.scale(self.slot(k)), out=out, out_t=out_t, dbias=dbias,
                                workspace=self.ws if dbias is not None else None, stream=stream)

    def forward(self, x: torch.Tensor, stream=None, is_first_microbatch=None) -> torch.Tensor:
        st = self.state
        tr = self.training
        if self.scaling == "current":
            if is_first_microbatch is not None:
                raise RuntimeError("the weight cache keeps codes at a delayed scale; current scaling recasts")
            self._current_cast(x, E4M3, IN, self.qx, self.qxT if tr else None, stream)
            self._current_cast(self.w, E4M3, WEIGHT, self.qw, self.qwT if tr else None, stream)
            self.w_sinv = st.scale_inv(self.slot(WEIGHT))
            fp8_gemm(self.qx, E4M3, self.qw, E4M3, st.scale_inv(self.slot(IN)), self.w_sinv, self.y, bias=self.b,
                     stream=stream)
            return self.y
        self.wcache.check(is_first_microbatch)
        x_item = dict(x=x, scale=st.scale(self.slot(IN)), out=self.qx, out_t=self.qxT if tr else None,
                      amax=st.amax(self.slot(IN)))
        if is_first_microbatch is not False and x.dtype == self.w.dtype:
            # input and weight in one grouped cast
            keep = bool(is_first_microbatch)
            c = self.wcache
            fp8_cast_amax_transpose_multi([x_item, dict(x=self.w, scale=st.scale(self.slot(WEIGHT)), out=c.q,
                                                        out_t=c.q_t, amax=st.amax(self.slot(WEIGHT)),
                                                        scale_inv_out=c.scale_inv if keep else None)],
                                          E4M3, stream=stream)
            c.valid = keep
            self.w_sinv = c.scale_inv if keep else st.scale_inv(self.slot(WEIGHT))
        else:
            fp8_cast_amax_transpose(x, E4M3, x_item["scale"], out=self.qx, out_t=x_item["out_t"],
                                    amax=x_item["amax"], stream=stream)
            self.w_sinv = self.wcache.cast(self.w, st, self.slot(WEIGHT), is_first_microbatch, stream)
        fp8_gemm(self.qx, E4M3, self.qw, E4M3, st.scale_inv(self.slot(IN)), self.w_sinv, self.y, bias=self.b,
                 stream=stream)
        return self.y

    def backward(self, dy: torch.Tensor, stream=None):
        st = self.state
        g = self.slot(GRAD)
        if self.scaling == "current":
            self._current_cast(dy, self.bwd_dtype, GRAD, self.qdy, self.qdyT, stream, dbias=self.db)
        else:
            fp8_cast_amax_transpose(dy, self.bwd_dtype, st.scale(g), out=self.qdy, out_t=self.qdyT,
                                    amax=st.amax(g), dbias=self.db, workspace=self.ws if self.db is not None else None,
                                    stream=stream)
        fp8_gemm(self.qdy, self.bwd_dtype, self.qwT, E4M3, st.scale_inv(g), self.w_sinv, self.dx, stream=stream)
        fp8_gemm(self.qdyT, self.bwd_dtype, self.qxT, E4M3, st.scale_inv(g), st.scale_inv(self.slot(IN)),
                 self.dw, stream=stream)
        return self.dx, self.dw, self.db
