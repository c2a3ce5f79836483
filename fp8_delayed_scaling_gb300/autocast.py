"""fp8_autocast: the region whose casts record amaxes, closed by the scale update.

"FP8 低精度训练：Transformer Engine 简析" §三.3 (FP8框架TE计算流程): inside the
FP8 autocast the modules cast with the scales stored in fp8_meta and record
their tensors' amaxes; at autocast exit the amaxes of the processes in
fp8_group are reduced (MAX) and every scale is updated from its amax history,
for use by the next step.  That is this context manager:

    with fp8_autocast(state, group=None):
        y = layer.forward(x)
        layer.backward(dy)
    # exit: amaxes MAX-reduced over `group` (if any), then fp8_update_scale

The update is one launch over all slots of the state, enqueued on the current
stream; nothing synchronises with the host.  `step` counts the exits (it
drives the recipe's `interval`).  If the block raises, no update is made: a
step that did not finish records nothing.
"""
from __future__ import annotations

import threading

import torch

_active = threading.local()


def amax_view(buf: torch.Tensor, n_slots: int, stride: int) -> torch.Tensor:
    """The [n_slots] fp32 amax fields of a scaling-state block (bytes 8-11 of each slot),
    as a strided view of `buf`."""
    rows = buf.view(n_slots, stride)
    return rows[:, 8:12].view(torch.float32).view(n_slots)


def reduce_amax_(buf: torch.Tensor, n_slots: int, stride: int, group=None) -> None:
    """MAX all-reduce of the recorded amaxes over `group`, in place in `buf`.  After it
    every replica updates its scales from the same amaxes, so all replicas hold
    identical scales (the only exchange delayed scaling adds to data parallelism)."""
    am = amax_view(buf, n_slots, stride)
    flat = am.contiguous()
    torch.distributed.all_reduce(flat, op=torch.distributed.ReduceOp.MAX, group=group)
    am.copy_(flat)


class fp8_autocast:
    """Context manager closing each step of a ScalingState (see the module docstring).

    state    the ScalingState whose slots the block's casts record into
    enabled  False: a plain region, no update at exit
    group    a torch.distributed process group whose replicas share the scales, or None
    step     the step number of the first exit (default: continue the state's count)"""

    def __init__(self, state, enabled: bool = True, group=None, step: int | None = None, stream=None):
        self.state = state
        self.enabled = enabled
        self.group = group
        self.stream = stream
        if step is not None:
            state.step = step
        elif not hasattr(state, "step"):
            state.step = 0

    def __enter__(self):
        stack = getattr(_active, "stack", None)
        if stack is None:
            stack = _active.stack = []
        stack.append(self)
        return self

    def __exit__(self, exc_type, exc, tb):
        _active.stack.pop()
        if exc_type is not None or not self.enabled:
            return False
        st = self.state
        if self.group is not None:
            reduce_amax_(st.buf, st.n_slots, st.stride, self.group)
        st.update(st.step, self.stream)
        st.step += 1
        return False


def active() -> fp8_autocast | None:
    """The innermost fp8_autocast of this thread, or None."""
    stack = getattr(_active, "stack", None)
    return stack[-1] if stack else None
