"""StepGraph: a training step captured once as a CUDA graph and replayed.

A step of this library is a fixed sequence of launches on one stream.  The
launches take every scale, scale_inv and amax from device memory, and every
buffer is allocated before the first step.  A captured step therefore stays
valid while the scales evolve, and replaying it removes the per-launch host
cost, which decides the step time of small layers.

The one host argument that changes between steps is the step counter passed
to fp8_update_scale: it decides whether the step recomputes the scales
(every `interval` steps).  StepGraph captures one graph per residue of the
counter modulo `interval` and replays the matching one.  Anything else a step
function passes from the host (shapes, pointers, flags) is frozen at capture.
"""
from __future__ import annotations

from typing import Callable

import torch


class StepGraph:
    """step_fn(step_no) enqueues one whole step on the current stream (casts, GEMMs, the update
    with `step_no`).  interval: the recipe's scale-update interval.  warmup: eager steps run on
    a side stream before capture (library setup, allocator warm-up); they are real steps and
    advance the state, numbered from `first_step`."""

    def __init__(self, step_fn: Callable[[int], None], interval: int = 1, warmup: int = 1, first_step: int = 0):
        assert interval >= 1
        self.interval = interval
        self.graphs = []
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        n = first_step
        with torch.cuda.stream(side):
            for _ in range(warmup):
                step_fn(n)
                n += 1
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        for r in range(interval):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                step_fn(r)  # only the residue modulo interval matters to the launches
            self.graphs.append(g)
        torch.cuda.synchronize()
        self.next_step = n

    def replay(self, step_no: int | None = None) -> None:
        """Enqueue one step (the graph for step_no modulo interval) on the current stream."""
        if step_no is None:
            step_no = self.next_step
        self.graphs[step_no % self.interval].replay()
        self.next_step = step_no + 1
