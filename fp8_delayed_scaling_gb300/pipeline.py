"""HostStepPipeline: training steps over host-resident inputs and outputs, with the
host<->device copies taken off the compute stream.

A step reads device input tensors (X, dY, ...) and writes device outputs (weight
and bias gradients, dx, ...).  When the data lives in pinned host memory, each
step needs an H2D copy of its inputs and a D2H copy of its results.  Issued in
order on one stream, those copies add to every step's time.  Here they run on
two copy streams beside the compute stream:

    h2d stream      copy inputs(i+1) -> set (i+1)%2   (after step i-1 read that set)
    compute stream  step(i) on set i%2; snapshot outputs -> stage i%2 (device copy)
    d2h stream      stage i%2 -> host outputs(i)      (after the snapshot)

Events order every reuse: an input set is refilled only after the step that read
it has run, and a snapshot stage is rewritten only after its D2H has finished.
The snapshot is a device-to-device copy of the outputs (HBM speed), so the next
step may overwrite the outputs while their host copy is still in flight.

With two output sets (out_sets) there is no snapshot: step i writes output set
i%2 directly (the step function receives it), its D2H reads that set, and step
i+2 waits for that D2H before it writes the set again.
"""
from __future__ import annotations

from typing import Callable, Sequence

import torch


class HostStepPipeline:
    """dev_inputs: the device tensors a step reads; a second set of the same shapes is
    allocated for double buffering.  dev_outputs: the device tensors a step writes.
    out_sets=True: a second set of outputs is allocated too, and the step function is
    called as step(inputs, outputs) with the set to write (no snapshot copies)."""

    def __init__(self, dev_inputs: Sequence[torch.Tensor], dev_outputs: Sequence[torch.Tensor],
                 out_sets: bool = False):
        dev = dev_inputs[0].device
        self.sets = [list(dev_inputs), [torch.empty_like(t) for t in dev_inputs]]
        self.direct = out_sets
        self.outputs = list(dev_outputs)
        if out_sets:
            self.out_sets = [list(dev_outputs), [torch.empty_like(t) for t in dev_outputs]]
            self.stage = self.out_sets
        else:
            self.stage = [[torch.empty_like(t) for t in dev_outputs] for _ in range(2)]
        self.h2d = torch.cuda.Stream(dev)
        self.d2h = torch.cuda.Stream(dev)
        ev = lambda: [torch.cuda.Event(), torch.cuda.Event()]  # noqa: E731
        self.in_ready, self.in_free, self.staged, self.out_done = ev(), ev(), ev(), ev()

    @staticmethod
    def _copy(dst: Sequence[torch.Tensor], src: Sequence[torch.Tensor]) -> None:
        assert len(dst) == len(src)
        for d, s in zip(dst, src):
            d.copy_(s, non_blocking=True)

    def run(self, n_steps: int, step: Callable[[list], None], host_inputs: Callable[[int], Sequence[torch.Tensor]],
            host_outputs: Callable[[int], Sequence[torch.Tensor]]) -> None:
        """Run n_steps steps.  step(inputs) (or step(inputs, outputs) with out_sets) enqueues one
        step on the current stream reading the device tensors `inputs`; host_inputs(i) gives
        step i's pinned host inputs and host_outputs(i) the pinned host tensors that receive
        its outputs.  Returns when every copy has been enqueued; the caller synchronises."""
        compute = torch.cuda.current_stream()
        self.h2d.wait_stream(compute)
        self.d2h.wait_stream(compute)
        with torch.cuda.stream(self.h2d):
            self._copy(self.sets[0], host_inputs(0))
            self.in_ready[0].record(self.h2d)
        for i in range(n_steps):
            b = i % 2
            if i + 1 < n_steps:
                with torch.cuda.stream(self.h2d):
                    if i >= 1:
                        self.h2d.wait_event(self.in_free[1 - b])  # step i-1 has read set 1-b
                    self._copy(self.sets[1 - b], host_inputs(i + 1))
                    self.in_ready[1 - b].record(self.h2d)
            compute.wait_event(self.in_ready[b])
            if self.direct:
                if i >= 2:
                    compute.wait_event(self.out_done[b])  # the D2H of step i-2 has left output set b
                step(self.sets[b], self.out_sets[b])
                self.in_free[b].record(compute)
            else:
                step(self.sets[b])
                self.in_free[b].record(compute)
                if i >= 2:
                    compute.wait_event(self.out_done[b])  # the D2H of step i-2 has left stage b
                self._copy(self.stage[b], self.outputs)
            self.staged[b].record(compute)
            with torch.cuda.stream(self.d2h):
                self.d2h.wait_event(self.staged[b])
                self._copy(host_outputs(i), self.stage[b])
                self.out_done[b].record(self.d2h)
        compute.wait_stream(self.h2d)
        compute.wait_stream(self.d2h)
