"""Host-to-host execution of a device step with copies overlapped.

A caller that starts from host memory and needs its results back on the host
(the end-to-end use of the library) pays two copies per batch besides the
GEMMs.  Issued in order on one stream they leave the copy engines and the
SMs idle in turn.  CopyComputePipeline keeps them busy together: the
host-to-device copies of batch i+1 run on one stream, the step on batch i on
the caller's stream, and the device-to-host copy of batch i-1 on a third
stream, with `depth` sets of device buffers and CUDA events ordering each
buffer's reuse.  Every batch's inputs are still copied in and its result
copied out; only their order in time changes.

The step itself is the library's (quantizers, GEMMs, MoE layer); this module
only orders copies and launches.
"""
from __future__ import annotations

from typing import Callable, Sequence

import torch


class CopyComputePipeline:
    """Run ``step(slot)`` over a stream of host batches.

    step(slot)    enqueues, on the current stream, the computation that reads
                  ``dev_inputs[slot]`` and writes ``dev_outputs[slot]``
    dev_inputs    per slot, the device tensors the host inputs are copied into
    dev_outputs   per slot, the device tensor copied back to the host

    submit(host_inputs, host_output) enqueues one batch (pinned host tensors
    for truly asynchronous copies); finish() makes the current stream wait for
    every copy back.  Nothing here synchronises the host.
    """

    def __init__(self, step: Callable[[int], None], dev_inputs: Sequence[Sequence[torch.Tensor]],
                 dev_outputs: Sequence[torch.Tensor]):
        if len(dev_inputs) != len(dev_outputs) or not dev_outputs:
            raise ValueError("one input set and one output per slot")
        self.step = step
        self.din = [list(d) for d in dev_inputs]
        self.dout = list(dev_outputs)
        self.depth = len(self.dout)
        self.s_in = torch.cuda.Stream()
        self.s_out = torch.cuda.Stream()
        self.in_done = [torch.cuda.Event() for _ in range(self.depth)]
        self.compute_done = [torch.cuda.Event() for _ in range(self.depth)]
        self.out_done = [torch.cuda.Event() for _ in range(self.depth)]
        self.used = [False] * self.depth
        self.i = 0

    def submit(self, host_inputs: Sequence[torch.Tensor], host_output: torch.Tensor) -> None:
        s = self.i % self.depth
        compute = torch.cuda.current_stream()
        with torch.cuda.stream(self.s_in):
            if self.used[s]:
                self.s_in.wait_event(self.compute_done[s])      # slot s's inputs consumed
            for h, d in zip(host_inputs, self.din[s]):
                d.copy_(h, non_blocking=True)
            self.in_done[s].record(self.s_in)
        compute.wait_event(self.in_done[s])
        if self.used[s]:
            compute.wait_event(self.out_done[s])                # slot s's output read back
        self.step(s)
        self.compute_done[s].record(compute)
        with torch.cuda.stream(self.s_out):
            self.s_out.wait_event(self.compute_done[s])
            host_output.copy_(self.dout[s], non_blocking=True)
            self.out_done[s].record(self.s_out)
        self.used[s] = True
        self.i += 1

    def finish(self) -> None:
        torch.cuda.current_stream().wait_stream(self.s_out)
