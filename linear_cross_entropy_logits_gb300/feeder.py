"""Double-buffered host-to-device input feeding for a training loop around the fused op.

A step's token rows and targets live in pinned host memory. The feeder copies step k+1's
inputs into the second of two device buffer sets on a dedicated copy stream while step k
runs on the compute stream. CUDA events order the two streams:

  * ready[slot]: recorded on the copy stream after the slot's copies; the compute stream
    waits on it before the step that reads the slot;
  * free[slot]: recorded on the compute stream after the step that read the slot; the copy
    stream waits on it before overwriting the slot.

Only torch streams, events and copies are used here (plumbing); every step of the op runs
in the library's kernels.
"""

from __future__ import annotations

import torch


class DoubleBufferedInputs:
    """Two device copies of a dict of host tensors, refilled on a copy stream."""

    def __init__(self, host_like: dict, device, copy_stream: torch.cuda.Stream | None = None):
        self.device = torch.device(device)
        self.copy_stream = copy_stream or torch.cuda.Stream(self.device)
        self.slots = [{k: torch.empty_like(v, device=self.device) for k, v in host_like.items()}
                      for _ in range(2)]
        self.ready = [torch.cuda.Event() for _ in range(2)]
        self.free = [None, None]
        self.h2d_bytes = sum(v.numel() * v.element_size() for v in host_like.values())
        self._next = 0

    def stage(self, host: dict, after: torch.cuda.Event | None = None) -> int:
        """Enqueue the copies of `host` (pinned CPU tensors) into the next slot; returns the
        slot. `after` (optional) is an event the copies must also wait for."""
        slot = self._next
        self._next ^= 1
        with torch.cuda.stream(self.copy_stream):
            if after is not None:
                self.copy_stream.wait_event(after)
            if self.free[slot] is not None:
                self.copy_stream.wait_event(self.free[slot])
            dst = self.slots[slot]
            for k, v in host.items():
                dst[k].copy_(v, non_blocking=True)
            self.ready[slot].record(self.copy_stream)
        return slot

    def acquire(self, slot: int, stream: torch.cuda.Stream) -> dict:
        """Make `stream` wait for the slot's copies; returns its device tensors."""
        stream.wait_event(self.ready[slot])
        return self.slots[slot]

    def release(self, slot: int, stream: torch.cuda.Stream) -> None:
        """Mark the slot reusable once the work enqueued so far on `stream` is done."""
        ev = torch.cuda.Event()
        ev.record(stream)
        self.free[slot] = ev
