"""Training steps on host-resident batches with the host<->device copies
hidden behind the kernels of neighbouring steps.

Each step copies its inputs (x, router logits, dOut) in from pinned host
memory and its results (out, dx, dlogits) back out.  Run naively the copies
sit between the steps; here they run on two copy streams while the compute
stream works on the neighbouring step:

* the inputs of step i+1 go into the second of two device input buffers
  while step i computes (they may start once step i-1, the previous reader
  of that buffer, has finished);
* the results of step i are first copied on the device into one of two
  staging buffers (a few microseconds), then to the host while step i+1
  computes; step i+2 waits for that host copy before it refills the buffer.

Every step still moves all of its own bytes across the host link; only their
placement in time changes.  The layer's calls are the same as in
`MoEExpertMLP.step`.
"""
from __future__ import annotations

import torch


class HostStepPipeline:
    def __init__(self, layer, device=None):
        self.layer = layer
        dev = torch.device(device) if device is not None else layer.w2.device
        T, E, d = max(layer.T, 1), layer.E, layer.d
        bf, f32 = torch.bfloat16, torch.float32
        self.inp = [dict(x=torch.empty((T, d), dtype=bf, device=dev),
                         logits=torch.empty((T, E), dtype=f32, device=dev),
                         dout=torch.empty((T, d), dtype=bf, device=dev)) for _ in range(2)]
        self.stage = [dict(out=torch.empty((T, d), dtype=bf, device=dev),
                           dx=torch.empty((T, d), dtype=bf, device=dev),
                           dlogits=torch.empty((T, E), dtype=f32, device=dev)) for _ in range(2)]
        self.h2d = torch.cuda.Stream(device=dev)
        self.d2h = torch.cuda.Stream(device=dev)

    def run(self, host_inputs, host_outputs, bias=None):
        """host_inputs: list of dicts {x, logits, dout} (pinned host tensors),
        one per step; host_outputs: list of dicts {out, dx, dlogits} (pinned
        host tensors), one per step (entries may repeat).  Enqueues every
        step on the current stream and returns; the caller synchronises."""
        layer = self.layer
        comp = torch.cuda.current_stream()
        n = len(host_inputs)
        if n == 0:
            return
        in_ready = [torch.cuda.Event() for _ in range(2)]
        step_done = [torch.cuda.Event() for _ in range(2)]
        out_copied = [torch.cuda.Event() for _ in range(2)]
        started = torch.cuda.Event()
        started.record(comp)

        def copy_in(i):
            b = i % 2
            with torch.cuda.stream(self.h2d):
                self.h2d.wait_event(started)
                if i >= 2:                       # step i-2 was the buffer's last reader
                    self.h2d.wait_event(step_done[b])
                for k in ("x", "logits", "dout"):
                    self.inp[b][k].copy_(host_inputs[i][k], non_blocking=True)
                in_ready[b].record(self.h2d)

        copy_in(0)
        for i in range(n):
            b = i % 2
            if i + 1 < n:
                copy_in(i + 1)
            comp.wait_event(in_ready[b])
            if i >= 2:                           # staging buffer b drained to the host
                comp.wait_event(out_copied[b])
            src = self.inp[b]
            layer.step(src["x"], src["logits"], bias, src["dout"])
            st = self.stage[b]
            st["out"].copy_(layer.out[:st["out"].shape[0]], non_blocking=True)
            st["dx"].copy_(layer.dx[:st["dx"].shape[0]], non_blocking=True)
            st["dlogits"].copy_(layer.dlogits[:st["dlogits"].shape[0]], non_blocking=True)
            step_done[b].record(comp)
            with torch.cuda.stream(self.d2h):
                self.d2h.wait_event(step_done[b])
                for k in ("out", "dx", "dlogits"):
                    host_outputs[i][k].copy_(st[k], non_blocking=True)
                out_copied[b].record(self.d2h)
        # the last results reach the host before the caller's next work
        comp.wait_event(out_copied[(n - 1) % 2])
        if n >= 2:
            comp.wait_event(out_copied[(n - 2) % 2])
