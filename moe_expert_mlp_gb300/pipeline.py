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


class GroupedHostStepPipeline:
    """Expert-MLP steps (groups given directly, no router) on host-resident
    batches: each step copies in its expert-ordered rows x_perm and their
    upstream gradient dY (both [capacity, d] in the library's padded row
    layout, padding rows zero) and the group sizes, runs the forward and
    backward of the expert MLP, and copies its per-row results Y and dX_perm
    back out.  The weight gradients stay in device memory, where the
    optimizer that consumes them runs.

    The layer alternates between two sets of per-row device buffers (inputs
    and results), so no device-side staging copy is needed: the inputs of
    step i+1 are copied into the other set while step i computes, and the
    results of step i go to the host while step i+1 computes; step i+2 waits
    for both before it reuses the set.
    """

    def __init__(self, layer, device=None):
        self.layer = layer
        dev = torch.device(device) if device is not None else layer.w2.device
        cap, d, E = layer.capacity, layer.d, layer.E
        bf = torch.bfloat16
        self.sets = [dict(x_perm=layer.x_perm, dy=layer.dy, y=layer.y, dx_perm=layer.dx_perm)]
        self.sets.append({k: torch.zeros((cap, d), dtype=bf, device=dev)
                          for k in ("x_perm", "dy", "y", "dx_perm")})
        self.counts = [torch.zeros(E, dtype=torch.int32, device=dev) for _ in range(2)]
        self.h2d = torch.cuda.Stream(device=dev)
        self.d2h = torch.cuda.Stream(device=dev)

    def run(self, host_inputs, host_outputs):
        """host_inputs: list of dicts {x_perm, dy, counts} (pinned host
        tensors: [capacity, d] bf16, [capacity, d] bf16, [E] int32), one per
        step; host_outputs: list of dicts {y, dx_perm} (pinned host tensors
        [capacity, d] bf16), one per step (entries may repeat).  Enqueues
        every step on the current stream and returns; the caller
        synchronises."""
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
                if i >= 2:                       # step i-2 was the set's last reader
                    self.h2d.wait_event(step_done[b])
                self.sets[b]["x_perm"].copy_(host_inputs[i]["x_perm"], non_blocking=True)
                self.sets[b]["dy"].copy_(host_inputs[i]["dy"], non_blocking=True)
                self.counts[b].copy_(host_inputs[i]["counts"], non_blocking=True)
                in_ready[b].record(self.h2d)

        copy_in(0)
        for i in range(n):
            b = i % 2
            if i + 1 < n:
                copy_in(i + 1)
            comp.wait_event(in_ready[b])
            if i >= 2:                           # results of step i-2 are on the host
                comp.wait_event(out_copied[b])
            s = self.sets[b]
            layer.grouped_step(counts=self.counts[b], x_perm=s["x_perm"], dy=s["dy"], y=s["y"],
                               dx_perm=s["dx_perm"])
            step_done[b].record(comp)
            with torch.cuda.stream(self.d2h):
                self.d2h.wait_event(step_done[b])
                host_outputs[i]["y"].copy_(s["y"], non_blocking=True)
                host_outputs[i]["dx_perm"].copy_(s["dx_perm"], non_blocking=True)
                out_copied[b].record(self.d2h)
        comp.wait_event(out_copied[(n - 1) % 2])
        if n >= 2:
            comp.wait_event(out_copied[(n - 2) % 2])
        # leave the layer on its own buffers
        s0 = self.sets[0]
        layer.x_perm, layer.dy, layer.y, layer.dx_perm = (s0["x_perm"], s0["dy"], s0["y"],
                                                          s0["dx_perm"])
