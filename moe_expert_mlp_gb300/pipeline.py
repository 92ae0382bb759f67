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
        bf, f32 = layer.act_dtype, torch.float32
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
    batches: each step copies in its expert-ordered rows x and their
    upstream gradient dY (both [R, d] bf16, the R real rows only, group after
    group) and the group sizes, runs the forward and backward of the expert
    MLP, and copies its per-row results Y and dX (again the R real rows)
    back out.  The weight gradients stay in device memory, where the
    optimizer that consumes them runs.

    Rows move group by group between the host's dense row order and the
    library's padded device layout (each group starting at a multiple of 128
    rows), so no padding row crosses the host link; padding rows of the
    device buffers are kept zero (they are cleared whenever the group sizes,
    and with them the layout, change).  The layer cycles through `depth`
    sets of per-row device buffers (default two), so no device-side staging
    copy is needed: the inputs of the next depth-1 steps stream in while a
    step computes, and each step's results go to the host while the
    following steps compute; step i+depth waits for both before it reuses
    step i's set.  (Where the host link, not the kernels, sets the pace, a
    third set does not shorten the step: both directions are already busy
    all the time.)
    """

    def __init__(self, layer, device=None, depth=2):
        if depth < 2:
            raise ValueError("depth must be at least 2")
        self.layer = layer
        dev = torch.device(device) if device is not None else layer.w2.device
        cap, d, E = layer.capacity, layer.d, layer.E
        bf = layer.act_dtype
        self.depth = depth
        self.sets = [dict(x_perm=layer.x_perm, dy=layer.dy, y=layer.y, dx_perm=layer.dx_perm)]
        for _ in range(depth - 1):
            self.sets.append({k: torch.zeros((cap, d), dtype=bf, device=dev)
                              for k in ("x_perm", "dy", "y", "dx_perm")})
        self.layout = [None] * depth             # group sizes each set was last laid out for
        self.counts = [torch.zeros(E, dtype=torch.int32, device=dev) for _ in range(depth)]
        self.h2d = torch.cuda.Stream(device=dev)
        self.d2h = torch.cuda.Stream(device=dev)

    @staticmethod
    def _segments(counts):
        """(host row, device row, rows) of every non-empty group."""
        segs, src, dst = [], 0, 0
        for m in (int(c) for c in counts):
            if m > 0:
                segs.append((src, dst, m))
            src += m
            dst += (m + 127) // 128 * 128
        return segs

    def run(self, host_inputs, host_outputs):
        """host_inputs: list of dicts {x, dy, counts} (x, dy: pinned host
        tensors [R, d] bf16 in group order; counts: host int32 tensor [E]
        with sum R), one per step; host_outputs: list of dicts {y, dx}
        (pinned host tensors [R, d] bf16), one per step (entries may
        repeat).  Enqueues every step on the current stream and returns; the
        caller synchronises."""
        layer = self.layer
        comp = torch.cuda.current_stream()
        n = len(host_inputs)
        if n == 0:
            return
        D = self.depth
        in_ready = [torch.cuda.Event() for _ in range(D)]
        step_done = [torch.cuda.Event() for _ in range(D)]
        out_copied = [torch.cuda.Event() for _ in range(D)]
        started = torch.cuda.Event()
        started.record(comp)
        segs = [None] * n

        def copy_in(i):
            b = i % D
            hin = host_inputs[i]
            key = tuple(int(c) for c in hin["counts"])
            segs[i] = self._segments(key)
            dev = self.sets[b]
            with torch.cuda.stream(self.h2d):
                self.h2d.wait_event(started)
                if i >= D:                       # step i-D was the set's last reader
                    self.h2d.wait_event(step_done[b])
                if self.layout[b] != key:        # new layout: padding rows back to zero
                    dev["x_perm"].zero_()
                    dev["dy"].zero_()
                    self.layout[b] = key
                for src, dst, m in segs[i]:
                    dev["x_perm"][dst:dst + m].copy_(hin["x"][src:src + m], non_blocking=True)
                    dev["dy"][dst:dst + m].copy_(hin["dy"][src:src + m], non_blocking=True)
                self.counts[b].copy_(hin["counts"], non_blocking=True)
                in_ready[b].record(self.h2d)

        for i in range(min(D - 1, n)):
            copy_in(i)
        for i in range(n):
            b = i % D
            if i + D - 1 < n:
                copy_in(i + D - 1)
            comp.wait_event(in_ready[b])
            if i >= D:                           # results of step i-D are on the host
                comp.wait_event(out_copied[b])
            s = self.sets[b]
            layer.grouped_step(counts=self.counts[b], x_perm=s["x_perm"], dy=s["dy"], y=s["y"],
                               dx_perm=s["dx_perm"])
            step_done[b].record(comp)
            with torch.cuda.stream(self.d2h):
                self.d2h.wait_event(step_done[b])
                hout = host_outputs[i]
                for src, dst, m in segs[i]:
                    hout["y"][src:src + m].copy_(s["y"][dst:dst + m], non_blocking=True)
                    hout["dx"][src:src + m].copy_(s["dx_perm"][dst:dst + m], non_blocking=True)
                out_copied[b].record(self.d2h)
        for i in range(max(0, n - D), n):
            comp.wait_event(out_copied[i % D])
        # leave the layer on its own buffers
        s0 = self.sets[0]
        layer.x_perm, layer.dy, layer.y, layer.dx_perm = (s0["x_perm"], s0["dy"], s0["y"],
                                                          s0["dx_perm"])
