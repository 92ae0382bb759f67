#!/usr/bin/env python3
"""Benchmark: one routed-expert MLP layer, forward + backward, on GB300.

A step is one whole pass of the hot path over one batch of synthetic input:
routing + permute -> FC1 grouped GEMM with the GLU epilogue -> FC2 grouped
GEMM -> weighted combine -> combine backward -> FC2 dgrad with the dGLU
epilogue -> FC2 wgrad -> FC1 dgrad -> FC1 wgrad -> permute backward ->
router backward.  For layers whose groups are given directly (no router) the
step is the expert MLP alone: the activation quantizations and the six
grouped GEMMs.  Default workload: the DeepSeek-V3-shaped local experts,
16384 routed rows over 32 experts with Zipf(1.2) group sizes (4 empty),
d=7168, F=2048, SwiGLU, MXFP8 GEMM operands (E4M3 with an E8M0 scale per 32
elements).

The K timed steps are captured in one CUDA graph (no host synchronisation
inside) with timing events around the dominant GEMM's calls only, replayed
once between a barrier + synchronize on both sides; a second capture of the
same steps with events around every library call, replayed before the timed
region, gives the per-call breakdown.  value = algorithmic TFLOPS (18*d*F
per routed row, padding not counted) of the whole job.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload NAME] [--dtype bf16|mxfp8|nvfp4|fp32]

The JSON line also carries: `roofline` (the GEMM with the largest time,
against the roof that bounds it: its FLOPs over the measured tensor peak of
its operand type or its algorithmic bytes over the measured HBM bandwidth,
whichever takes longer, with both fractions given and the DRAM traffic of an
ncu capture of the same kernel source), `attainable` (the whole step against
max(FLOP / peak, algorithmic bytes / measured HBM bandwidth)), `e2e` (the
same steps through the public API with host-resident inputs and results,
copies overlapped by HostStepPipeline, and in line), `cpu_baseline` (the
oracle on a bounded sample on the host cores), `clocks` (sampled during the
timed region), per-call times in `kernels`, and the fused-vs-unfused,
overlap and router measurements unless switched off.

--impl reference times the CPU fp64 oracle (the method written out plainly)
on a bounded sample of the same workload on the host cores.
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

from workloads import WORKLOADS, bf16_bits_to_f64, make_inputs  # noqa: E402

METRIC = "MoE expert-MLP fwd+bwd TFLOPS & tokens/s on 1 GB300; % of tensor-core peak"
DEFAULT_WORKLOAD = "dsv3_r16384_e32"
DEFAULT_DTYPE = "mxfp8"
PEAKS_FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}

# DRAM bytes (read + write) per launch of each grouped GEMM, from one ncu
# capture per workload and operand type (summaries under profiles/), with the
# hash of the GEMM sources the counters were taken on; a changed kernel
# reports null.
_NCU_SRC = "9ee4fad3d5167224"
NCU_TRAFFIC = {
    # FC1 weight gradient of the default layer: full-layer one-pass capture
    ("fc1_wgrad", "dsv3_r16384_e32", "mxfp8"): {"bytes": 261881344.0 + 1823199232.0,
                                                 "src": _NCU_SRC},
}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return dict(PEAKS_FALLBACK), "fallback"


def gemm_source_hash():
    h = hashlib.sha256()
    for fn in ("moe_gemm.cu", "moe_ptx.cuh", "moe_internal.h", "moe_mx.cuh", "moe_act.cuh"):
        with open(os.path.join(ROOT, "moe_expert_mlp_gb300", "csrc", fn), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


# --------------------------------------------------------------- per-call work
def call_work(wl, name, R, dtype="bf16"):
    """Algorithmic FLOPs or bytes of one library call over R real routed rows.
    GEMMs: 2*M*N*K with M = routed rows.  Memory-bound calls: bytes of the
    tensors they must read and write once (bf16 rows, fp32 on the fp32 path;
    index arrays ignored)."""
    d, F, T, k = wl.d, wl.F, wl.T, wl.k
    n1 = 2 * F if wl.gated else F          # FC1 outputs (gate + linear halves when gated)
    gemm = {
        "fc1_glu_fwd": 2.0 * R * d * n1,
        "fc2_fwd": 2.0 * R * F * d,
        "fc2_dgrad_dglu": 2.0 * R * d * F,
        "fc2_wgrad": 2.0 * R * d * F,
        "fc1_dgrad": 2.0 * R * n1 * d,
        "fc1_wgrad": 2.0 * R * n1 * d,
    }
    if name in gemm:
        return "flop", gemm[name]
    mem = {
        "route_permute": T * wl.E * 4 + T * d * 2 + R * d * 2,
        "combine": R * d * 2 + T * d * 2,
        "combine_bwd": T * d * 2 + R * d * 2 + R * d * 2,
        "permute_bwd": R * d * 2 + T * d * 2,
        "route_bwd": T * k * 12 + T * wl.E * 4,
        "bias_grads": R * d * 2 * int(wl.has_b2) + R * n1 * 2 * int(wl.has_b1),
        # bf16 rows in; rowwise and transposed E4M3 codes + one scale per 32 out
        "quant_x": R * d * (2 + 2 + 2 / 32),
        "quant_dy": R * d * (2 + 2 + 2 / 32),
    }
    if dtype == "mxfp8" and wl.router != "direct":
        # routed MXFP8 layers: the permutation and the combine backward also
        # write the rowwise copies of x_perm / dY; the passes only the
        # transposed copies
        q = 1 + 1 / 32
        mem.update(route_permute=mem["route_permute"] + R * d * q,
                   combine_bwd=mem["combine_bwd"] + R * d * q,
                   quant_x=R * d * (2 + q), quant_dy=R * d * (2 + q))
    if dtype == "fp32":
        # fp32 rows (twice the bytes); the transposes of x_perm and dY read
        # and write them once
        mem = {key: 2.0 * v for key, v in mem.items() if key not in ("quant_x", "quant_dy")}
        mem.update(route_permute=T * wl.E * 4 + T * d * 4 + R * d * 4, route_bwd=T * k * 12 + T * wl.E * 4,
                   transpose_x=R * d * 8, transpose_dy=R * d * 8)
    if dtype == "nvfp4":
        # bf16 rows in; rowwise and rotated transposed E2M1 codes (half a
        # byte each) + one scale per 16 out; x and dY also read once for amax
        mem.update(quant_x=R * d * (2 + 2 + 1 + 2 / 16), quant_dy=R * d * (2 + 2 + 1 + 2 / 16),
                   quant_a=R * F * (2 + 1 + 2 / 16), quant_dh=R * n1 * (2 + 1 + 2 / 16))
    return "byte", float(mem.get(name, 0.0))


def gemm_bytes(wl, name, R, dtype="bf16", keep_bf16=False):
    """Algorithmic HBM bytes of one grouped GEMM call: its operands read once
    and its outputs written once (R real rows; padding ignored).  Operands
    are bf16 (2 bytes), fp32 (4) or MXFP8 codes with a scale per 32
    (1 + 1/32); the transposed copies the backward reads are the same size.
    Outputs: H, Y, dX and dW in bf16 (fp32 on the fp32 path); A and dH as
    their two MXFP8 copies on the MXFP8 path (plus the bf16 tensor when
    keep_bf16), in bf16 otherwise (NVFP4: bf16, quantized by later passes),
    with the fp32 path's transposed A and dH counted too."""
    d, F, E = wl.d, wl.F, wl.E
    n1 = 2 * F if wl.gated else F
    q = {"bf16": 2.0, "mxfp8": 1.0 + 1.0 / 32, "nvfp4": 0.5 + 1.0 / 16, "fp32": 4.0}[dtype]
    o = 4.0 if dtype == "fp32" else 2.0                    # stored bf16 / fp32 element
    if dtype == "mxfp8":
        act_out = 2 * q + (2.0 if keep_bf16 else 0.0)      # rowwise + transposed copies
    elif dtype == "nvfp4":
        act_out = 2.0            # bf16 (its NVFP4 copies come from separate passes)
    else:
        act_out = 2 * o if dtype == "fp32" else o          # fp32: plus the transposed copy
    b = {
        "fc1_glu_fwd": R * d * q + E * n1 * d * q + R * n1 * o + R * F * act_out,
        "fc2_fwd": R * F * q + E * d * F * q + R * d * o,
        "fc2_dgrad_dglu": R * d * q + E * d * F * q + R * n1 * o + R * n1 * act_out,
        "fc2_wgrad": R * d * q + R * F * q + E * d * F * o,
        "fc1_dgrad": R * n1 * q + E * n1 * d * q + R * d * o,
        "fc1_wgrad": R * n1 * q + R * d * q + E * n1 * d * o,
    }
    return float(b[name])


def step_bytes(wl, dtype="bf16"):
    """Algorithmic HBM bytes of one fwd+bwd step (the attainable-roofline
    byte model): every weight read once per GEMM that uses it (the bf16
    masters, or the quantized copies on the block-scaled paths, whose
    preparation runs outside the step), every dW written once in bf16, every
    per-row tensor written once and read once per consumer (x_perm by FC1 and
    FC1 wgrad, H by the dGLU, A by FC2 and FC2 wgrad, Y by the combine, dY
    by FC2 dgrad and FC2 wgrad, dH by FC1 dgrad and FC1 wgrad, dX_perm by the
    permute backward); on the block-scaled paths each quantized operand copy
    is written once and read by its GEMM, after one bf16 read of its source
    (two for x_perm / dY on NVFP4: the amax pass); routed layers add the
    token-side x, out, dOut, dx.  Padding rows and index arrays are ignored."""
    d, F, E = wl.d, wl.F, wl.E
    n1 = 2 * F if wl.gated else F
    R = wl.routed_rows
    w_el = E * (n1 * d + d * F)
    q = {"bf16": 2.0, "mxfp8": 1.0 + 1.0 / 32, "nvfp4": 0.5 + 1.0 / 16, "fp32": 4.0}[dtype]
    b = 2.0 * w_el * (2.0 if dtype == "bf16" else q)      # two GEMMs per weight
    b += (4.0 if dtype == "fp32" else 2.0) * w_el         # dW in bf16 (fp32)
    if dtype == "fp32":
        # every weight-gradient GEMM reads transposed copies: x_perm and dY
        # transposed by a pass (read + write), A^T and dH^T written by their
        # epilogues; the transposed weights are made outside the step
        per_row = 4 * (5 * d        # x_perm: written, FC1, transpose; x^T written, FC1 wgrad
                       + 2 * n1     # H: FC1 writes, dGLU reads
                       + 4 * F      # A and A^T: written, read by FC2 / FC2 wgrad
                       + 2 * d      # Y
                       + 5 * d      # dY: written, FC2 dgrad, transpose; dY^T written, wgrad
                       + 4 * n1     # dH and dH^T: written, read by FC1 dgrad / FC1 wgrad
                       + 2 * d)     # dX_perm
    elif dtype == "bf16":
        per_row = 2 * (3 * d        # x_perm: written (permute or input), FC1, FC1 wgrad
                       + 2 * n1     # H: FC1 writes, dGLU reads
                       + 3 * F      # A: FC1 writes, FC2 and FC2 wgrad read
                       + 2 * d      # Y: FC2 writes, combine reads
                       + 3 * d      # dY: combine bwd writes, FC2 dgrad and wgrad read
                       + 3 * n1     # dH: dGLU writes, FC1 dgrad and wgrad read
                       + 2 * d)     # dX_perm: FC1 dgrad writes, permute bwd reads
    else:
        amax_reads = 2 if dtype == "nvfp4" else 1
        per_row = (2 * d + 2 * d * amax_reads + 4 * d * q          # x_perm + its two copies
                   + 2 * 2 * n1                                    # H written, read by dGLU
                   + 2 * F + 2 * F + 4 * F * q                     # A (bf16) + its copies
                   + 2 * 2 * d                                     # Y
                   + 2 * d + 2 * d * amax_reads + 4 * d * q        # dY + its copies
                   + 2 * n1 + 2 * n1 + 4 * n1 * q                  # dH + its copies
                   + 2 * 2 * d)                                    # dX_perm
    b += R * per_row
    if wl.router != "direct":
        b += wl.T * 4 * d * (4 if dtype == "fp32" else 2) + wl.T * wl.E * 4 * 2   # x, out, dOut, dx; logits
    return float(b)


# ------------------------------------------------------------ multi-rank
def max_over_ranks(value, dist, device):
    """Largest value over all ranks (the slowest replica sets the job time)."""
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(work_per_step, steps, world, ms_max):
    """Whole-job rate: the work of every rank's steps over the slowest time."""
    return work_per_step * steps * world / (ms_max * 1e-3)


# ------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi clock / throttle sampling while the GPU works."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id):
        self.path = tempfile.mktemp(prefix="moe_clocks_", suffix=".csv")
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
               "-lms", "100"]
        if gpu_id is not None:
            cmd += ["-i", gpu_id]
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(cmd, stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        sm, smax, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 8:
                    continue
                try:
                    sm.append(float(parts[0]))
                    smax.append(float(parts[1]))
                    power.append(float(parts[2]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[4:8]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "power_w_max": max(power) if power else None, "samples": len(sm),
                "reasons": sorted(reasons)}


def gpu_uuid(torch, dev):
    try:
        u = str(torch.cuda.get_device_properties(dev).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        return None


# ------------------------------------------------------------ oracle timing
def _oracle_routed_mx(oracle, x, logits, bias, dout, W1, b1, W2, b2, k, p):
    """The routed layer with the MXFP8 expert MLP (routing, combine and their
    backward as in the bf16 oracle; dY rounded to the stored bf16)."""
    E = W1.shape[0]
    topk_idx, topk_w, counts = oracle.route(logits, bias, k)
    _, padded, _ = oracle.group_offsets(counts, 128)
    row_src, row_of = oracle.permute_index(topk_idx, E, padded)
    xp = oracle.gather_rows(x, row_src)
    Hh, A, Y = oracle.grouped_forward_mx(xp, padded, counts, W1, b1, W2, b2, p)
    oracle.combine(Y, row_of, topk_w)
    dY, dw = oracle.combine_backward(dout, Y, row_of, topk_w, xp.shape[0])
    dX = oracle.grouped_backward_mx(xp, Hh, A, oracle.bf16_round(dY), padded, counts, W1, W2,
                                    p)[0]
    oracle.permute_backward(dX, row_of)
    oracle.route_backward(dw, topk_w, topk_idx, E)


def _oracle_routed_nv(oracle, x, logits, bias, dout, W1, b1, W2, b2, k, p):
    """The routed layer with the NVFP4 expert MLP (routing and combine as in
    the bf16 oracle; dY rounded to the stored bf16)."""
    E = W1.shape[0]
    topk_idx, topk_w, counts = oracle.route(logits, bias, k)
    _, padded, _ = oracle.group_offsets(counts, 128)
    row_src, row_of = oracle.permute_index(topk_idx, E, padded)
    xp = oracle.gather_rows(x, row_src)
    Hh, A, Y = oracle.grouped_forward_nv(xp, padded, counts, W1, b1, W2, b2, p)
    oracle.combine(Y, row_of, topk_w)
    dY, dw = oracle.combine_backward(dout, Y, row_of, topk_w, xp.shape[0])
    dX = oracle.grouped_backward_nv(xp, Hh, A, oracle.bf16_round(dY), padded, counts, W1, W2,
                                    p)[0]
    oracle.permute_backward(dX, row_of)
    oracle.route_backward(dw, topk_w, topk_idx, E)


def oracle_sample_run(wl, inp, n_tokens, fmt="bf16"):
    """Time the CPU oracle (its MXFP8 / NVFP4 variant for fmt "mxfp8" /
    "nvfp4") on the first n_tokens
    tokens (routed workloads) or on the first experts holding about n_tokens
    rows (direct workloads).  Returns (seconds, flops of the sample,
    description)."""
    import oracle
    p = oracle.GluParams(wl.act, wl.alpha, wl.limit, wl.linear_offset, wl.out_scale)
    W1 = bf16_bits_to_f64(inp["w1"])
    W2 = bf16_bits_to_f64(inp["w2"])
    b1 = bf16_bits_to_f64(inp["b1"]) if inp["b1"] is not None else None
    b2 = bf16_bits_to_f64(inp["b2"]) if inp["b2"] is not None else None
    if wl.router != "direct":
        n = min(n_tokens, wl.T)
        x = bf16_bits_to_f64(inp["x"][:n])
        dout = bf16_bits_to_f64(inp["dout"][:n])
        t0 = time.perf_counter()
        if fmt in ("mxfp8", "nvfp4"):
            run = _oracle_routed_mx if fmt == "mxfp8" else _oracle_routed_nv
            run(oracle, x, inp["logits"][:n], inp["bias"], dout, W1, b1, W2, b2, wl.k, p)
        else:
            fwd = oracle.moe_forward(x, inp["logits"][:n], inp["bias"], W1, b1, W2, b2, wl.k, p)
            oracle.moe_backward(fwd, dout, W1, W2, p)
        dt = time.perf_counter() - t0
        rows = n * wl.k
        desc = f"first {n} of {wl.T} tokens ({rows} routed rows), full fwd+bwd"
    else:
        sizes = inp["group_sizes"]
        keep = np.zeros_like(sizes)
        acc = 0
        for e in np.argsort(sizes):
            if sizes[e] == 0:
                continue
            if acc + sizes[e] > max(n_tokens, 1) and acc > 0:
                break
            keep[e] = sizes[e]
            acc += sizes[e]
        offsets, padded, _ = oracle.group_offsets(keep, align=128)
        xr = np.zeros((int(padded[-1]), wl.d))
        dyr = np.zeros((int(padded[-1]), wl.d))
        src_off = np.concatenate([[0], np.cumsum(sizes)])
        for e in range(wl.E):
            if keep[e]:
                lo = int(padded[e])
                xr[lo:lo + keep[e]] = bf16_bits_to_f64(inp["x"][src_off[e]:src_off[e] + keep[e]])
                dyr[lo:lo + keep[e]] = bf16_bits_to_f64(inp["dout"][src_off[e]:src_off[e] + keep[e]])
        t0 = time.perf_counter()
        if fmt == "mxfp8":
            Hh, A, Y = oracle.grouped_forward_mx(xr, padded, keep, W1, b1, W2, b2, p)
            oracle.grouped_backward_mx(xr, Hh, A, dyr, padded, keep, W1, W2, p)
        elif fmt == "nvfp4":
            Hh, A, Y = oracle.grouped_forward_nv(xr, padded, keep, W1, b1, W2, b2, p)
            oracle.grouped_backward_nv(xr, Hh, A, dyr, padded, keep, W1, W2, p)
        else:
            Hh, A, Y = oracle.grouped_forward(xr, padded, keep, W1, b1, W2, b2, p)
            oracle.grouped_backward(xr, Hh, A, dyr, padded, keep, W1, W2, p)
        dt = time.perf_counter() - t0
        rows = int(acc)
        desc = f"{int((keep > 0).sum())} smallest experts ({rows} of {wl.R} rows), fwd+bwd"
    flops = (18 if wl.gated else 12) * wl.d * wl.F * rows
    return dt, float(flops), desc


def run_reference(args, wl):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    inp = make_inputs(wl)
    n_tok = args.ref_sample_tokens
    for _ in range(max(args.warmup, 0)):
        oracle_sample_run(wl, inp, n_tok, args.dtype)
    times = []
    flops = 0.0
    desc = ""
    for _ in range(args.steps):
        dt, flops, desc = oracle_sample_run(wl, inp, n_tok, args.dtype)
        times.append(dt)
    total = sum(times)
    value = flops * args.steps / total / 1e12
    cores = host_cores()
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOPS",
        "n_gpus": 0, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * total / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(wl, args.dtype),
        "cpu_baseline": {"value": value, "unit": "TFLOPS", "cores": cores, "kind": "oracle",
                         "sample": "each step: " + desc},
        "e2e": {"value": value, "unit": "TFLOPS", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


def workload_config(wl, dtype="bf16"):
    cfg = {"workload": wl.name, "E": wl.E, "d": wl.d, "F": wl.F, "act": wl.act,
           "routed_rows": wl.routed_rows, "gemm_operands": dtype}
    if wl.router != "direct":
        cfg.update({"T": wl.T, "k": wl.k, "router_bias": wl.router_bias})
    else:
        cfg.update({"groups": "zipf s=%.1f, %d empty" % (wl.zipf_s, wl.zipf_empty)
                    if wl.E > 1 else "one group"})
    if wl.limit != float("inf"):
        cfg.update({"limit": wl.limit, "alpha": wl.alpha, "linear_offset": wl.linear_offset})
    cfg["bias"] = bool(wl.has_b1 or wl.has_b2)
    cfg["l2"] = "no flush: working set (weights + activations) far above the 129 MB L2"
    return cfg


# --------------------------------------------------------------- GPU bench
def run_quantize_only(args, wl):
    """The MXFP8 activation quantizer alone (rowwise + transposed, scales in
    the MMA layout) on a [routed rows, d] bf16 tensor of the workload: a
    small-memory command for kernel profiles.  Prints one JSON line with the
    kernel's CUDA-event time and its algorithmic bytes over that time."""
    import torch
    import __graft_entry__
    __graft_entry__.build()
    from moe_expert_mlp_gb300 import _lib as L
    rows, cols = wl.routed_rows, wl.d
    torch.manual_seed(0)
    x = torch.randn(rows, cols, device="cuda").to(torch.bfloat16)
    u8 = dict(dtype=torch.uint8, device="cuda")
    out = dict(q=torch.empty((rows, cols), **u8),
               scale=torch.empty(L.moe_mx_scale_bytes(rows, cols), **u8),
               qt=torch.empty((cols, rows), **u8),
               scale_t=torch.empty(L.moe_mx_scale_bytes(cols, rows), **u8), layout="mma")
    for _ in range(args.warmup):
        L.moe_quantize_mx_bf16(x, 1, rows, cols, out)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        L.moe_quantize_mx_bf16(x, 1, rows, cols, out)
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / max(args.steps, 1)
    nbytes = rows * cols * 2 + 2 * rows * cols * (1 + 1 / 32)   # bf16 in; codes + scales twice
    print(json.dumps({"kernel": "mx_quantize", "rows": rows, "cols": cols, "ms": round(ms, 5),
                      "gbs": round(nbytes / (ms * 1e-3) / 1e9, 1), "steps": args.steps,
                      "warmup": args.warmup, "l2": "no flush: input and outputs far above L2"}))
    return 0


def run_ours(args, wl):
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    import __graft_entry__
    __graft_entry__.build()
    from moe_expert_mlp_gb300 import MoEExpertMLP, moe_read_device_status

    def bits_to_dev(bits, device):
        t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)
        return t.float() if args.dtype == "fp32" else t    # fp32 layer: the same values in fp32

    inp = make_inputs(wl)
    routed = wl.router != "direct"
    cap = None
    if not routed:
        sizes = inp["group_sizes"]
        cap = int(sum((int(m) + 127) // 128 * 128 for m in sizes))
        cap = max(cap, 128)
    layer = MoEExpertMLP(wl.E, wl.d, wl.F, T=wl.T if routed else 0, k=wl.k, act=wl.act,
                         alpha=wl.alpha, limit=wl.limit, linear_offset=wl.linear_offset,
                         out_scale=wl.out_scale, has_b1=wl.has_b1, has_b2=wl.has_b2,
                         capacity=cap, device=dev, dtype=args.dtype)
    mx = args.dtype in ("mxfp8", "nvfp4")      # block-scaled operands
    w1 = bits_to_dev(inp["w1"], dev)
    w2 = bits_to_dev(inp["w2"], dev)
    b1 = bits_to_dev(inp["b1"], dev) if inp["b1"] is not None else None
    b2 = bits_to_dev(inp["b2"], dev) if inp["b2"] is not None else None
    # weight preparation (FC1 repack, and the MXFP8 copies on that path): once
    # per optimizer step, timed on its own, outside the step
    for _ in range(2):
        layer.load_weights(w1, b1, w2, b2)
    if args.amax:      # fused NVFP4-prep outputs inside the timed step
        layer.amax_a = torch.zeros(2, dtype=torch.float32, device=dev)
        layer.amax_dh = torch.zeros(2, dtype=torch.float32, device=dev)
    torch.cuda.synchronize()
    p0, p1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    p0.record()
    for _ in range(5):
        layer.load_weights(w1, b1, w2, b2)
    p1.record()
    torch.cuda.synchronize()
    weight_prep_ms = p0.elapsed_time(p1) / 5
    del w1, w2
    if routed:
        x = bits_to_dev(inp["x"], dev)
        logits = torch.from_numpy(inp["logits"]).to(dev)
        bias = torch.from_numpy(inp["bias"]).to(dev) if inp["bias"] is not None else None
        dout = bits_to_dev(inp["dout"], dev)

        def step(timer=None):
            layer.step(x, logits, bias, dout, timer=timer)
    else:
        layer.set_groups(torch.from_numpy(inp["group_sizes"].astype(np.int32)).to(dev))
        po = layer.padded_offsets.cpu().numpy()          # set-up only, outside timing
        xs, dys = bits_to_dev(inp["x"], dev), bits_to_dev(inp["dout"], dev)
        src = 0
        for e, m in enumerate(inp["group_sizes"]):
            m = int(m)
            layer.x_perm[po[e]:po[e] + m].copy_(xs[src:src + m])
            layer.dy[po[e]:po[e] + m].copy_(dys[src:src + m])
            src += m
        del xs, dys

        def step(timer=None):
            layer.grouped_step(timer=timer)

    R = wl.routed_rows
    flops_step = wl.flops_fwd_bwd()
    K, W = args.steps, max(args.warmup, 3)
    stream = torch.cuda.current_stream()

    # timing events inside the graph: one pair per library call per step
    names = []
    step(timer=lambda n: (names.append(n), _Null())[1])
    torch.cuda.synchronize()
    try:
        torch.cuda.Event(enable_timing=True, external=True)
        ext = True
    except TypeError:
        ext = False

    class Timer:
        def __init__(self):
            self.ev = []

        def __call__(self, name):
            a = torch.cuda.Event(enable_timing=True, external=ext)
            b = torch.cuda.Event(enable_timing=True, external=ext)
            self.ev.append((name, a, b))
            return _Rec(a, b)

    def dominant_of(per):
        """The GEMM call with the largest total time."""
        best, best_ms = None, -1.0
        for name, ts in per.items():
            if call_work(wl, name, R, args.dtype)[0] == "flop" and sum(ts) > best_ms:
                best, best_ms = name, sum(ts)
        return best

    use_graph = ext and not args.no_graph
    graph = None
    breakdown = Timer()
    if use_graph:
        # two captures of the same K steps: one with an event pair around
        # every library call (the per-call breakdown, replayed outside the
        # timed region), and the timed one with events only around the
        # dominant GEMM (an event pair between every pair of kernels costs
        # about 5 us of device time, ~3 % of the step)
        warm = torch.cuda.CUDAGraph()
        with torch.cuda.graph(warm):
            step()
        g_break = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_break):
            for _ in range(K):
                step(timer=breakdown)
        torch.cuda.synchronize()
        for _ in range(2):
            warm.replay()
        g_break.replay()
        torch.cuda.synchronize()
        per_break = {}
        for name, a, b in breakdown.ev:
            per_break.setdefault(name, []).append(a.elapsed_time(b))
        dom_name = dominant_of(per_break)
        timer = Timer()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for _ in range(K):
                step(timer=lambda n: timer(n) if n == dom_name else _Null())
        torch.cuda.synchronize()
    else:
        timer = breakdown

    sampler = ClockSampler(gpu_uuid(torch, local))
    # warm-up: W steps, then more until about a second of work has run so
    # that the clock samples describe the loaded GPU
    t_w = time.perf_counter()
    i = 0
    while i < W or time.perf_counter() - t_w < 1.0:
        if use_graph:
            warm.replay()
        else:
            step()
        i += 1
        if i % 8 == 0:
            torch.cuda.synchronize()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    if use_graph:
        graph.replay()
    else:
        for _ in range(K):
            step(timer=timer)
    t1.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clocks = sampler.stop()
    ms_total = t0.elapsed_time(t1)
    status = moe_read_device_status()
    if status != 0:
        raise RuntimeError(f"device status word {status:#x} set during the timed region")

    # per-call durations: the dominant GEMM's from the timed region, every
    # call's from the breakdown replay (graph) or the timed steps (no graph)
    per = {}
    for name, a, b in timer.ev:
        per.setdefault(name, []).append(a.elapsed_time(b))
    if use_graph:
        per_all = dict(per_break)
        per_all.update(per)
    else:
        per_all = per
    ms_max = max_over_ranks(ms_total, dist, dev) if world > 1 else ms_total

    # fused vs unfused expert MLP (same kernels, activation as its own pass)
    fusion = None
    if not args.no_fusion and args.dtype not in ("nvfp4", "fp32") and wl.gated:
        fusion = measure_fusion(torch, layer, K)
    overlap = None
    if args.overlap and not mx and args.dtype != "fp32":
        overlap = measure_overlap(torch, layer)
    router = None
    if routed and not args.no_router and args.dtype != "fp32":
        router = measure_router(torch, layer, x, logits, bias)

    # end-to-end: host buffers in pinned memory, copies inside the timed region
    e2e = None
    if not args.no_e2e:
        if routed:
            e2e = run_e2e(torch, layer, inp, dev, K, W, flops_step, world, dist)
        else:
            e2e = run_e2e_grouped(torch, layer, inp, dev, K, W, flops_step, world, dist)

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return 0

    peaks, peak_src = load_peaks()
    ms_step = ms_max / K
    value = job_rate(flops_step, K, world, ms_max) / 1e12
    kernels = {}
    for name, ts in per_all.items():
        kind, work = call_work(wl, name, R, args.dtype)
        avg = sum(ts) / len(ts)
        ent = {"ms": round(avg, 5)}
        if kind == "flop":
            ent["tflops"] = round(work / (avg * 1e-3) / 1e12, 2)
        elif work > 0:
            ent["gbs"] = round(work / (avg * 1e-3) / 1e9, 1)
        kernels[name] = ent
    dominant = dominant_of(per)
    kind, work = call_work(wl, dominant, R, args.dtype)
    dom_avg = sum(per[dominant]) / len(per[dominant])
    achieved = work / (dom_avg * 1e-3) / 1e12
    dom_bytes = gemm_bytes(wl, dominant, R, args.dtype, keep_bf16=getattr(layer, "keep_bf16", False))
    peak = float(peaks.get("bf16_tflops", PEAKS_FALLBACK["bf16_tflops"]))
    peak_note = f"{peak_src} bf16 burst (cuBLAS)"
    if args.dtype == "mxfp8":   # no measured FP8 figure: bf16 measured x nominal FP8/BF16 (2)
        peak *= 2.0
        peak_note = f"{peak_src} bf16 burst (cuBLAS) x 2, the nominal FP8/BF16 dense ratio"
    elif args.dtype == "nvfp4":  # bf16 measured x the nominal FP4/BF16 dense ratio (13.5/2.25)
        peak *= 6.0
        peak_note = f"{peak_src} bf16 burst (cuBLAS) x 6, the nominal FP4/BF16 dense ratio"
    elif args.dtype == "fp32":   # TF32 MMA: bf16 measured x the nominal TF32/BF16 ratio (1.1/2.25)
        peak *= 1100.0 / 2250.0
        peak_note = f"{peak_src} bf16 burst (cuBLAS) x 1.1/2.25, the nominal TF32/BF16 dense ratio"
    # attainable-roofline view of the whole step: max(FLOP / tensor peak,
    # algorithmic bytes / measured HBM bandwidth), and the nominal peak
    hbm = float(peaks.get("hbm_gbs", PEAKS_FALLBACK["hbm_gbs"]))
    nominal = {"bf16": 2250.0, "mxfp8": 4500.0, "nvfp4": 13500.0, "fp32": 1100.0}[args.dtype]
    sb = step_bytes(wl, args.dtype)
    t_tc, t_hbm = flops_step / (peak * 1e12) * 1e3, sb / (hbm * 1e9) * 1e3
    attainable = {"bytes_per_step": round(sb), "t_tensor_ms": round(t_tc, 4),
                  "t_hbm_ms": round(t_hbm, 4), "bound": "hbm" if t_hbm > t_tc else "tensor",
                  "pct_of_attainable": round(100.0 * max(t_tc, t_hbm) / ms_step, 2),
                  "pct_of_nominal_peak": round(100.0 * value / world / nominal, 2),
                  "nominal_peak_tflops": nominal, "hbm_gbs": hbm}
    tr = NCU_TRAFFIC.get((dominant, wl.name, args.dtype))
    traffic = tr["bytes"] if tr and tr.get("src") == gemm_source_hash() else None
    # the dominant GEMM against both roofs; the one that takes longer bounds it
    gbs = dom_bytes / (dom_avg * 1e-3) / 1e9
    t_tc_dom, t_hbm_dom = work / (peak * 1e12), dom_bytes / (hbm * 1e9)
    tensor_roof = {"achieved": round(achieved, 2), "peak": peak, "unit": "TFLOP/s",
                   "frac": round(achieved / peak, 4), "peak_source": peak_note}
    hbm_roof = {"achieved": round(gbs, 1), "peak": hbm, "unit": "GB/s",
                "frac": round(gbs / hbm, 4), "bytes": round(dom_bytes),
                "peak_source": f"{peak_src} copy bandwidth"}
    if t_hbm_dom > t_tc_dom:
        roofline = dict(bound="hbm", kernel=dominant, **{k: v for k, v in hbm_roof.items()
                                                         if k != "bytes"})
    else:
        roofline = dict(bound="tensor", kernel=dominant, **tensor_roof)
    roofline.update(traffic=traffic, algorithmic_bytes=round(dom_bytes), tensor=tensor_roof,
                    hbm=hbm_roof)
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOPS", "n_gpus": world,
        "steps": K, "warmup": W, "ms_per_step": round(ms_step, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": args.dtype, "data": "synthetic",
        "config": dict(workload_config(wl, args.dtype), amax_outputs=bool(args.amax),
                       parallelism=f"replicas x{world}",
                       graph=bool(use_graph)),
        "tokens_per_s": round(job_rate(wl.T if routed else R, K, world, ms_max), 1),
        "pct_of_tc_peak": round(100.0 * value / world / peak, 2),
        "attainable": attainable,
        "roofline": roofline,
        "kernels": kernels,
        "gpu_launches": layer.kernels_per_step(routed) * K,
        "weight_prep_ms": round(weight_prep_ms, 4),
        "clocks": clocks,
        "e2e": e2e,
        "fusion": fusion,
        "overlap": overlap,
        "router": router,
    }
    if not args.no_cpu_baseline:
        dt, fl, desc = oracle_sample_run(wl, inp, args.cpu_sample_tokens, args.dtype)
        line["cpu_baseline"] = {"value": fl / dt / 1e12, "unit": "TFLOPS", "cores": host_cores(),
                                "kind": "oracle", "sample": desc}
    print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()
    return 0


def measure_fusion(torch, layer, K):
    """Forward and backward of the expert MLP, fused epilogues against the
    unfused arrangement the pages measure their kernels against: the group
    sizes read back to the host each pass (a device-to-host copy and a
    synchronisation), plain grouped GEMMs, and the activation (GLU / dGLU)
    and, on the MXFP8 path, the quantization of its output (rowwise and
    transposed) as separate memory-bound passes.  CUDA events, K reps each
    after 3 warm-ups.  The pages report up to 1.3x forward and 2.1x backward
    for their fused kernels.  Also the backward with activation recompute (H
    regenerated from the forward's operands instead of read back)."""
    def timed(fn):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(K):
            fn()
        b.record()
        torch.cuda.synchronize()
        return a.elapsed_time(b) / K
    f_fused = timed(layer.mlp_forward)
    f_unf = timed(layer.mlp_forward_unfused)
    b_fused = timed(layer.mlp_backward)
    b_unf = timed(layer.mlp_backward_unfused)
    from moe_expert_mlp_gb300 import _lib as L
    if layer.mx:
        # the MXFP8 backward regenerating H (moe_fc1_recompute_h_mx) first
        layer.recompute_h = True
        b_rec = timed(layer.mlp_backward)
        layer.recompute_h = False
    else:
        # the bf16 backward regenerating H in its workspace
        desc_r = type(layer.desc).from_buffer_copy(layer.desc)
        desc_r.recompute_h = 1
        ws_r = torch.zeros(L.moe_workspace_size(desc_r), dtype=torch.uint8,
                           device=layer.ws.device)
        b_rec = timed(lambda: L.moe_mlp_bwd(
            desc_r, layer.dy, layer.x_perm, None, layer.a, layer.counts, layer.padded_offsets,
            layer.w1p, layer.w2, layer.dh, layer.dx_perm, layer.dw1p, layer.db1p, layer.dw2,
            layer.db2, ws_r, b1p=layer.b1p))
        del ws_r
    layer.mlp_forward()                      # leave the fused results in place
    layer.mlp_backward()
    what = ("host-synchronised group sizes, plain grouped GEMMs, GLU / dGLU as separate "
            "passes" + (", MXFP8 quantize + transpose of A / dH as separate passes"
                        if layer.mx else ""))
    return {"fwd_fused_ms": round(f_fused, 4), "fwd_unfused_ms": round(f_unf, 4),
            "fwd_speedup": round(f_unf / f_fused, 3), "bwd_fused_ms": round(b_fused, 4),
            "bwd_unfused_ms": round(b_unf, 4), "bwd_speedup": round(b_unf / b_fused, 3),
            "bwd_recompute_h_ms": round(b_rec, 4), "unfused": what,
            "pages_reported": "up to 1.3x forward, 2.1x backward (their fused vs unfused)"}


def measure_router(torch, layer, x, logits, bias, reps=20):
    """Routing from given logits (the step's moe_route_permute) against the
    fused router, which computes the logits itself (router GEMM x W_r^T,
    W_r seeded bf16 [E,d]), takes the top-k in the GEMM epilogue and runs
    the same permutation in the same launch; each captured in a CUDA graph,
    CUDA events around the replays, medians."""
    g = torch.Generator(device="cpu").manual_seed(5)
    w_r = (torch.randn((layer.E, layer.d), generator=g) / layer.d ** 0.5).to(torch.bfloat16)
    w_r = w_r.to(x.device)

    def timed(fn):
        # captured in a CUDA graph, as the step is: device time only
        fn()
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            fn()
        ts = []
        for i in range(reps + 3):
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record()
            graph.replay()
            b.record()
            torch.cuda.synchronize()
            if i >= 3:
                ts.append(a.elapsed_time(b))
        return statistics.median(ts)

    given = timed(lambda: layer.route(x, logits, bias))
    fused = timed(lambda: layer.route_fused(x, w_r, bias))
    layer.route(x, logits, bias)          # leave the step's routing in place
    torch.cuda.synchronize()
    return {"route_permute_ms": round(given, 4), "route_fused_ms": round(fused, 4),
            "fused": "one cooperative launch: router GEMM x W_r^T + top-k/softmax/histogram "
                     "epilogue, then (after grid-wide barriers) the same scan/assign/gather"}


def measure_overlap(torch, layer, reps=10):
    """sm_margin: the grouped GEMM leaves `sm_margin` SMs free so that a
    concurrent kernel (in the pages, the expert-parallel communication
    kernels) progresses beside it.  Stand-in concurrent kernel: a 512 MB
    device copy (torch's elementwise copy, SM-bound memory streaming) on a
    second stream.  For each margin: FC1+GLU alone, the copy alone, and both
    launched together (time until both finish), CUDA events, medians."""
    from moe_expert_mlp_gb300 import _lib as L
    src = torch.empty(256 * 2**20, dtype=torch.bfloat16, device=layer.w2.device)
    dst = torch.empty_like(src)
    s_main = torch.cuda.current_stream()
    s_side = torch.cuda.Stream()
    c, po = layer.counts, layer.padded_offsets

    def gemm(desc, stream):
        L.moe_fc1_glu_fwd(desc, layer.x_perm, c, po, layer.w1p, layer.b1p, layer.h, layer.a,
                          stream)

    def timed(fn):
        ts = []
        for i in range(reps + 3):
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            a.record(s_main)
            fn()
            b.record(s_main)
            torch.cuda.synchronize()
            if i >= 3:
                ts.append(a.elapsed_time(b))
        return statistics.median(ts)

    def both(desc):
        start = torch.cuda.Event()
        start.record(s_main)
        s_side.wait_event(start)
        gemm(desc, s_main)
        with torch.cuda.stream(s_side):
            dst.copy_(src)
        done = torch.cuda.Event()
        done.record(s_side)
        s_main.wait_event(done)

    def side_only():
        start = torch.cuda.Event()
        start.record(s_main)
        s_side.wait_event(start)
        with torch.cuda.stream(s_side):
            dst.copy_(src)
        done = torch.cuda.Event()
        done.record(s_side)
        s_main.wait_event(done)

    side = timed(side_only)
    out = {"concurrent": "512 MB device copy on a second stream", "copy_alone_ms": round(side, 4)}
    rows = []
    for m in (0, 16, 32):
        desc = type(layer.desc).from_buffer_copy(layer.desc)
        desc.sm_margin = m
        g = timed(lambda: gemm(desc, s_main))
        bt = timed(lambda: both(desc))
        rows.append({"sm_margin": m, "fc1_glu_alone_ms": round(g, 4), "both_ms": round(bt, 4),
                     "serial_ms": round(g + side, 4)})
    out["by_margin"] = rows
    del src, dst
    return out


def run_e2e(torch, layer, inp, dev, K, W, flops_step, world, dist):
    """The same step through the public API with host-resident inputs and
    results: pinned host -> device copies of x, logits, dout for every step
    and device -> host copies of out, dx, dlogits after it.  Headline: the
    library's HostStepPipeline (each step's copies overlapped with the
    neighbouring steps' kernels); also reported: the same copies issued in
    line, one step after another, on one stream."""
    from moe_expert_mlp_gb300.pipeline import HostStepPipeline
    host = lambda b: torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).to(layer.act_dtype)
    xh = host(inp["x"]).pin_memory()
    lh = torch.from_numpy(inp["logits"]).pin_memory()
    dh = host(inp["dout"]).pin_memory()
    bias = torch.from_numpy(inp["bias"]).to(dev) if inp["bias"] is not None else None
    xd, ld, dd = (torch.empty_like(t, device=dev) for t in (xh, lh, dh))
    outs = [dict(out=torch.empty(layer.out.shape, dtype=layer.out.dtype).pin_memory(),
                 dx=torch.empty(layer.dx.shape, dtype=layer.dx.dtype).pin_memory(),
                 dlogits=torch.empty(layer.dlogits.shape, dtype=torch.float32).pin_memory())
            for _ in range(2)]
    host_in = dict(x=xh, logits=lh, dout=dh)
    pipe = HostStepPipeline(layer, dev)

    def serial():
        xd.copy_(xh, non_blocking=True)
        ld.copy_(lh, non_blocking=True)
        dd.copy_(dh, non_blocking=True)
        layer.step(xd, ld, bias, dd)
        for k, t in (("out", layer.out), ("dx", layer.dx), ("dlogits", layer.dlogits)):
            outs[0][k].copy_(t, non_blocking=True)

    def timed(fn):
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        fn()
        b.record()
        torch.cuda.synchronize()
        ms = a.elapsed_time(b)
        return max_over_ranks(ms, dist, dev) if world > 1 else ms

    pipe.run([host_in] * W, [outs[i % 2] for i in range(W)], bias)
    ms = timed(lambda: pipe.run([host_in] * K, [outs[i % 2] for i in range(K)], bias))
    for _ in range(W):
        serial()
    ms_serial = timed(lambda: [serial() for _ in range(K)])
    h2d = sum(t.numel() * t.element_size() for t in (xh, lh, dh))
    d2h = sum(t.numel() * t.element_size() for t in outs[0].values())
    return {"value": round(job_rate(flops_step, K, world, ms) / 1e12, 2), "unit": "TFLOPS",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "ms_per_step": round(ms / K, 5), "api": "HostStepPipeline (copies overlapped)",
            "serial": {"value": round(job_rate(flops_step, K, world, ms_serial) / 1e12, 2),
                       "ms_per_step": round(ms_serial / K, 5),
                       "api": "MoEExpertMLP.step with in-line copies"}}


def run_e2e_grouped(torch, layer, inp, dev, K, W, flops_step, world, dist):
    """End to end for groups given directly (no router): every step copies
    in, from pinned host memory, the R expert-ordered rows x and their
    upstream gradient dY and the group sizes, recomputes the group offsets
    on the device, runs the expert MLP forward and backward, and copies the
    R rows of Y and dX back to pinned host memory (group by group, between
    the host's dense row order and the library's padded layout).  The
    weight gradients stay on the device for the optimizer.  Headline:
    GroupedHostStepPipeline (copies overlapped with the neighbouring steps'
    kernels); also reported: the same copies issued in line on one stream."""
    from moe_expert_mlp_gb300.pipeline import GroupedHostStepPipeline
    R, d = int(inp["group_sizes"].sum()), layer.d
    host = lambda b: torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).to(layer.act_dtype)
    host_in = dict(x=host(inp["x"]).pin_memory(), dy=host(inp["dout"]).pin_memory(),
                   counts=torch.from_numpy(inp["group_sizes"].astype(np.int32)).pin_memory())
    outs = [dict(y=torch.empty((R, d), dtype=layer.act_dtype).pin_memory(),
                 dx=torch.empty((R, d), dtype=layer.act_dtype).pin_memory()) for _ in range(2)]
    pipe = GroupedHostStepPipeline(layer, dev)
    segs = pipe._segments(inp["group_sizes"])
    cnt_dev = torch.zeros_like(layer.counts)

    def serial():
        for src, dst, m in segs:
            layer.x_perm[dst:dst + m].copy_(host_in["x"][src:src + m], non_blocking=True)
            layer.dy[dst:dst + m].copy_(host_in["dy"][src:src + m], non_blocking=True)
        cnt_dev.copy_(host_in["counts"], non_blocking=True)
        layer.grouped_step(counts=cnt_dev)
        for src, dst, m in segs:
            outs[0]["y"][src:src + m].copy_(layer.y[dst:dst + m], non_blocking=True)
            outs[0]["dx"][src:src + m].copy_(layer.dx_perm[dst:dst + m], non_blocking=True)

    def timed(fn):
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        fn()
        b.record()
        torch.cuda.synchronize()
        ms = a.elapsed_time(b)
        return max_over_ranks(ms, dist, dev) if world > 1 else ms

    pipe.run([host_in] * W, [outs[i % 2] for i in range(W)])
    ms = timed(lambda: pipe.run([host_in] * K, [outs[i % 2] for i in range(K)]))
    for _ in range(W):
        serial()
    ms_serial = timed(lambda: [serial() for _ in range(K)])
    h2d = sum(t.numel() * t.element_size() for t in host_in.values())
    d2h = sum(t.numel() * t.element_size() for t in outs[0].values())
    return {"value": round(job_rate(flops_step, K, world, ms) / 1e12, 2), "unit": "TFLOPS",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "ms_per_step": round(ms / K, 5),
            "api": "GroupedHostStepPipeline (copies overlapped); inputs x, dY (real rows) and "
                   "group sizes; results Y, dX (real rows); weight gradients stay on the device",
            "serial": {"value": round(job_rate(flops_step, K, world, ms_serial) / 1e12, 2),
                       "ms_per_step": round(ms_serial / K, 5),
                       "api": "MoEExpertMLP.grouped_step with in-line copies"}}


class _Null:
    def __enter__(self):
        return self

    def __exit__(self, *a):
        return False


class _Rec:
    def __init__(self, a, b):
        self.a, self.b = a, b

    def __enter__(self):
        self.a.record()
        return self

    def __exit__(self, *exc):
        self.b.record()
        return False


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(WORKLOADS))
    ap.add_argument("--cpu-sample-tokens", type=int, default=None,
                    help="tokens (routed layers; default 1024) or rows (direct groups: the "
                         "smallest experts up to this many rows; default one expert) of the "
                         "oracle sample in the cpu_baseline leg")
    ap.add_argument("--ref-sample-tokens", type=int, default=None,
                    help="the same for each step of --impl reference (default 256 tokens, or "
                         "the smallest expert)")
    ap.add_argument("--dtype", choices=["bf16", "mxfp8", "nvfp4", "fp32"], default=DEFAULT_DTYPE,
                    help="GEMM operand type (mxfp8: E4M3 + E8M0 block scales; nvfp4: E2M1 + "
                         "UE4M3 scales per 16 + per-tensor scales; fp32: fp32 tensors, TF32 "
                         "tensor-core GEMMs)")
    ap.add_argument("--act", choices=["swiglu", "geglu", "sreglu", "srelu"], default=None,
                    help="override the workload's activation (the dense sweep)")
    ap.add_argument("--amax", action="store_true",
                    help="also produce the fused per-tensor amax of A and dH (NVFP4 prep)")
    ap.add_argument("--overlap", action="store_true",
                    help="also time FC1 beside a concurrent kernel for several sm_margin values")
    ap.add_argument("--no-router", action="store_true",
                    help="skip timing the fused router against routing from given logits")
    ap.add_argument("--no-graph", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--quantize-only", action="store_true",
                    help="time only the MXFP8 activation quantizer on a [routed rows, d] "
                         "tensor of the workload (a small-memory command for kernel profiles)")
    ap.add_argument("--no-fusion", action="store_true",
                    help="skip the fused-vs-unfused expert MLP comparison")
    args = ap.parse_args()
    wl = WORKLOADS[args.workload]
    # oracle samples: the oracle quantizes each sampled expert's weights
    # (tens of millions of elements, seconds each at the DeepSeek-shaped
    # size), so on layers with directly given groups the sample is the
    # smallest non-empty expert and all of its rows
    direct = wl.router == "direct"
    if args.cpu_sample_tokens is None:
        args.cpu_sample_tokens = 1 if direct else 1024
    if args.ref_sample_tokens is None:
        args.ref_sample_tokens = 1 if direct else 256
    if args.act is not None:
        wl = dataclasses.replace(wl, act=args.act)
    if args.impl == "reference":
        return run_reference(args, wl)
    if args.quantize_only:
        return run_quantize_only(args, wl)
    return run_ours(args, wl)


if __name__ == "__main__":
    sys.exit(main())
