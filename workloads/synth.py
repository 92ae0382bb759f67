"""Seeded synthetic MoE-layer inputs shaped like the pages' workloads.

Every array is drawn with numpy's PCG64 generator from a stated seed, in
fp32, and then rounded (round-to-nearest-even) to the storage type the
library consumes: bf16 bit patterns (``uint16``) for activations, weights
and upstream gradients, fp32 for router logits and bias.  The same arrays
are handed to the CUDA path and to the CPU oracle.

Workloads (names say what they are; sizes follow the MoE layer shapes in
"Boosting MoE training throughput with advanced fused kernels", section
"Overcoming training bottlenecks in the MoE block", and the DeepSeek-V3 /
GPT-OSS layer shapes it and "Dropless MoE training with JAX and Transformer
Engine" refer to):

* ``tiny_t256_e8``      T=256, d=256, E=8, F=512, k=2, SwiGLU.  x and the
  router matrix ~N(0,1)/sqrt(d); logits = x @ W_r (fp64, rounded to fp32).
* ``bf16_t4096_e64``    T=4096, d=2048, E=64, F=1408, k=6, SwiGLU, logits
  ~N(0,1) plus a per-expert selection bias ~N(0,1) that skews the load.
* ``dsv3_r16384_e32``   16384 routed rows over 32 local experts with
  Zipf(s=1.2) group sizes and 4 empty experts, d=7168, F=2048, SwiGLU,
  weights ~N(0,0.006).  Rows and group sizes are given directly (no router).
* ``gptoss_t16384_e32`` T=16384, d=2880, E=32, F=2880, k=4, SwiGLU with gate
  clamp 7.0, gate scale alpha=1.702, linear offset 1, biases ~N(0,0.01).
* ``dense_m16384``      one group of 16384 rows, d=4096, F=14336 (a dense
  MLP); the activation is chosen per run.
* ``dsv3_r4096_e8``     the DeepSeek-shaped layer cut to 8 experts / 4096
  rows (one empty), for hardware-counter captures.

Unstated scales are read as: x ~ N(0,1), expert weights ~ N(0,0.02),
upstream gradient ~ N(0,1).
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    E: int
    d: int
    F: int
    k: int = 1
    T: int = 0                 # tokens; 0 when the groups are given directly
    R: int = 0                 # routed rows when the groups are given directly
    act: str = "swiglu"        # swiglu | geglu | sreglu | srelu (non-gated)
    alpha: float = 1.0
    limit: float = math.inf
    linear_offset: float = 0.0
    out_scale: float = 1.0
    has_b1: bool = False
    has_b2: bool = False
    b_std: float = 0.0
    router: str = "logits"     # logits | xw | direct
    router_bias: bool = False
    zipf_s: float = 0.0        # direct groups: Zipf exponent (0 = one even split)
    zipf_empty: int = 0        # direct groups: experts forced empty
    x_std: float = 1.0
    w_std: float = 0.02
    seed: int = 0

    @property
    def gated(self) -> bool:
        return self.act != "srelu"

    @property
    def routed_rows(self) -> int:
        return self.R if self.router == "direct" else self.T * self.k

    def flops_fwd_bwd(self) -> float:
        """Algorithmic FLOPs of one fwd+bwd pass: 18*d*F per routed row for a
        gated MLP (FC1 d->2F and FC2 F->d, forward once and twice backward);
        12*d*F for the non-gated form."""
        per_row = (18 if self.gated else 12) * self.d * self.F
        return float(per_row) * self.routed_rows


WORKLOADS = {
    "tiny_t256_e8": Workload(
        name="tiny_t256_e8", T=256, E=8, d=256, F=512, k=2, router="xw",
        x_std=1.0 / 16.0, w_std=0.02),
    "bf16_t4096_e64": Workload(
        name="bf16_t4096_e64", T=4096, E=64, d=2048, F=1408, k=6,
        router="logits", router_bias=True),
    "dsv3_r16384_e32": Workload(
        name="dsv3_r16384_e32", R=16384, E=32, d=7168, F=2048, router="direct",
        zipf_s=1.2, zipf_empty=4, w_std=0.006),
    "gptoss_t16384_e32": Workload(
        name="gptoss_t16384_e32", T=16384, E=32, d=2880, F=2880, k=4,
        limit=7.0, alpha=1.702, linear_offset=1.0, has_b1=True, has_b2=True,
        b_std=0.01),
    "dense_m16384": Workload(
        name="dense_m16384", R=16384, E=1, d=4096, F=14336, router="direct"),
    # the DeepSeek-shaped layer cut to 8 experts and 4096 rows (same d, F and
    # group-size law, about 2 GB on the device in MXFP8): small enough for
    # per-kernel hardware-counter captures
    "dsv3_r4096_e8": Workload(
        name="dsv3_r4096_e8", R=4096, E=8, d=7168, F=2048, router="direct",
        zipf_s=1.2, zipf_empty=1, w_std=0.006),
}


def scaled(base: Workload, **changes) -> Workload:
    """A smaller (or otherwise changed) copy of a workload, e.g. for parity
    cases the oracle finishes in seconds."""
    return dataclasses.replace(base, **changes)


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round finite fp32 values to bf16 (nearest, ties to even); return the
    16-bit patterns."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f64(b: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to fp64."""
    u = np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u.view(np.float32).astype(np.float64)


def zipf_group_sizes(R: int, E: int, s: float, n_empty: int,
                     rng: np.random.Generator) -> np.ndarray:
    """Group sizes that sum to R.  Ranks 1..E-n_empty get R*r^-s/sum(r^-s)
    rows (largest-remainder rounding); the n_empty lowest ranks get 0 rows;
    ranks are mapped to experts by a seeded permutation.  s=0 gives an even
    split."""
    n = E - n_empty
    r = np.arange(1, n + 1, dtype=np.float64)
    share = r ** (-s) if s > 0 else np.ones(n)
    exact = R * share / share.sum()
    base = np.floor(exact).astype(np.int64)
    rest = R - int(base.sum())
    frac_order = np.argsort(-(exact - base), kind="stable")
    base[frac_order[:rest]] += 1
    sizes_by_rank = np.concatenate([base, np.zeros(n_empty, dtype=np.int64)])
    perm = rng.permutation(E)
    sizes = np.zeros(E, dtype=np.int64)
    sizes[perm] = sizes_by_rank
    return sizes


def _normal_bf16(rng: np.random.Generator, shape, std: float) -> np.ndarray:
    out = np.empty(shape, dtype=np.uint16)
    flat = out.reshape(-1)
    chunk = 1 << 24
    for i in range(0, flat.size, chunk):
        n = min(chunk, flat.size - i)
        v = rng.standard_normal(n, dtype=np.float32)
        if std != 1.0:
            v *= np.float32(std)
        flat[i:i + n] = f32_to_bf16_bits(v)
    return out


def make_inputs(wl: Workload, seed: Optional[int] = None,
                with_weights: bool = True) -> dict:
    """Draw one layer's inputs.

    Returns a dict of numpy arrays:
      logits f32 [T,E], bias f32 [E] or None       (router workloads)
      group_sizes i64 [E]                          (direct workloads)
      x    u16 [T,d] (router) or [R,d] rows in expert order (direct)
      dout u16 [T,d] (router) or [R,d] rows in expert order (direct)
      w1   u16 [E,2F,d] (gated: rows 0..F-1 gate, F..2F-1 linear) or [E,F,d]
      b1   u16 [E,2F] / [E,F] or None,  w2 u16 [E,d,F],  b2 u16 [E,d] or None
    """
    rng = np.random.Generator(np.random.PCG64(wl.seed if seed is None else seed))
    out: dict = {}
    n1 = 2 * wl.F if wl.gated else wl.F
    if wl.router == "direct":
        if wl.E == 1:
            sizes = np.array([wl.R], dtype=np.int64)
        else:
            sizes = zipf_group_sizes(wl.R, wl.E, wl.zipf_s, wl.zipf_empty, rng)
        out["group_sizes"] = sizes
        out["logits"] = None
        out["bias"] = None
        out["x"] = _normal_bf16(rng, (wl.R, wl.d), wl.x_std)
    else:
        x32 = rng.standard_normal((wl.T, wl.d), dtype=np.float32) * np.float32(wl.x_std)
        out["x"] = f32_to_bf16_bits(x32)
        if wl.router == "xw":
            wr = rng.standard_normal((wl.d, wl.E)) / math.sqrt(wl.d)
            xb = bf16_bits_to_f64(out["x"])
            out["logits"] = (xb @ wr).astype(np.float32)
        else:
            out["logits"] = rng.standard_normal((wl.T, wl.E), dtype=np.float32)
        out["bias"] = (rng.standard_normal(wl.E, dtype=np.float32)
                       if wl.router_bias else None)
        out["group_sizes"] = None
    if with_weights:
        out["w1"] = _normal_bf16(rng, (wl.E, n1, wl.d), wl.w_std)
        out["w2"] = _normal_bf16(rng, (wl.E, wl.d, wl.F), wl.w_std)
        out["b1"] = _normal_bf16(rng, (wl.E, n1), wl.b_std) if wl.has_b1 else None
        out["b2"] = _normal_bf16(rng, (wl.E, wl.d), wl.b_std) if wl.has_b2 else None
    rows = wl.R if wl.router == "direct" else wl.T
    out["dout"] = _normal_bf16(rng, (rows, wl.d), 1.0)
    return out


def make_inputs_fp32(wl: Workload, seed: Optional[int] = None) -> dict:
    """fp32 inputs of a routed layer (x, logits, dout, w1, w2, optional
    biases; no bf16 rounding), drawn from the workload's distributions with
    their own seeded stream: for the fp32 configuration, whose values reach
    a bf16 path only after rounding."""
    rng = np.random.Generator(np.random.PCG64(wl.seed if seed is None else seed))
    n1 = 2 * wl.F if wl.gated else wl.F
    f32 = np.float32
    x = rng.standard_normal((wl.T, wl.d), dtype=f32) * f32(wl.x_std)
    if wl.router == "xw":
        wr = rng.standard_normal((wl.d, wl.E)) / math.sqrt(wl.d)
        logits = (x.astype(np.float64) @ wr).astype(f32)
    else:
        logits = rng.standard_normal((wl.T, wl.E), dtype=f32)
    bias = rng.standard_normal(wl.E, dtype=f32) if wl.router_bias else None
    return {
        "x": x, "logits": logits, "bias": bias,
        "dout": rng.standard_normal((wl.T, wl.d), dtype=f32),
        "w1": rng.standard_normal((wl.E, n1, wl.d), dtype=f32) * f32(wl.w_std),
        "w2": rng.standard_normal((wl.E, wl.d, wl.F), dtype=f32) * f32(wl.w_std),
        "b1": rng.standard_normal((wl.E, n1), dtype=f32) * f32(wl.b_std) if wl.has_b1 else None,
        "b2": rng.standard_normal((wl.E, wl.d), dtype=f32) * f32(wl.b_std) if wl.has_b2 else None,
    }
