"""Routed-expert MLP in fp64: routing, permute, FC1 + GLU, FC2, combine, and
the analytic backward.  Test infrastructure only (see the package header).

Row layout.  Routed rows are stored expert after expert ("ragged tensor",
Accelerating dropless MoE training..., "Claims and evidence"); each expert's
group starts at a multiple of ``align`` rows and the rows between the end of
a group and the next start are padding.  Every per-row tensor is zero on
padding rows.  Inside a group rows are in ascending token order.
"""
from __future__ import annotations

import math

import numpy as np
from scipy.special import erf

__all__ = [
    "ACTS", "GluParams", "route", "group_offsets", "permute_index", "gather_rows",
    "glu_forward", "glu_backward", "fc1_packed_columns", "repack_fc1", "unpack_fc1",
    "expert_forward", "expert_backward", "moe_forward", "moe_backward",
    "grouped_forward", "grouped_backward", "combine", "combine_backward",
    "permute_backward", "route_backward",
]

ACTS = ("swiglu", "geglu", "sreglu", "srelu")


class GluParams:
    """Activation settings of the FC1 epilogue.

    The supported activations are SwiGLU, GeGLU and sReLU, with optional
    clamping and scaling (Improving MoE training throughput..., "Overcoming
    training bottlenecks in the MoE block"), and the epilogue also applies
    feature scaling, tensor clamping and a bias add ("Optimizing GLU
    activations with fused GEMM epilogues", last paragraph).

    Readings where the pages are silent:
      gate g (first half of FC1's output), linear l (second half);
      g' = min(g, limit), l' = clip(l, -limit, limit);
      swiglu:  phi(g') = g' * sigmoid(alpha * g')
      geglu:   phi(g') = 0.5 * g' * (1 + erf(g' / sqrt 2))
      sreglu:  phi(g') = max(g', 0)^2         (gated squared ReLU)
      srelu:   phi(g')  with no linear half    (non-gated squared ReLU)
      A = out_scale * phi(g') * (l' + linear_offset)   (gated)
      A = out_scale * phi(g')                          (srelu)
    """

    def __init__(self, act="swiglu", alpha=1.0, limit=math.inf,
                 linear_offset=0.0, out_scale=1.0):
        assert act in ACTS
        self.act = act
        self.alpha = float(alpha)
        self.limit = float(limit)
        self.linear_offset = float(linear_offset)
        self.out_scale = float(out_scale)

    @property
    def gated(self):
        return self.act != "srelu"


# --------------------------------------------------------------------------
# Routing: top-k expert choice per token; the per-expert token counts are only
# known at run time (Improving MoE training throughput..., "Overcoming
# training bottlenecks in the MoE block", CPU constraint bullet) and stay in
# device memory ("Eliminating host-device synchronisation ...").
# --------------------------------------------------------------------------

def route(logits_f32, bias_f32, k):
    """Top-k routing.

    Selection score s[t,e] = logits[t,e] + bias[e], evaluated in fp32 (the
    precision the kernel decides in).  The k experts with the largest scores
    are chosen, equal scores going to the lower expert index, listed in
    descending score.  The gate weights are the softmax of the selected raw
    logits (the bias only steers selection).  Returns topk_idx int32 [T,k],
    topk_w fp64 [T,k] and counts int64 [E].
    """
    logits_f32 = np.asarray(logits_f32, dtype=np.float32)
    T, E = logits_f32.shape
    score = logits_f32.copy()
    if bias_f32 is not None:
        score = (score + np.asarray(bias_f32, dtype=np.float32)[None, :]).astype(np.float32)
    # stable sort of the negated score: equal scores keep ascending expert order
    order = np.argsort(-score, axis=1, kind="stable")
    topk_idx = order[:, :k].astype(np.int32)
    sel = np.take_along_axis(logits_f32, topk_idx, axis=1).astype(np.float64)
    z = np.exp(sel - sel.max(axis=1, keepdims=True))
    topk_w = z / z.sum(axis=1, keepdims=True)
    counts = np.bincount(topk_idx.reshape(-1), minlength=E).astype(np.int64)
    return topk_idx, topk_w, counts


def group_offsets(counts, align=128, tile_m=128):
    """Exclusive scans of the group sizes.

    offsets[e]        = sum of counts[:e]               (offsets[E] = R)
    padded_offsets[e] = sum of ceil(counts/align)*align over [:e]
    tile_prefix[e]    = sum of ceil(counts/tile_m) over [:e]
    """
    counts = np.asarray(counts, dtype=np.int64)
    E = counts.shape[0]
    offsets = np.zeros(E + 1, dtype=np.int64)
    padded = np.zeros(E + 1, dtype=np.int64)
    tiles = np.zeros(E + 1, dtype=np.int64)
    for e in range(E):
        offsets[e + 1] = offsets[e] + counts[e]
        padded[e + 1] = padded[e] + (counts[e] + align - 1) // align * align
        tiles[e + 1] = tiles[e] + (counts[e] + tile_m - 1) // tile_m
    return offsets, padded, tiles


def permute_index(topk_idx, E, padded_offsets):
    """Stable counting sort of the (token, slot) pairs by expert.

    Row j of expert e's group holds the j-th smallest token that chose e.
    Returns row_src int32 [padded_offsets[E]] (token of each row, -1 on
    padding) and row_of int32 [T,k] (row of each (token, slot)).
    """
    T, k = topk_idx.shape
    R_pad = int(padded_offsets[E])
    row_src = np.full(R_pad, -1, dtype=np.int32)
    row_of = np.full((T, k), -1, dtype=np.int32)
    fill = np.array(padded_offsets[:E], dtype=np.int64)
    for t in range(T):                       # ascending token order
        for s in range(k):
            e = int(topk_idx[t, s])
            row_src[fill[e]] = t
            row_of[t, s] = fill[e]
            fill[e] += 1
    return row_src, row_of


def gather_rows(x, row_src):
    """x_perm[j] = x[row_src[j]]; padding rows are zero."""
    out = np.zeros((row_src.shape[0],) + x.shape[1:], dtype=x.dtype)
    real = row_src >= 0
    out[real] = x[row_src[real]]
    return out


# --------------------------------------------------------------------------
# GLU activation and its derivative (Improving MoE training throughput...,
# "Optimizing GLU activations with fused GEMM epilogues": FC1's output is
# split into two chunks that are combined into the GLU output; the backward
# epilogue computes dSwiGLU from the GEMM output).
# --------------------------------------------------------------------------

def _sigmoid(x):
    return 0.5 * (1.0 + np.tanh(0.5 * x))


def _phi(gc, p):
    if p.act == "swiglu":
        return gc * _sigmoid(p.alpha * gc)
    if p.act == "geglu":
        return 0.5 * gc * (1.0 + erf(gc / math.sqrt(2.0)))
    return np.maximum(gc, 0.0) ** 2            # sreglu, srelu


def _dphi(gc, p):
    if p.act == "swiglu":
        s = _sigmoid(p.alpha * gc)
        return s + p.alpha * gc * s * (1.0 - s)
    if p.act == "geglu":
        cdf = 0.5 * (1.0 + erf(gc / math.sqrt(2.0)))
        pdf = np.exp(-0.5 * gc * gc) / math.sqrt(2.0 * math.pi)
        return cdf + gc * pdf
    return 2.0 * np.maximum(gc, 0.0)


def glu_forward(g, l, p):
    """A = out_scale * phi(min(g,limit)) * (clip(l,-limit,limit) + offset);
    for the non-gated form ``l`` is ignored and A = out_scale * phi(g')."""
    gc = np.minimum(g, p.limit)
    if not p.gated:
        return p.out_scale * _phi(gc, p)
    lc = np.clip(l, -p.limit, p.limit)
    return p.out_scale * _phi(gc, p) * (lc + p.linear_offset)


def glu_backward(dA, g, l, p):
    """Gradients of glu_forward w.r.t. g and l.  The clamps pass the gradient
    where the input lies inside their bounds, bounds included."""
    gc = np.minimum(g, p.limit)
    pass_g = (g <= p.limit).astype(np.float64)
    da = p.out_scale * dA
    if not p.gated:
        return da * _dphi(gc, p) * pass_g, None
    lc = np.clip(l, -p.limit, p.limit)
    pass_l = ((l >= -p.limit) & (l <= p.limit)).astype(np.float64)
    dg = da * (lc + p.linear_offset) * _dphi(gc, p) * pass_g
    dl = da * _phi(gc, p) * pass_l
    return dg, dl


# --------------------------------------------------------------------------
# FC1 weight repack (Improving MoE training throughput..., "Optimizing GLU
# activations with fused GEMM epilogues", Figure 2): the weight is repacked
# into input and gate columns so one thread block holds half a tile width of
# each.  Reading: packed block b of 2h rows holds gate rows [b*h, b*h+h)
# then linear rows [b*h, b*h+h); F is zero-padded to a multiple of h.
# --------------------------------------------------------------------------

def fc1_packed_columns(F, h=128):
    """Logical FC1 output column of each packed column (-1 on padding).
    Logical columns 0..F-1 are the gate, F..2F-1 the linear half."""
    F_pad = (F + h - 1) // h * h
    src = np.full(2 * F_pad, -1, dtype=np.int64)
    for b in range(F_pad // h):
        for j in range(h):
            f = b * h + j
            if f < F:
                src[2 * b * h + j] = f               # gate
                src[2 * b * h + h + j] = F + f       # linear
    return src


def repack_fc1(w1, b1=None, h=128):
    """w1 [E,2F,d] (logical) -> w1p [E,2F_pad,d]; b1 [E,2F] -> b1p [E,2F_pad]."""
    E, twoF, d = w1.shape
    src = fc1_packed_columns(twoF // 2, h)
    w1p = np.zeros((E, src.shape[0], d), dtype=w1.dtype)
    ok = src >= 0
    w1p[:, ok, :] = w1[:, src[ok], :]
    b1p = None
    if b1 is not None:
        b1p = np.zeros((E, src.shape[0]), dtype=b1.dtype)
        b1p[:, ok] = b1[:, src[ok]]
    return w1p, b1p


def unpack_fc1(w1p, F, h=128):
    """Inverse of repack_fc1 on the weight (padding rows dropped)."""
    src = fc1_packed_columns(F, h)
    E, _, d = w1p.shape
    w1 = np.zeros((E, 2 * F, d), dtype=w1p.dtype)
    ok = src >= 0
    w1[:, src[ok], :] = w1p[:, ok, :]
    return w1


# --------------------------------------------------------------------------
# One expert's MLP (per-group GEMMs of the grouped GEMM) and its backward.
# --------------------------------------------------------------------------

def expert_forward(X, W1, b1, W2, b2, p):
    """X [m,d]; W1 [2F,d] (gated) or [F,d]; W2 [d,F].
    H = X W1^T + b1; A = GLU(H); Y = A W2^T + b2.  Returns H, A, Y."""
    H = X @ W1.T
    if b1 is not None:
        H = H + b1[None, :]
    F = W2.shape[1]
    if p.gated:
        A = glu_forward(H[:, :F], H[:, F:], p)
    else:
        A = glu_forward(H, None, p)
    Y = A @ W2.T
    if b2 is not None:
        Y = Y + b2[None, :]
    return H, A, Y


def expert_backward(X, H, A, dY, W1, W2, p):
    """Backward of expert_forward given dY [m,d].
    Returns dX [m,d], dH, dW1 (shape of W1), db1, dW2 [d,F], db2."""
    F = W2.shape[1]
    dA = dY @ W2
    dW2 = dY.T @ A
    db2 = dY.sum(axis=0)
    if p.gated:
        dG, dL = glu_backward(dA, H[:, :F], H[:, F:], p)
        dH = np.concatenate([dG, dL], axis=1)
    else:
        dH, _ = glu_backward(dA, H, None, p)
    dW1 = dH.T @ X
    db1 = dH.sum(axis=0)
    dX = dH @ W1
    return dX, dH, dW1, db1, dW2, db2


def grouped_forward(x_perm, padded_offsets, counts, W1, b1, W2, b2, p):
    """Grouped FC1/GLU/FC2 over the padded row layout: expert e owns rows
    [padded_offsets[e], padded_offsets[e]+counts[e]).  Padding rows of H, A
    and Y are zero."""
    E = W1.shape[0]
    R_pad = x_perm.shape[0]
    n1 = W1.shape[1]
    F = W2.shape[2]
    d = W2.shape[1]
    H = np.zeros((R_pad, n1))
    A = np.zeros((R_pad, F))
    Y = np.zeros((R_pad, d))
    for e in range(E):
        lo, m = int(padded_offsets[e]), int(counts[e])
        if m == 0:
            continue
        h, a, y = expert_forward(x_perm[lo:lo + m], W1[e],
                                 None if b1 is None else b1[e], W2[e],
                                 None if b2 is None else b2[e], p)
        H[lo:lo + m], A[lo:lo + m], Y[lo:lo + m] = h, a, y
    return H, A, Y


def grouped_backward(x_perm, H, A, dY, padded_offsets, counts, W1, W2, p):
    """Backward of grouped_forward.  Experts with no rows get dW = 0, db = 0."""
    E = W1.shape[0]
    dX = np.zeros_like(x_perm, dtype=np.float64)
    dH = np.zeros_like(H)
    dW1 = np.zeros(W1.shape)
    db1 = np.zeros(W1.shape[:2])
    dW2 = np.zeros(W2.shape)
    db2 = np.zeros(W2.shape[:2])
    for e in range(E):
        lo, m = int(padded_offsets[e]), int(counts[e])
        if m == 0:
            continue
        sl = slice(lo, lo + m)
        dx, dh, dw1, dbb1, dw2, dbb2 = expert_backward(
            x_perm[sl], H[sl], A[sl], dY[sl], W1[e], W2[e], p)
        dX[sl], dH[sl] = dx, dh
        dW1[e], db1[e], dW2[e], db2[e] = dw1, dbb1, dw2, dbb2
    return dX, dH, dW1, db1, dW2, db2


# --------------------------------------------------------------------------
# Weighted unpermute/combine and the backward of routing.
# --------------------------------------------------------------------------

def combine(Y, row_of, topk_w):
    """out[t] = sum over slots s of topk_w[t,s] * Y[row_of[t,s]]."""
    T, k = row_of.shape
    out = np.zeros((T, Y.shape[1]))
    for s in range(k):
        out += topk_w[:, s:s + 1] * Y[row_of[:, s]]
    return out


def combine_backward(dout, Y, row_of, topk_w, R_pad):
    """dY[row_of[t,s]] = topk_w[t,s] * dout[t];  dw[t,s] = <dout[t], Y[row_of[t,s]]>.
    Padding rows of dY are zero."""
    T, k = row_of.shape
    dY = np.zeros((R_pad, dout.shape[1]))
    dw = np.zeros((T, k))
    for s in range(k):
        dY[row_of[:, s]] = topk_w[:, s:s + 1] * dout
        dw[:, s] = np.sum(dout * Y[row_of[:, s]], axis=1)
    return dY, dw


def permute_backward(dX_perm, row_of):
    """dx[t] = sum over slots s of dX_perm[row_of[t,s]]."""
    T, k = row_of.shape
    dx = np.zeros((T, dX_perm.shape[1]))
    for s in range(k):
        dx += dX_perm[row_of[:, s]]
    return dx


def route_backward(dw, topk_w, topk_idx, E):
    """Softmax backward over the selected experts:
    dlogits[t, idx[t,s]] = w[t,s] * (dw[t,s] - sum_s' w[t,s'] dw[t,s']);
    unselected experts (and the selection bias) get 0."""
    T, k = topk_idx.shape
    dl = np.zeros((T, E))
    inner = np.sum(topk_w * dw, axis=1, keepdims=True)
    g = topk_w * (dw - inner)
    for s in range(k):
        dl[np.arange(T), topk_idx[:, s]] = g[:, s]
    return dl


# --------------------------------------------------------------------------
# Whole layer.
# --------------------------------------------------------------------------

def moe_forward(x, logits_f32, bias_f32, W1, b1, W2, b2, k, p, align=128):
    """Routing -> permute -> grouped FC1/GLU/FC2 -> weighted combine.
    x [T,d] fp64; W1 [E,2F,d] logical; W2 [E,d,F].  Returns a dict of every
    intermediate in the padded row layout."""
    E = W1.shape[0]
    topk_idx, topk_w, counts = route(logits_f32, bias_f32, k)
    offsets, padded, tiles = group_offsets(counts, align)
    row_src, row_of = permute_index(topk_idx, E, padded)
    x_perm = gather_rows(x, row_src)
    H, A, Y = grouped_forward(x_perm, padded, counts, W1, b1, W2, b2, p)
    out = combine(Y, row_of, topk_w)
    return dict(topk_idx=topk_idx, topk_w=topk_w, counts=counts, offsets=offsets,
                padded_offsets=padded, tile_prefix=tiles, row_src=row_src,
                row_of=row_of, x_perm=x_perm, H=H, A=A, Y=Y, out=out)


def moe_backward(fwd, dout, W1, W2, p):
    """Backward of moe_forward for the upstream gradient dout [T,d]."""
    E = W1.shape[0]
    R_pad = fwd["x_perm"].shape[0]
    dY, dw = combine_backward(dout, fwd["Y"], fwd["row_of"], fwd["topk_w"], R_pad)
    dX, dH, dW1, db1, dW2, db2 = grouped_backward(
        fwd["x_perm"], fwd["H"], fwd["A"], dY, fwd["padded_offsets"], fwd["counts"],
        W1, W2, p)
    dx = permute_backward(dX, fwd["row_of"])
    dlogits = route_backward(dw, fwd["topk_w"], fwd["topk_idx"], E)
    return dict(dY=dY, dw=dw, dX_perm=dX, dH=dH, dW1=dW1, db1=db1, dW2=dW2,
                db2=db2, dx=dx, dlogits=dlogits)
