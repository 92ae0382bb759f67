"""Runs one synthetic layer through the CUDA library and through the oracle
on the same seeded inputs, and compares the results.

The CUDA side goes through the C-ABI (via the thin binding); the oracle side
is the fp64 CPU oracle.  The two share only the input generator.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from workloads import bf16_bits_to_f64

TOL_REL = 1e-2      # max|gpu - ref| <= 1e-2 * max|ref| + 1e-3 (bf16 path)
TOL_ABS = 1e-3


def bits_to_dev(bits, device="cuda"):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)


def to_np(t):
    if t.dtype == torch.bfloat16:
        return t.float().cpu().numpy().astype(np.float64)
    return t.cpu().numpy()


def assert_close(name, got, ref, rel=TOL_REL, abs_=TOL_ABS):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (name, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{name}: non-finite values"
    err = float(np.max(np.abs(got - ref))) if got.size else 0.0
    bound = rel * (float(np.max(np.abs(ref))) if ref.size else 0.0) + abs_
    assert err <= bound, f"{name}: max err {err:.3e} > bound {bound:.3e}"
    return err, bound


def glu_params(wl):
    return oracle.GluParams(wl.act, wl.alpha, wl.limit, wl.linear_offset, wl.out_scale)


def oracle_weights(inp):
    W1 = bf16_bits_to_f64(inp["w1"])
    W2 = bf16_bits_to_f64(inp["w2"])
    b1 = bf16_bits_to_f64(inp["b1"]) if inp["b1"] is not None else None
    b2 = bf16_bits_to_f64(inp["b2"]) if inp["b2"] is not None else None
    return W1, b1, W2, b2


def run_oracle_routed(wl, inp):
    p = glu_params(wl)
    W1, b1, W2, b2 = oracle_weights(inp)
    x = bf16_bits_to_f64(inp["x"])
    fwd = oracle.moe_forward(x, inp["logits"], inp["bias"], W1, b1, W2, b2, wl.k, p, align=128)
    bwd = oracle.moe_backward(fwd, bf16_bits_to_f64(inp["dout"]), W1, W2, p)
    return fwd, bwd


def make_layer(wl, **kw):
    """A layer for the workload; the parity tests compare the bf16 A and dH
    too, so they are kept on every path unless the caller says otherwise."""
    from moe_expert_mlp_gb300 import MoEExpertMLP
    kw.setdefault("keep_bf16_copies", True)
    return MoEExpertMLP(wl.E, wl.d, wl.F, T=wl.T, k=wl.k, act=wl.act, alpha=wl.alpha,
                        limit=wl.limit, linear_offset=wl.linear_offset, out_scale=wl.out_scale,
                        has_b1=wl.has_b1, has_b2=wl.has_b2, **kw)


def load_layer_weights(layer, inp):
    w1 = bits_to_dev(inp["w1"])
    w2 = bits_to_dev(inp["w2"])
    b1 = bits_to_dev(inp["b1"]) if inp["b1"] is not None else None
    b2 = bits_to_dev(inp["b2"]) if inp["b2"] is not None else None
    layer.load_weights(w1, b1, w2, b2)


def run_gpu_routed(wl, inp, layer=None, **kw):
    layer = layer or make_layer(wl, **kw)
    load_layer_weights(layer, inp)
    x = bits_to_dev(inp["x"])
    logits = torch.from_numpy(inp["logits"]).cuda()
    bias = torch.from_numpy(inp["bias"]).cuda() if inp["bias"] is not None else None
    dout = bits_to_dev(inp["dout"])
    layer.step(x, logits, bias, dout)
    torch.cuda.synchronize()
    return layer


def padded_rows(rows_bits, sizes, padded_offsets, width):
    """Place rows given in expert order into the padded layout (input prep
    for workloads whose groups are given directly)."""
    R_pad = int(padded_offsets[-1])
    out = np.zeros((R_pad, width), dtype=np.uint16)
    src = 0
    for e, m in enumerate(sizes):
        lo = int(padded_offsets[e])
        out[lo:lo + m] = rows_bits[src:src + m]
        src += m
    return out


def run_both_direct(wl, inp):
    """Groups given directly: x rows and dY rows in expert order."""
    sizes = inp["group_sizes"]
    p = glu_params(wl)
    W1, b1, W2, b2 = oracle_weights(inp)
    offsets, padded, tiles = oracle.group_offsets(sizes, align=128)
    xp_bits = padded_rows(inp["x"], sizes, padded, wl.d)
    dy_bits = padded_rows(inp["dout"], sizes, padded, wl.d)
    xp = bf16_bits_to_f64(xp_bits)
    dyp = bf16_bits_to_f64(dy_bits)
    H, A, Y = oracle.grouped_forward(xp, padded, sizes, W1, b1, W2, b2, p)
    dX, dH, dW1, db1, dW2, db2 = oracle.grouped_backward(xp, H, A, dyp, padded, sizes, W1, W2, p)
    ref = dict(H=H, A=A, Y=Y, dX_perm=dX, dH=dH, dW1=dW1, db1=db1, dW2=dW2, db2=db2,
               padded_offsets=padded, offsets=offsets, tile_prefix=tiles, counts=sizes)

    cap = max(128, int(padded[-1]))
    layer = make_layer(wl, capacity=cap)
    load_layer_weights(layer, inp)
    layer.set_groups(torch.from_numpy(sizes.astype(np.int32)).cuda())
    R_pad = int(padded[-1])
    layer.x_perm[:R_pad].copy_(bits_to_dev(xp_bits))
    layer.dy[:R_pad].copy_(bits_to_dev(dy_bits))
    layer.mlp_forward()
    layer.mlp_backward()
    torch.cuda.synchronize()
    return layer, ref


def packed_to_logical_cols(t_np, F):
    """GPU packed FC1-shaped columns -> logical (gate then linear) columns;
    also returns the packed padding columns for a zero check.  A tensor F
    wide is the non-gated activation's, which is not packed."""
    if t_np.shape[-1] == F:
        return t_np, t_np[..., :0]
    src = oracle.fc1_packed_columns(F)
    out = np.zeros(t_np.shape[:-1] + (2 * F,))
    ok = src >= 0
    out[..., src[ok]] = t_np[..., ok]
    return out, t_np[..., ~ok]


# --------------------------------------------------------------------------
# MXFP8 path
# --------------------------------------------------------------------------
TOL_MX = 6e-2       # the MXFP8 path's tolerance (met here with the bf16 bound, below)
# Against the unquantized fp64 oracle the MXFP8 format's own error (E4M3
# payloads with 3 mantissa bits, chained through H -> A -> Y and dY -> dA ->
# dH) is 6-8 % in relative Frobenius norm on these layers and reaches 15 %
# of max|ref| in single elements (a block maximum saturated at 448 by the
# OCP floor scale).  That comparison is a format sanity bound, which a
# wiring error (a dropped K block, a wrong scale atom) exceeds by far; the
# kernel check is the quantization-matched one.
TOL_MX_FRO = 1e-1

# Achieved error ratios of the MXFP8 checks, printed at the end of the run
# (tests/conftest.py): (name, max err / max|ref| against the oracle with the
# same MXFP8 quantization, relative Frobenius error against the unquantized
# oracle).
MX_RATIOS = []
# Achieved max err / max|ref| of the fp32 (TF32 tensor core) checks against
# the fp64 oracle on the same fp32 inputs, printed with the above.
TF32_RATIOS = []


def assert_mx(name, got, ref_mx, ref_plain=None):
    """An output of the MXFP8 path.  Against the oracle that quantizes the
    same operands the same way, the only differences are fp32 accumulation
    order, the bf16 rounding of stored tensors, and rare single-code flips
    where an intermediate the GPU re-quantizes (A, dH) lands one bf16 ulp
    away from the oracle's on the other side of an E4M3 rounding point: the
    bf16 bound applies.  Against the unquantized fp64 oracle the format's
    own error is bounded in relative Frobenius norm by TOL_MX_FRO."""
    err, _ = assert_close(name, got, ref_mx)
    scale = float(np.max(np.abs(ref_mx))) if np.size(ref_mx) else 0.0
    r_u = None
    if ref_plain is not None:
        g = np.asarray(got, dtype=np.float64)
        r = np.asarray(ref_plain, dtype=np.float64)
        assert g.shape == r.shape, (name, g.shape, r.shape)
        nr = float(np.linalg.norm(r))
        r_u = float(np.linalg.norm(g - r)) / nr if nr > 0 else 0.0
        assert r_u <= TOL_MX_FRO, f"{name} vs unquantized: relative Frobenius {r_u:.3e}"
    MX_RATIOS.append((name, err / scale if scale > 0 else 0.0, r_u))


def mma_scales_to_rowmajor(buf, rows, cols):
    """Scales stored in the MMA layout (include/moe.h, MOE_MX_SCALES_MMA)
    -> [rows, cols/32] row-major, by the layout's index formula."""
    buf = np.asarray(buf).reshape(-1)
    ra = 2 * ((rows + 255) // 256)
    r = np.arange(rows)[:, None]
    j = np.arange(cols // 32)[None, :]
    off = ((j // 4) * ra + r // 128) * 512 + (r % 32) * 16 + ((r // 32) % 4) * 4 + j % 4
    return buf[off]


def run_oracle_routed_mx(wl, inp):
    """The routed layer with the MXFP8 expert MLP: routing, permute, combine
    and their backward as in the bf16 oracle; dY rounded to bf16 (the stored
    tensor the quantizer reads) before the MXFP8 backward."""
    p = glu_params(wl)
    W1, b1, W2, b2 = oracle_weights(inp)
    x = bf16_bits_to_f64(inp["x"])
    topk_idx, topk_w, counts = oracle.route(inp["logits"], inp["bias"], wl.k)
    offsets, padded, tiles = oracle.group_offsets(counts, 128)
    row_src, row_of = oracle.permute_index(topk_idx, wl.E, padded)
    xp = oracle.gather_rows(x, row_src)
    H, A, Y = oracle.grouped_forward_mx(xp, padded, counts, W1, b1, W2, b2, p)
    out = oracle.combine(Y, row_of, topk_w)
    dY, dw = oracle.combine_backward(bf16_bits_to_f64(inp["dout"]), Y, row_of, topk_w,
                                     xp.shape[0])
    dY16 = oracle.bf16_round(dY)
    dX, dH, dW1, db1, dW2, db2 = oracle.grouped_backward_mx(xp, H, A, dY16, padded, counts,
                                                           W1, W2, p)
    dx = oracle.permute_backward(dX, row_of)
    dlogits = oracle.route_backward(dw, topk_w, topk_idx, wl.E)
    return dict(topk_idx=topk_idx, counts=counts, padded_offsets=padded, x_perm=xp, H=H, A=A,
                Y=Y, out=out, dY=dY16, dw=dw, dX_perm=dX, dH=dH, dW1=dW1, db1=db1, dW2=dW2,
                db2=db2, dx=dx, dlogits=dlogits)


def run_both_direct_mx(wl, inp):
    """Groups given directly, MXFP8 expert MLP on both sides."""
    sizes = inp["group_sizes"]
    p = glu_params(wl)
    W1, b1, W2, b2 = oracle_weights(inp)
    offsets, padded, tiles = oracle.group_offsets(sizes, align=128)
    xp_bits = padded_rows(inp["x"], sizes, padded, wl.d)
    dy_bits = padded_rows(inp["dout"], sizes, padded, wl.d)
    xp = bf16_bits_to_f64(xp_bits)
    dyp = bf16_bits_to_f64(dy_bits)
    H, A, Y = oracle.grouped_forward_mx(xp, padded, sizes, W1, b1, W2, b2, p)
    dX, dH, dW1, db1, dW2, db2 = oracle.grouped_backward_mx(xp, H, A, dyp, padded, sizes, W1,
                                                           W2, p)
    ref = dict(H=H, A=A, Y=Y, dX_perm=dX, dH=dH, dW1=dW1, db1=db1, dW2=dW2, db2=db2,
               padded_offsets=padded, counts=sizes)
    cap = max(128, int(padded[-1]))
    layer = make_layer(wl, capacity=cap, dtype="mxfp8")
    load_layer_weights(layer, inp)
    layer.set_groups(torch.from_numpy(sizes.astype(np.int32)).cuda())
    R_pad = int(padded[-1])
    layer.x_perm[:R_pad].copy_(bits_to_dev(xp_bits))
    layer.dy[:R_pad].copy_(bits_to_dev(dy_bits))
    layer.mlp_forward()
    layer.mlp_backward()
    torch.cuda.synchronize()
    return layer, ref


# ------------------------------------------------------------------ NVFP4
TOL_NV = 0.1        # max|gpu - ref| <= 0.1 * max|ref| downstream of a requantized intermediate
TOL_NV_FRO = 2e-2   # and ||gpu - ref||_F <= 2e-2 ||ref||_F

E2M1_SIGNED = np.array([0, .5, 1, 1.5, 2, 3, 4, 6, 0, -.5, -1, -1.5, -2, -3, -4, -6])


def unpack_fp4_codes(q):
    """Packed E2M1 bytes [..., n/2] -> 4-bit codes [..., n] (element 2i in
    the low nibble)."""
    q = np.asarray(q, dtype=np.uint8)
    out = np.empty(q.shape[:-1] + (2 * q.shape[-1],), dtype=np.uint8)
    out[..., 0::2] = q & 0xF
    out[..., 1::2] = q >> 4
    return out


def nv_scales_to_rowmajor(buf, rows, cols):
    """NVFP4 scales in the MMA layout (16-element blocks) -> [rows, cols/16]."""
    buf = np.asarray(buf).reshape(-1)
    ra = 2 * ((rows + 255) // 256)
    r = np.arange(rows)[:, None]
    j = np.arange(cols // 16)[None, :]
    off = ((j // 4) * ra + r // 128) * 512 + (r % 32) * 16 + ((r // 32) % 4) * 4 + j % 4
    return buf[off]


def nv_dequant(q, scale_buf, amax, rows, cols):
    """Values of an NVFP4 tensor [rows, cols] as the GPU encoded it (codes,
    UE4M3 scales in the MMA layout, encode amax), decoded with the oracle's
    formula value = code * s / g."""
    codes = unpack_fp4_codes(np.asarray(q).reshape(rows, cols // 2))
    s = oracle.e4m3_decode(nv_scales_to_rowmajor(scale_buf, rows, cols))
    g = oracle.nvfp4_global_scale(float(amax))
    return oracle.nvfp4_dequantize_rows(E2M1_SIGNED[codes], s, g)


def run_both_direct_nv(wl, inp):
    """Groups given directly, NVFP4 expert MLP on both sides."""
    sizes = inp["group_sizes"]
    p = glu_params(wl)
    W1, b1, W2, b2 = oracle_weights(inp)
    offsets, padded, tiles = oracle.group_offsets(sizes, align=128)
    xp_bits = padded_rows(inp["x"], sizes, padded, wl.d)
    dy_bits = padded_rows(inp["dout"], sizes, padded, wl.d)
    xp = bf16_bits_to_f64(xp_bits)
    dyp = bf16_bits_to_f64(dy_bits)
    H, A, Y = oracle.grouped_forward_nv(xp, padded, sizes, W1, b1, W2, b2, p)
    dX, dH, dW1, db1, dW2, db2 = oracle.grouped_backward_nv(xp, H, A, dyp, padded, sizes, W1,
                                                           W2, p)
    ref = dict(H=H, A=A, Y=Y, dX_perm=dX, dH=dH, dW1=dW1, db1=db1, dW2=dW2, db2=db2,
               padded_offsets=padded, counts=sizes)
    cap = max(128, int(padded[-1]))
    layer = make_layer(wl, capacity=cap, dtype="nvfp4")
    load_layer_weights(layer, inp)
    layer.set_groups(torch.from_numpy(sizes.astype(np.int32)).cuda())
    R_pad = int(padded[-1])
    layer.x_perm[:R_pad].copy_(bits_to_dev(xp_bits))
    layer.dy[:R_pad].copy_(bits_to_dev(dy_bits))
    layer.mlp_forward()
    layer.mlp_backward()
    torch.cuda.synchronize()
    return layer, ref


def run_oracle_routed_nv(wl, inp):
    """The routed layer with the NVFP4 expert MLP: routing, permute, combine
    and their backward as in the bf16 oracle; dY rounded to bf16 (the stored
    tensor the quantizer reads) before the NVFP4 backward."""
    p = glu_params(wl)
    W1, b1, W2, b2 = oracle_weights(inp)
    x = bf16_bits_to_f64(inp["x"])
    topk_idx, topk_w, counts = oracle.route(inp["logits"], inp["bias"], wl.k)
    offsets, padded, tiles = oracle.group_offsets(counts, 128)
    row_src, row_of = oracle.permute_index(topk_idx, wl.E, padded)
    xp = oracle.gather_rows(x, row_src)
    H, A, Y = oracle.grouped_forward_nv(xp, padded, counts, W1, b1, W2, b2, p)
    out = oracle.combine(Y, row_of, topk_w)
    dY, dw = oracle.combine_backward(bf16_bits_to_f64(inp["dout"]), Y, row_of, topk_w,
                                     xp.shape[0])
    dY16 = oracle.bf16_round(dY)
    dX, dH, dW1, db1, dW2, db2 = oracle.grouped_backward_nv(xp, H, A, dY16, padded, counts,
                                                           W1, W2, p)
    dx = oracle.permute_backward(dX, row_of)
    dlogits = oracle.route_backward(dw, topk_w, topk_idx, wl.E)
    return dict(topk_idx=topk_idx, counts=counts, padded_offsets=padded, x_perm=xp, H=H, A=A,
                Y=Y, out=out, dY=dY16, dw=dw, dX_perm=dX, dH=dH, dW1=dW1, db1=db1, dW2=dW2,
                db2=db2, dx=dx, dlogits=dlogits)
