"""NVFP4 quantization and the NVFP4 expert MLP (fp64 oracle).

TEST INFRASTRUCTURE ONLY (see the package docstring).

"Improving MoE training throughput with advanced fused kernels", section
"Reducing exposed memory overhead by fusing MXFP8 and NVFP4 quantization":
for NVFP4 the fused kernels emit the BF16 output with its per-tensor amax,
and in the backward the amax of the output's transposed Hadamard rotation;
those amax values set the per-tensor scales with which the tensors are then
quantized for the next NVFP4 GEMMs.

Readings (the pages name NVFP4 and the amax outputs only):

* Value format E2M1 (sign, 2 exponent bits, 1 mantissa bit): +-{0, 0.5, 1,
  1.5, 2, 3, 4, 6}; round to nearest, ties to the even code, saturate at 6.
* Blocks of 16 consecutive elements along a GEMM's contraction axis, each
  with an E4M3 scale; one fp32 encode scale per tensor,
  g = 2688 / amax (2688 = 448 * 6, the largest E4M3 times the largest E2M1;
  g = 1 for an all-zero tensor).
* In fp32, the precision the kernels decide in (so both sides round the same
  values): block scale code = E4M3(RNE, saturating)((amax_b / 6) * g);
  s = its value; codes = E2M1(x * (g / s)) (all zero when s = 0);
  dequantized value = code * s / g.
* Weight-gradient operands (contraction over tokens) are first rotated along
  tokens by H16 / 4 (orthonormal Sylvester Hadamard, no random signs) in
  16-row segments inside each expert group; both operands get the same
  rotation, so their product is unchanged up to quantization, and their
  encode scale uses the amax of the rotated tensor.
"""
import numpy as np

from .mx_oracle import e4m3_decode, e4m3_encode, e4m3_round, hadamard16
from .moe_oracle import glu_backward, glu_forward
from .mx_mlp_oracle import bf16_round

__all__ = ["E2M1_VALUES", "e2m1_round", "e2m1_encode", "nvfp4_global_scale",
           "nvfp4_quantize_rows", "nvfp4_dequantize_rows", "nvfp4_fake_rows", "nvfp4_fake_cols",
           "rht16_rows", "grouped_forward_nv", "grouped_backward_nv"]

E2M1_VALUES = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
_F32 = np.float32


def e2m1_round(y):
    """Nearest E2M1 value (ties to the even code), saturating at +-6."""
    y = np.asarray(y, dtype=np.float64)
    a = np.minimum(np.abs(y), 6.0)
    # candidates: the grid point below and above; ties go to the even code
    idx_hi = np.searchsorted(E2M1_VALUES, a, side="left")
    idx_hi = np.minimum(idx_hi, 7)
    idx_lo = np.maximum(idx_hi - 1, 0)
    lo, hi = E2M1_VALUES[idx_lo], E2M1_VALUES[idx_hi]
    d_lo, d_hi = a - lo, hi - a
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (idx_hi % 2 == 0) & (idx_hi != idx_lo))
    mag = np.where(pick_hi, hi, lo)
    return np.copysign(mag, y)


def e2m1_encode(v):
    """4-bit codes (sign bit 3, magnitude index 0..7) of E2M1 values."""
    v = np.asarray(v, dtype=np.float64)
    mag = np.searchsorted(E2M1_VALUES, np.abs(v))
    assert np.all(E2M1_VALUES[mag] == np.abs(v)), "not an E2M1 value"
    return (mag | (np.signbit(v).astype(np.int64) << 3)).astype(np.uint8)


def nvfp4_global_scale(amax):
    """fp32 encode scale 2688 / amax (1 for amax 0)."""
    amax = _F32(amax)
    return _F32(1.0) if amax == 0 else _F32(_F32(2688.0) / amax)


def nvfp4_quantize_rows(v, g):
    """Blocks of 16 along the last axis of fp32 values v [rows, cols]
    (cols % 16 == 0) with encode scale g.  Returns E2M1 values [rows, cols]
    (fp64), E4M3 scale codes uint8 [rows, cols/16] and their values."""
    v = np.asarray(v, dtype=_F32)
    rows, cols = v.shape
    blk = v.reshape(rows, cols // 16, 16)
    amax = np.max(np.abs(blk), axis=-1).astype(_F32)
    target = ((amax / _F32(6.0)).astype(_F32) * _F32(g)).astype(_F32)
    s = e4m3_round(target.astype(np.float64))            # RNE, saturating at 448
    codes = e4m3_encode(s)
    s32 = s.astype(_F32)
    with np.errstate(divide="ignore", invalid="ignore"):
        inv = np.where(s32 > 0, (_F32(g) / s32).astype(_F32), _F32(0))
    y = (blk * inv[..., None]).astype(_F32)
    q = e2m1_round(y.astype(np.float64))
    return q.reshape(rows, cols), codes, s


def nvfp4_dequantize_rows(q, s, g):
    rows, cols = q.shape
    return (q.reshape(rows, cols // 16, 16) * (np.asarray(s, np.float64) / float(g))[..., None]
            ).reshape(rows, cols)


def nvfp4_fake_rows(v, amax=None):
    """Quantize-dequantize along the last axis with the tensor's own encode
    scale (from amax, default max|v|)."""
    v = np.asarray(v, dtype=np.float64)
    a = float(np.max(np.abs(v))) if amax is None else float(amax)
    g = nvfp4_global_scale(a)
    shp = v.shape
    q, _, s = nvfp4_quantize_rows(v.reshape(-1, shp[-1]).astype(_F32), g)
    return nvfp4_dequantize_rows(q, s, g).reshape(shp)


def nvfp4_fake_cols(v, amax=None):
    """Quantize-dequantize with blocks of 16 rows down each column."""
    return nvfp4_fake_rows(np.asarray(v, np.float64).T, amax).T


def rht16_rows(v):
    """H16/4 applied to every 16-row segment of each column of v [rows, cols]
    (rows % 16 == 0)."""
    v = np.asarray(v, dtype=np.float64)
    H = hadamard16() / 4.0
    seg = v.reshape(v.shape[0] // 16, 16, v.shape[1])
    return np.einsum("ij,sjc->sic", H, seg).reshape(v.shape)


def _pad16(v):
    out = np.zeros(((v.shape[0] + 15) // 16 * 16,) + v.shape[1:])
    out[:v.shape[0]] = v
    return out


def _groups(padded_offsets, counts):
    return [(e, int(padded_offsets[e]), int(counts[e])) for e in range(len(counts))
            if int(counts[e]) > 0]


def _amax(parts):
    return max([float(np.max(np.abs(p))) for p in parts if p.size] + [0.0])


def grouped_forward_nv(x_perm, padded_offsets, counts, W1, b1, W2, b2, p):
    """NVFP4 grouped FC1/GLU/FC2: X and W1 quantized along d, A (bf16) and W2
    along F, each with its tensor's encode scale (amax over all experts /
    rows).  W1 logical [E, 2F, d] (gated) or [E, F, d].  Returns H (bf16), A
    (bf16), Y; padding rows zero."""
    E = W1.shape[0]
    F, d = W2.shape[2], W2.shape[1]
    gs = _groups(padded_offsets, counts)
    ax = _amax([x_perm[lo:lo + m] for _, lo, m in gs])
    aw1, aw2 = float(np.max(np.abs(W1))), float(np.max(np.abs(W2)))
    H = np.zeros((x_perm.shape[0], W1.shape[1]))
    A = np.zeros((x_perm.shape[0], F))
    Y = np.zeros((x_perm.shape[0], d))
    for e, lo, m in gs:
        h = nvfp4_fake_rows(x_perm[lo:lo + m], ax) @ nvfp4_fake_rows(W1[e], aw1).T
        if b1 is not None:
            h = h + b1[e][None, :]
        a = glu_forward(h[:, :F], h[:, F:], p) if p.gated else glu_forward(h, None, p)
        H[lo:lo + m], A[lo:lo + m] = bf16_round(h), bf16_round(a)
    aa = _amax([A[lo:lo + m] for _, lo, m in gs])
    for e, lo, m in gs:
        y = nvfp4_fake_rows(A[lo:lo + m], aa) @ nvfp4_fake_rows(W2[e], aw2).T
        if b2 is not None:
            y = y + b2[e][None, :]
        Y[lo:lo + m] = y
    return H, A, Y


def grouped_backward_nv(x_perm, H, A, dY, padded_offsets, counts, W1, W2, p):
    """Backward of grouped_forward_nv for bf16 dY.  dgrads: dY and W2 along d,
    dH (bf16) and W1 along the FC1 width; weight gradients: both operands
    rotated by H16/4 along the group's rows and quantized in those 16-row
    blocks, with the rotated tensors' encode scales."""
    E = W1.shape[0]
    F = W2.shape[2]
    gs = _groups(padded_offsets, counts)
    aw1, aw2 = float(np.max(np.abs(W1))), float(np.max(np.abs(W2)))
    ady = _amax([dY[lo:lo + m] for _, lo, m in gs])
    dX = np.zeros(x_perm.shape)
    dH = np.zeros(H.shape)
    for e, lo, m in gs:
        da = nvfp4_fake_rows(dY[lo:lo + m], ady) @ nvfp4_fake_cols(W2[e], aw2)
        if p.gated:
            dg, dl = glu_backward(da, H[lo:lo + m, :F], H[lo:lo + m, F:], p)
            dH[lo:lo + m] = bf16_round(np.concatenate([dg, dl], axis=1))
        else:
            dH[lo:lo + m] = bf16_round(glu_backward(da, H[lo:lo + m], None, p)[0])
    adh = _amax([dH[lo:lo + m] for _, lo, m in gs])
    for e, lo, m in gs:
        dX[lo:lo + m] = nvfp4_fake_rows(dH[lo:lo + m], adh) @ nvfp4_fake_cols(W1[e], aw1)
    rot = {name: {e: rht16_rows(_pad16(T[lo:lo + m])) for e, lo, m in gs}
           for name, T in (("dY", dY), ("A", A), ("dH", dH), ("X", x_perm))}
    ramax = {name: _amax(list(r.values())) for name, r in rot.items()}
    dW1 = np.zeros(W1.shape)
    dW2 = np.zeros(W2.shape)
    db1 = np.zeros(W1.shape[:2])
    db2 = np.zeros(W2.shape[:2])
    for e, lo, m in gs:
        q = {n: nvfp4_fake_cols(rot[n][e], ramax[n]) for n in rot}
        dW2[e] = q["dY"].T @ q["A"]
        dW1[e] = q["dH"].T @ q["X"]
        db2[e] = dY[lo:lo + m].sum(axis=0)
        db1[e] = dH[lo:lo + m].sum(axis=0)
    return dX, dH, dW1, db1, dW2, db2
