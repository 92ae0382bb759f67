"""fp64 oracle of the MXFP8 expert MLP (forward and backward).

TEST INFRASTRUCTURE ONLY (see the package docstring).

"Improving MoE training throughput with advanced fused kernels", sections
"Reducing exposed memory overhead by fusing MXFP8 and NVFP4 quantization"
and "Optimizing GLU activations with fused GEMM epilogues": the GEMMs of the
MoE block consume MXFP8 operands (E4M3 payload, one E8M0 scale per 32
elements), the activation output is written in MXFP8 for the next GEMM
together with a transposed MXFP8 copy for the backward, and the backward's
dSwiGLU epilogue quantizes its output the same way.

Readings (the pages name the format and which tensors are quantized, not the
arithmetic around it):

* Every GEMM operand is quantized along that GEMM's contraction (K) axis, as
  block scaling requires: FC1 X and W1 along d; FC2 A and W2 along F; FC2
  dgrad dY along d and W2 along d; FC1 dgrad dH and W1 along 2F; the weight
  gradients take both operands along the tokens of one expert group, in
  32-row blocks of the padded layout (groups start at multiples of 128, so a
  block never spans two experts; rows past the group's count are zero).
* The quantizer reads what the GPU stores: H, A and dH are rounded to bf16
  first (RNE), A is computed from the unrounded H, the dGLU reads the stored
  bf16 H.  dY arrives in bf16.
* Bias gradients are sums of the bf16 dY / dH rows (no quantization).
* Accumulation is exact here (fp64); the GPU accumulates in fp32.
"""
import numpy as np

from .moe_oracle import glu_backward, glu_forward
from .mx_oracle import e4m3_decode, mx_quantize_rows

__all__ = ["bf16_round", "mx_fake_rows", "mx_fake_cols", "expert_forward_mx",
           "expert_backward_mx", "grouped_forward_mx", "grouped_backward_mx"]


def bf16_round(v):
    """Round fp64 values to the nearest bf16 value, ties to even (8
    significant bits).  Finite normal range only (no bf16 subnormals or
    overflow occur in the workloads)."""
    v = np.asarray(v, dtype=np.float64)
    m, e = np.frexp(v)                       # v = m * 2^e, 0.5 <= |m| < 1
    return np.ldexp(np.rint(np.ldexp(m, 8)), e - 8)


def mx_fake_rows(v):
    """Quantize to MXFP8 with blocks along the last axis and dequantize:
    each value becomes decode(code) * 2^(scale - 127)."""
    v = np.asarray(v, dtype=np.float64)
    shp = v.shape
    flat = v.reshape(-1, shp[-1])
    codes, sc = mx_quantize_rows(flat.astype(np.float32))
    rows, cols = codes.shape
    val = e4m3_decode(codes).reshape(rows, cols // 32, 32)
    val = val * np.exp2(sc.astype(np.float64) - 127.0)[..., None]
    return val.reshape(shp)


def mx_fake_cols(v):
    """Quantize-dequantize with blocks of 32 consecutive rows down each
    column of v [rows, cols] (rows % 32 == 0)."""
    return mx_fake_rows(np.asarray(v, dtype=np.float64).T).T


def _pad_rows32(v):
    m = v.shape[0]
    out = np.zeros(((m + 31) // 32 * 32, v.shape[1]))
    out[:m] = v
    return out


def expert_forward_mx(X, W1, b1, W2, b2, p):
    """One expert.  X [m,d] bf16 values; W1 [2F,d] (logical gate | linear
    rows; [F,d] for the non-gated activation), W2 [d,F].  Returns H (bf16), A (bf16), Y (fp64, before the bf16
    store)."""
    F = W2.shape[1]
    H = mx_fake_rows(X) @ mx_fake_rows(W1).T
    if b1 is not None:
        H = H + b1[None, :]
    A = glu_forward(H[:, :F], H[:, F:], p) if p.gated else glu_forward(H, None, p)
    A16 = bf16_round(A)
    Y = mx_fake_rows(A16) @ mx_fake_rows(W2).T
    if b2 is not None:
        Y = Y + b2[None, :]
    return bf16_round(H), A16, Y


def expert_backward_mx(X, H16, A16, dY, W1, W2, p):
    """Backward of expert_forward_mx for dY [m,d] (bf16 values), given the
    stored bf16 H and A.  Returns dX, dH (bf16), dW1, db1, dW2, db2."""
    F = W2.shape[1]
    m = X.shape[0]
    dA = mx_fake_rows(dY) @ mx_fake_cols(W2)             # K = d
    if p.gated:
        dG, dL = glu_backward(dA, H16[:, :F], H16[:, F:], p)
        dH16 = bf16_round(np.concatenate([dG, dL], axis=1))
    else:
        dH16 = bf16_round(glu_backward(dA, H16, None, p)[0])
    dX = mx_fake_rows(dH16) @ mx_fake_cols(W1)           # K = 2F
    # weight gradients: K = the group's tokens, 32-row blocks from its start
    dW2 = mx_fake_cols(_pad_rows32(dY)).T @ mx_fake_cols(_pad_rows32(A16))
    dW1 = mx_fake_cols(_pad_rows32(dH16)).T @ mx_fake_cols(_pad_rows32(X))
    db2 = dY[:m].sum(axis=0)
    db1 = dH16.sum(axis=0)
    return dX, dH16, dW1, db1, dW2, db2


def grouped_forward_mx(x_perm, padded_offsets, counts, W1, b1, W2, b2, p):
    """MXFP8 grouped FC1/GLU/FC2 over the padded row layout (expert e owns
    rows [padded_offsets[e], padded_offsets[e] + counts[e])).  W1 is logical
    [E, 2F, d].  Returns H, A (bf16 values), Y; padding rows are zero."""
    E = W1.shape[0]
    R_pad = x_perm.shape[0]
    F, d = W2.shape[2], W2.shape[1]
    H = np.zeros((R_pad, W1.shape[1]))
    A = np.zeros((R_pad, F))
    Y = np.zeros((R_pad, d))
    for e in range(E):
        lo, m = int(padded_offsets[e]), int(counts[e])
        if m == 0:
            continue
        h, a, y = expert_forward_mx(x_perm[lo:lo + m], W1[e], None if b1 is None else b1[e],
                                    W2[e], None if b2 is None else b2[e], p)
        H[lo:lo + m], A[lo:lo + m], Y[lo:lo + m] = h, a, y
    return H, A, Y


def grouped_backward_mx(x_perm, H, A, dY, padded_offsets, counts, W1, W2, p):
    """Backward of grouped_forward_mx.  Experts with no rows get dW = 0."""
    E = W1.shape[0]
    dX = np.zeros(x_perm.shape)
    dH = np.zeros(H.shape)
    dW1 = np.zeros(W1.shape)
    db1 = np.zeros(W1.shape[:2])
    dW2 = np.zeros(W2.shape)
    db2 = np.zeros(W2.shape[:2])
    for e in range(E):
        lo, m = int(padded_offsets[e]), int(counts[e])
        if m == 0:
            continue
        sl = slice(lo, lo + m)
        dx, dh, dw1, dbb1, dw2, dbb2 = expert_backward_mx(x_perm[sl], H[sl], A[sl], dY[sl],
                                                          W1[e], W2[e], p)
        dX[sl], dH[sl] = dx, dh
        dW1[e], db1[e], dW2[e], db2[e] = dw1, dbb1, dw2, dbb2
    return dX, dH, dW1, db1, dW2, db2
