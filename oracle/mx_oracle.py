"""MXFP8 quantization and NVFP4 amax preparation in fp64.  Test
infrastructure only (see the package header).

Improving MoE training throughput..., "Reducing exposed memory overhead by
fusing MXFP8 and NVFP4 quantization": for MXFP8 the activation output is
written in MXFP8 plus a transposed MXFP8 copy for the backward; for NVFP4 the
kernel writes a per-tensor amax of the output and, in the backward, the amax
of the transposed Hadamard-rotated output.  The pages only name the formats;
the definitions below are the OCP Microscaling (MX) v1.0 ones:

* block of 32 consecutive elements along the contraction dimension;
* shared scale X = 2^(floor(log2(amax)) - 8), 8 being E4M3's largest
  exponent, exponent clamped to [-127, 127], stored as E8M0 (exponent+127);
  a block of zeros gets code 0;
* payload E4M3 (1 sign, 4 exponent bits with bias 7, 3 mantissa bits,
  subnormals kept, largest finite 448): v/X rounded to nearest, ties to an
  even mantissa, saturated to +-448; the sign of zero is kept.
"""
from __future__ import annotations

import math

import numpy as np

__all__ = [
    "E4M3_MAX", "e4m3_round", "e4m3_encode", "e4m3_decode", "mx_scale_exponent",
    "mx_quantize_rows", "mx_quantize_cols", "mx_dequantize_rows",
    "hadamard16", "amax_plain", "amax_hadamard_t",
]

E4M3_MAX = 448.0
_E4M3_EMIN = -6          # smallest normal exponent
_E4M3_MBITS = 3
_E4M3_EMAX = 8


def e4m3_round(y):
    """Round fp64 values to the E4M3 grid: nearest, ties to even mantissa,
    saturating at +-448.  Signed zeros are kept."""
    y = np.asarray(y, dtype=np.float64)
    a = np.abs(y)
    # exponent of the binade each value falls in (normal range), else the
    # subnormal quantum 2^(emin - mbits)
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.maximum(e, _E4M3_EMIN)
    q = np.exp2(e - _E4M3_MBITS)
    # np.round rounds halves to even; a/q is exact (power-of-two scaling)
    r = np.round(a / q) * q
    r = np.minimum(r, E4M3_MAX)
    return np.copysign(r, y)


def e4m3_encode(v):
    """Bit pattern (uint8) of E4M3-representable fp64 values."""
    v = np.asarray(v, dtype=np.float64)
    sign = np.signbit(v).astype(np.uint8) << 7
    a = np.abs(v)
    code = np.zeros(v.shape, dtype=np.uint8)
    sub = a < 2.0 ** _E4M3_EMIN
    mant_sub = np.round(a / 2.0 ** (_E4M3_EMIN - _E4M3_MBITS)).astype(np.int64)
    code[sub] = mant_sub[sub].astype(np.uint8)
    nrm = ~sub
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(nrm, a, 1.0))).astype(np.int64)
    mant = np.round((a / np.exp2(e) - 1.0) * 8).astype(np.int64)
    code[nrm] = (((e[nrm] + 7) << 3) | mant[nrm]).astype(np.uint8)
    return code | sign


def e4m3_decode(code):
    """fp64 value of each finite E4M3 bit pattern (0x7F/0xFF are NaN)."""
    c = np.asarray(code, dtype=np.int64)
    s = np.where(c & 0x80, -1.0, 1.0)
    ef = (c >> 3) & 0xF
    m = c & 0x7
    val = np.where(ef == 0, m * 2.0 ** (_E4M3_EMIN - _E4M3_MBITS),
                   (1.0 + m / 8.0) * np.exp2(ef - 7.0))
    val = np.where((ef == 0xF) & (m == 0x7), np.nan, val)
    return s * val


def mx_scale_exponent(amax):
    """floor(log2(amax)) - 8, clamped to [-127, 127]; -127 for amax == 0."""
    amax = np.asarray(amax, dtype=np.float64)
    out = np.full(amax.shape, -127, dtype=np.int64)
    pos = amax > 0
    mant, ex = np.frexp(amax[pos])         # amax = mant * 2^ex, mant in [0.5, 1)
    out[pos] = np.clip(ex - 1 - _E4M3_EMAX, -127, 127)
    return out


def _quantize_blocks(v):
    """v [..., nblk, 32] -> codes uint8 same shape, E8M0 scales [..., nblk]."""
    amax = np.max(np.abs(v), axis=-1)
    ex = mx_scale_exponent(amax)
    y = v / np.exp2(ex)[..., None]
    codes = e4m3_encode(e4m3_round(y))
    return codes, (ex + 127).astype(np.uint8)


def mx_quantize_rows(v):
    """Rowwise MXFP8 of fp32 values v [rows, cols] (cols % 32 == 0): blocks run
    along each row.  Returns codes uint8 [rows, cols], scales uint8 [rows, cols/32]."""
    v = np.asarray(v, dtype=np.float32).astype(np.float64)
    rows, cols = v.shape
    assert cols % 32 == 0
    codes, sc = _quantize_blocks(v.reshape(rows, cols // 32, 32))
    return codes.reshape(rows, cols), sc


def mx_quantize_cols(v):
    """Columnwise MXFP8 written transposed: blocks of 32 run down each column
    (along rows/tokens).  v [rows, cols] with rows % 32 == 0.  Returns
    codes uint8 [cols, rows] and scales uint8 [cols, rows/32]."""
    v = np.asarray(v, dtype=np.float32).astype(np.float64)
    return mx_quantize_rows(v.T.copy().astype(np.float32))


def mx_dequantize_rows(codes, scales):
    """Inverse map of mx_quantize_rows (value = decode(code) * 2^(scale-127))."""
    rows, cols = codes.shape
    val = e4m3_decode(codes).reshape(rows, cols // 32, 32)
    return (val * np.exp2(scales.astype(np.float64) - 127.0)[..., None]).reshape(rows, cols)


def hadamard16():
    """Sylvester Hadamard matrix of order 16: H[i,j] = (-1)^popcount(i & j)."""
    i = np.arange(16)
    bits = np.bitwise_and(i[:, None], i[None, :])
    pop = np.array([[bin(int(b)).count("1") for b in row] for row in bits])
    return np.where(pop % 2 == 0, 1.0, -1.0)


def amax_plain(v, real_rows):
    """max |v| over the rows where real_rows is True (padding excluded)."""
    v = np.asarray(v, dtype=np.float64)
    if not np.any(real_rows):
        return 0.0
    return float(np.max(np.abs(v[real_rows])))


def amax_hadamard_t(v, padded_offsets, counts):
    """amax of the transposed, Hadamard-rotated tensor.

    The transpose v^T [cols, rows] is cut along rows (tokens) into 16-element
    segments inside each expert group (a group's tail segment is completed
    with zeros); each segment s becomes H16 s / 4 (orthonormal rotation).
    Returns the largest magnitude over all rotated segments.
    """
    v = np.asarray(v, dtype=np.float64)
    H = hadamard16() / 4.0
    best = 0.0
    for e in range(len(counts)):
        lo, m = int(padded_offsets[e]), int(counts[e])
        if m == 0:
            continue
        nseg = (m + 15) // 16
        blk = np.zeros((nseg * 16, v.shape[1]))
        blk[:m] = v[lo:lo + m]
        seg = blk.reshape(nseg, 16, v.shape[1])            # [seg, 16 tokens, col]
        rot = np.einsum("ij,sjc->sic", H, seg)
        best = max(best, float(np.max(np.abs(rot))))
    return best

