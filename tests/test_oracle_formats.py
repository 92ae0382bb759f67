"""Pins of the oracle's FC1 repack, MXFP8 quantizer and Hadamard amax.

* Repack: hand-worked layout for a small case and unpack(repack) = identity.
* E4M3: brute force over all 254 finite codes, hand-derived golden codes.
* E8M0 scales: hand-derived golden codes and the closed form for powers of 2.
* Hadamard: scipy's Sylvester construction, orthogonality, one-hot values.
"""
import os

import numpy as np
import pytest
import scipy.linalg

import oracle
from tests.conftest import read_golden


# ------------------------------------------------------------------ repack
def test_repack_layout_by_hand():
    # F=3, h=2: packed rows [g0 g1 l0 l1 | g2 0 l2 0]
    E, F, d = 1, 3, 2
    w1 = np.arange(E * 2 * F * d, dtype=np.float64).reshape(E, 2 * F, d) + 1
    w1p, b1p = oracle.repack_fc1(w1, np.arange(2 * F, dtype=np.float64)[None] + 1, h=2)
    g = w1[0, :F]
    l = w1[0, F:]
    want = np.stack([g[0], g[1], l[0], l[1], g[2], np.zeros(d), l[2], np.zeros(d)])
    assert np.array_equal(w1p[0], want)
    assert list(b1p[0]) == [1, 2, 4, 5, 3, 0, 6, 0]


@pytest.mark.parametrize("F,h", [(8, 4), (10, 4), (384, 128), (2880, 128)])
def test_unpack_repack_identity(F, h):
    rng = np.random.default_rng(F)
    w1 = rng.standard_normal((2, 2 * F, 3))
    w1p, _ = oracle.repack_fc1(w1, None, h=h)
    assert w1p.shape[1] % (2 * h) == 0
    assert np.array_equal(oracle.unpack_fc1(w1p, F, h=h), w1)
    src = oracle.fc1_packed_columns(F, h)
    assert np.all(w1p[:, src < 0, :] == 0)
    assert sorted(src[src >= 0].tolist()) == list(range(2 * F))


# ------------------------------------------------------------------ E4M3
def _all_finite_e4m3():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    vals = np.array([_decode_by_hand(int(c)) for c in codes])
    return codes, vals


def _decode_by_hand(c):
    s = -1.0 if c & 0x80 else 1.0
    ef, m = (c >> 3) & 0xF, c & 7
    if ef == 0:
        return s * m * 2.0 ** -9
    return s * (1 + m / 8) * 2.0 ** (ef - 7)


def _brute_round(y, codes, vals):
    """Nearest finite E4M3 value; ties to the even code; beyond 448 saturate."""
    if abs(y) >= 448.0:
        return float(np.copysign(448.0, y))
    dist = np.abs(vals - y)
    best = np.flatnonzero(dist == dist.min())
    if len(best) > 1:
        even = [b for b in best if (codes[b] & 1) == 0]
        best = even
    v = vals[best[0]]
    if v == 0.0:
        return float(np.copysign(0.0, y))
    return float(v)


def test_e4m3_decode_table_and_roundtrip():
    codes, vals = _all_finite_e4m3()
    np.testing.assert_array_equal(oracle.e4m3_decode(codes), vals)
    nz = vals != 0
    assert np.array_equal(oracle.e4m3_encode(vals[nz]), codes[nz])
    assert oracle.e4m3_encode(np.array([-0.0]))[0] == 0x80
    assert len(np.unique(vals)) == 253           # +0 and -0 compare equal
    assert vals.max() == 448.0


def test_e4m3_round_brute_force():
    codes, vals = _all_finite_e4m3()
    rng = np.random.default_rng(0)
    ys = np.concatenate([
        rng.standard_normal(20000) * 100,
        rng.uniform(-2.0 ** -5, 2.0 ** -5, 5000),
        np.exp2(rng.uniform(-12, 10, 5000)) * rng.choice([-1, 1], 5000),
        (vals[:, None] + np.array([[0.0]])).ravel(),
        ((vals[:-1] + vals[1:]) / 2),            # midpoints of neighbouring codes
        np.array([464.0, 480.0, 500.0, -464.0, 2.0 ** -10, 3 * 2.0 ** -10, 7.5 * 2.0 ** -9]),
    ])
    got = oracle.e4m3_round(ys)
    want = np.array([_brute_round(y, codes, vals) for y in ys])
    assert np.array_equal(got, want)
    assert np.array_equal(np.signbit(got), np.signbit(want))


def test_e4m3_golden(golden_dir):
    for v, code, _why in read_golden(os.path.join(golden_dir, "e4m3_codes.txt")):
        y = np.array([float(v)])
        assert oracle.e4m3_encode(oracle.e4m3_round(y))[0] == int(code, 16), v


def test_e8m0_golden_and_closed_form(golden_dir):
    for amax, code, _why in read_golden(os.path.join(golden_dir, "e8m0_scales.txt")):
        a = np.array([np.float32(float(amax))], dtype=np.float64)
        assert oracle.mx_scale_exponent(a)[0] + 127 == int(code), amax
    for j in range(-140, 136):
        for m in (1.0, 1.5, 1.999):
            want = min(max(j - 8, -127), 127)
            assert oracle.mx_scale_exponent(np.array([m * 2.0 ** j]))[0] == want


def test_mx_quantize_blocks_properties():
    rng = np.random.default_rng(4)
    v = (rng.standard_normal((64, 96)) * np.exp2(rng.integers(-20, 20, (64, 1)))).astype(np.float32)
    v[3, :32] = 0
    codes, scales = oracle.mx_quantize_rows(v)
    assert codes.shape == v.shape and scales.shape == (64, 3)
    assert scales[3, 0] == 0 and np.all(codes[3, :32] == 0)
    deq = oracle.mx_dequantize_rows(codes, scales)
    blk = np.abs(v.astype(np.float64)).reshape(64, 3, 32).max(-1)
    X = np.exp2(scales.astype(np.float64) - 127)
    # after scaling every |v|/X < 512, so the error is at most half an ulp of
    # the top binade (16) or saturation (|v|/X in [448, 512))
    err = np.abs(deq - v).reshape(64, 3, 32).max(-1)
    assert np.all(err <= 64 * X + 0)
    assert np.all(blk / X < 512) and np.all((blk / X >= 256) | (blk == 0))
    # columnwise = rowwise of the transpose
    c2, s2 = oracle.mx_quantize_cols(v[:, :32].T.copy())
    assert np.array_equal(c2, codes[:, :32]) and np.array_equal(s2[:, 0], scales[:, 0])


# ---------------------------------------------------------------- Hadamard
def test_hadamard_matrix():
    H = oracle.hadamard16()
    assert np.array_equal(H, scipy.linalg.hadamard(16).astype(np.float64))
    assert np.array_equal(H @ H.T, 16 * np.eye(16))


def test_hadamard_amax_cases():
    R, C = 64, 5
    padded = np.array([0, 32, 64])
    counts = np.array([20, 32])
    v = np.zeros((R, C))
    v[5, 2] = 3.0                              # one-hot segment -> amax 3/4
    assert oracle.amax_hadamard_t(v, padded, counts) == 0.75
    rng = np.random.default_rng(1)
    v = rng.standard_normal((R, C))
    v[20:32] = 1e6                             # padding rows must be ignored
    Hs = scipy.linalg.hadamard(16) / 4.0
    best = 0.0
    for e in range(2):
        rows = v[padded[e]:padded[e] + counts[e]]
        rows = np.concatenate([rows, np.zeros((-len(rows) % 16, C))])
        for s in range(0, len(rows), 16):
            seg = rows[s:s + 16]
            rot = Hs @ seg
            # rotation keeps each column's 2-norm
            np.testing.assert_allclose(np.linalg.norm(rot, axis=0), np.linalg.norm(seg, axis=0))
            best = max(best, np.abs(rot).max())
    assert oracle.amax_hadamard_t(v, padded, counts) == pytest.approx(best, rel=1e-15)
    real = np.zeros(R, bool); real[:20] = True; real[32:64] = True
    assert oracle.amax_plain(v, real) == np.abs(v[real]).max()
