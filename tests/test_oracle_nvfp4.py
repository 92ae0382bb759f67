"""Pins of the NVFP4 oracle against things other than itself: brute-force
nearest-value search over the sixteen E2M1 codes, hand-derived tie cases,
lossless inputs on the NVFP4 grid, the invariants of the per-tensor encode
scale, the orthogonality of the 16-row Hadamard rotation, and closeness of
the NVFP4 grouped MLP to the (separately pinned) unquantized oracle."""
import numpy as np
import pytest

import oracle
from oracle.mx_oracle import e4m3_decode


def _brute_e2m1(y):
    """Nearest of all sixteen signed E2M1 values by exhaustive search; on a
    tie the candidate whose 3-bit magnitude code is even wins.  Values past
    6 in magnitude saturate."""
    mags = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    out = []
    for v in np.ravel(y):
        best = None
        for code in range(16):
            m = mags[code & 7]
            val = -m if code & 8 else m
            if (code & 8) and m == 0.0:
                continue
            d = abs(min(max(v, -6.0), 6.0) - val)
            key = (d, (code & 7) % 2)               # distance, then odd codes last
            if best is None or key < best[0]:
                best = (key, val)
        out.append(best[1])
    return np.array(out).reshape(np.shape(y))


def test_e2m1_round_brute_force():
    rng = np.random.default_rng(0)
    y = np.concatenate([rng.uniform(-8, 8, 4000),
                        np.arange(-7.0, 7.01, 0.25),          # every midpoint and grid point
                        [6.0, -6.0, 1e9, -1e9, 0.0]])
    got = oracle.e2m1_round(y)
    ref = _brute_e2m1(y)
    assert np.array_equal(np.abs(got), np.abs(ref))
    assert np.all((got == 0) | (np.sign(got) == np.sign(y)))


@pytest.mark.parametrize("y,want", [(0.25, 0.0), (0.75, 1.0), (1.25, 1.0), (1.75, 2.0),
                                    (2.5, 2.0), (3.5, 4.0), (5.0, 4.0), (7.0, 6.0),
                                    (-1.75, -2.0), (0.2499, 0.0), (0.2501, 0.5)])
def test_e2m1_ties_by_hand(y, want):
    """Midpoints between neighbouring grid values go to the even code:
    0|0.5 -> 0 (code 0), 0.5|1 -> 1 (code 2), 1|1.5 -> 1, 1.5|2 -> 2 (code 4),
    2|3 -> 2, 3|4 -> 4 (code 6), 4|6 -> 4; above 6 saturates."""
    assert float(oracle.e2m1_round(y)) == want


def test_e2m1_encode_codes():
    vals = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0, -0.5, -6.0])
    assert list(oracle.e2m1_encode(vals)) == [0, 1, 2, 3, 4, 5, 6, 7, 9, 15]


def test_lossless_grid_roundtrip():
    """A tensor whose amax is 2688 has encode scale 1; blocks whose largest
    magnitude is 6 * 2^e hold E2M1 values times 2^e exactly, so
    quantize-dequantize returns them unchanged and the block scales are 2^e."""
    rng = np.random.default_rng(1)
    rows, cols = 8, 64
    mags = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
    codes = mags[rng.integers(0, 8, (rows, cols))] * rng.choice([-1.0, 1.0], (rows, cols))
    codes.reshape(rows, -1, 16)[:, :, 0] = 6.0
    e = rng.integers(-4, 7, (rows, cols // 16))              # block scales 2^e <= 64
    v = (codes.reshape(rows, -1, 16) * np.exp2(e)[..., None]).reshape(rows, cols)
    v[0, :16] = codes[0, :16] * 448.0                         # amax 6 * 448 = 2688 -> g = 1
    g = oracle.nvfp4_global_scale(np.max(np.abs(v)))
    assert g == 1.0
    q, sc, s = oracle.nvfp4_quantize_rows(v.astype(np.float32), g)
    assert np.array_equal(oracle.nvfp4_dequantize_rows(q, s, g), v)
    assert s[0, 0] == 448.0
    assert np.array_equal(s.ravel()[1:], np.exp2(e).ravel()[1:])
    assert np.array_equal(e4m3_decode(sc), s)


def test_block_holding_the_tensor_amax():
    """The block that holds the tensor's largest magnitude gets the largest
    E4M3 scale (448) and that element the code +-6 (value amax exactly), for
    any amax; every dequantized value keeps its sign or becomes zero."""
    rng = np.random.default_rng(2)
    for amax in (1e-3, 0.37, 1.0, 913.5):
        v = rng.standard_normal((6, 48)).astype(np.float32)
        v *= np.float32(amax) / np.max(np.abs(v))
        i, j = np.unravel_index(np.argmax(np.abs(v)), v.shape)
        g = oracle.nvfp4_global_scale(np.max(np.abs(v)))
        q, sc, s = oracle.nvfp4_quantize_rows(v, g)
        assert s[i, j // 16] == 448.0
        assert abs(q[i, j]) == 6.0
        deq = oracle.nvfp4_dequantize_rows(q, s, g)
        assert abs(deq[i, j] - abs(v[i, j]) * np.sign(v[i, j])) <= 1e-6 * amax
        assert np.all((deq == 0) | (np.sign(deq) == np.sign(v)))


def test_quantization_error_bound():
    """Outside saturation each value lands on the E2M1 grid point nearest
    x*g/s, so its error is at most half the widest grid gap (1) times s/g;
    with s within 1/16 of amax_b * g / 6 this is below 0.18 amax_b."""
    rng = np.random.default_rng(3)
    v = (rng.standard_normal((64, 256)) * np.exp(rng.standard_normal((64, 1)))).astype(np.float32)
    deq = oracle.nvfp4_fake_rows(v)
    blk_amax = np.repeat(np.max(np.abs(v.reshape(64, 16, 16)), axis=-1), 16, axis=1)
    assert np.all(np.abs(deq - v) <= 0.18 * blk_amax + 1e-30)
    rel = np.linalg.norm(deq - v) / np.linalg.norm(v)
    assert 0.02 < rel < 0.15


def test_zero_tensor_and_zero_block():
    z = np.zeros((4, 32), np.float32)
    assert oracle.nvfp4_global_scale(0.0) == 1.0
    assert np.array_equal(oracle.nvfp4_fake_rows(z), z)
    v = np.ones((2, 32), np.float32)
    v[1, 16:] = 0.0
    q, sc, s = oracle.nvfp4_quantize_rows(v, oracle.nvfp4_global_scale(1.0))
    assert s[1, 1] == 0.0 and sc[1, 1] == 0 and np.all(q[1, 16:] == 0)


def test_fake_cols_is_rows_of_transpose():
    rng = np.random.default_rng(4)
    v = rng.standard_normal((32, 24))
    assert np.array_equal(oracle.nvfp4_fake_cols(v), oracle.nvfp4_fake_rows(v.T).T)


def test_rht16_orthonormal_and_product_invariant():
    rng = np.random.default_rng(5)
    a, b = rng.standard_normal((48, 7)), rng.standard_normal((48, 5))
    ra, rb = oracle.rht16_rows(a), oracle.rht16_rows(b)
    assert np.allclose(oracle.rht16_rows(ra), a, atol=1e-12)          # (H/4)^2 = I
    assert np.allclose(ra.T @ rb, a.T @ b, atol=1e-12)                # same rotation on both
    # a single 16-row segment: first output row is the segment mean times 4
    assert np.allclose(ra[0], a[:16].sum(axis=0) / 4.0)
    # segments do not mix
    a2 = a.copy()
    a2[16:] = 0
    assert np.array_equal(oracle.rht16_rows(a2)[16:], np.zeros((32, 7)))


def _grouped_case(seed=0, E=3, d=64, F=32, counts=(40, 0, 77), gated=True):
    rng = np.random.default_rng(seed)
    counts = np.array(counts)
    padded = np.concatenate([[0], np.cumsum((counts + 127) // 128 * 128)])
    R = int(padded[-1])
    x = np.zeros((R, d))
    dY = np.zeros((R, d))
    for e in range(E):
        lo, m = int(padded[e]), int(counts[e])
        x[lo:lo + m] = oracle.bf16_round(rng.standard_normal((m, d)))
        dY[lo:lo + m] = oracle.bf16_round(rng.standard_normal((m, d)))
    W1 = oracle.bf16_round(rng.standard_normal((E, (2 if gated else 1) * F, d)) / np.sqrt(d))
    W2 = oracle.bf16_round(rng.standard_normal((E, d, F)) / np.sqrt(F))
    b1 = oracle.bf16_round(rng.standard_normal((E, W1.shape[1])) * 0.1)
    b2 = oracle.bf16_round(rng.standard_normal((E, d)) * 0.1)
    p = oracle.GluParams() if gated else oracle.GluParams(act="srelu")
    return x, dY, padded, counts, W1, b1, W2, b2, p


@pytest.mark.parametrize("gated", [True, False])
def test_grouped_nv_close_to_unquantized(gated):
    """Every GEMM of the NVFP4 MLP sees operands within ~10% (rms) of the
    exact ones, so each output stays within 30% (Frobenius) of the
    unquantized grouped oracle and none is identical to it."""
    x, dY, padded, counts, W1, b1, W2, b2, p = _grouped_case(gated=gated)
    Hn, An, Yn = oracle.grouped_forward_nv(x, padded, counts, W1, b1, W2, b2, p)
    Hr, Ar, Yr = oracle.grouped_forward(x, padded, counts, W1, b1, W2, b2, p)
    gn = oracle.grouped_backward_nv(x, Hn, An, dY, padded, counts, W1, W2, p)
    gr = oracle.grouped_backward(x, Hr, Ar, dY, padded, counts, W1, W2, p)
    for name, a, b in [("H", Hn, Hr), ("A", An, Ar), ("Y", Yn, Yr), ("dX", gn[0], gr[0]),
                       ("dH", gn[1], gr[1]), ("dW1", gn[2], gr[2]), ("dW2", gn[4], gr[4])]:
        rel = np.linalg.norm(a - b) / np.linalg.norm(b)
        assert 0.0 < rel < 0.3, (name, rel)
    # the bias gradients are plain row sums of the (bf16) upstream gradients
    for e in range(len(counts)):
        lo, m = int(padded[e]), int(counts[e])
        assert np.allclose(gn[5][e], dY[lo:lo + m].sum(axis=0))
    # padding rows stay zero and an empty expert gets zero weight gradients
    assert np.all(Yn[40:128] == 0) and np.all(gn[2][1] == 0) and np.all(gn[4][1] == 0)


def test_grouped_nv_encode_scale_is_per_tensor():
    """Growing one expert's inputs raises X's tensor amax and so changes the
    other experts' quantized FC1 outputs; an expert's own rows alone do not
    decide its scale."""
    x, dY, padded, counts, W1, b1, W2, b2, p = _grouped_case(seed=6)
    H0 = oracle.grouped_forward_nv(x, padded, counts, W1, b1, W2, b2, p)[0]
    x2 = x.copy()
    lo = int(padded[2])
    x2[lo:lo + 77] *= 3.0
    H1 = oracle.grouped_forward_nv(x2, padded, counts, W1, b1, W2, b2, p)[0]
    assert not np.array_equal(H0[:40], H1[:40])


def test_wgrad_rotation_used():
    """The weight gradients of the NVFP4 oracle equal the products of the
    rotated-then-quantized operands (checked for one expert by brute force
    over explicit 16-row segments), not of the unrotated ones."""
    x, dY, padded, counts, W1, b1, W2, b2, p = _grouped_case(seed=7, counts=(48, 0, 0))
    Hn, An, Yn = oracle.grouped_forward_nv(x, padded, counts, W1, b1, W2, b2, p)
    dW2 = oracle.grouped_backward_nv(x, Hn, An, dY, padded, counts, W1, W2, p)[4][0]
    H16 = oracle.hadamard16() / 4.0
    m = 48
    dYr = np.concatenate([H16 @ dY[s:s + 16] for s in range(0, m, 16)])
    Ar = np.concatenate([H16 @ An[s:s + 16] for s in range(0, m, 16)])
    ref = oracle.nvfp4_fake_cols(dYr).T @ oracle.nvfp4_fake_cols(Ar)
    assert np.allclose(dW2, ref, rtol=1e-12, atol=1e-12)
    plain = oracle.nvfp4_fake_cols(dY[:m]).T @ oracle.nvfp4_fake_cols(An[:m])
    assert not np.allclose(dW2, plain, rtol=1e-3, atol=1e-6)
