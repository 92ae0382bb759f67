"""Pins of the MXFP8 expert-MLP oracle against things other than itself:
torch's bf16 conversion, lossless inputs on the MXFP8 grid, brute-force
block loops that quantize explicit 32-element vectors, and the (separately
pinned) unquantized oracle."""
import numpy as np
import pytest
import torch

import oracle
from oracle.mx_oracle import _quantize_blocks, e4m3_decode


def _params(**kw):
    return oracle.GluParams(**kw)


def test_bf16_round_matches_torch():
    rng = np.random.default_rng(0)
    v = (rng.standard_normal(20000) * np.exp2(rng.integers(-30, 30, 20000))).astype(np.float32)
    ref = torch.from_numpy(v).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(oracle.bf16_round(v.astype(np.float64)), ref)
    # ties go to the even significand
    assert oracle.bf16_round(1 + 2.0 ** -8) == 1.0
    assert oracle.bf16_round(1 + 3 * 2.0 ** -8) == 1 + 2.0 ** -6
    assert oracle.bf16_round(-(1 + 3 * 2.0 ** -8)) == -(1 + 2.0 ** -6)
    assert oracle.bf16_round(0.0) == 0.0


def _deq32(vec):
    """Quantize-dequantize one explicit 32-vector (the pinned block quantizer)."""
    codes, sc = _quantize_blocks(np.asarray(vec, np.float32).astype(np.float64)[None, :])
    return e4m3_decode(codes[0]) * 2.0 ** (int(sc[0]) - 127)


def _bf(v):
    return torch.from_numpy(np.asarray(v, np.float32)).to(torch.bfloat16).to(torch.float64).numpy()


def _tiny(seed=0, m=40, d=64, F=32):
    rng = np.random.default_rng(seed)
    X = _bf(rng.standard_normal((m, d)))
    W1 = _bf(rng.standard_normal((2 * F, d)) * 0.1)
    W2 = _bf(rng.standard_normal((d, F)) * 0.1)
    dY = _bf(rng.standard_normal((m, d)))
    return X, W1, W2, dY


def test_lossless_inputs_reduce_to_plain_fc1():
    """Blocks holding one +-16 and otherwise integers in [-15, 15] are exact
    in MXFP8 (scale 2^-4, payloads k*16), so the MXFP8 FC1 equals X W1^T."""
    rng = np.random.default_rng(3)

    def grid(shape):
        v = rng.integers(-15, 16, shape).astype(np.float64)
        v.reshape(-1, 32)[:, 0] = 16.0
        return v

    X, W1 = grid((16, 64)), grid((64, 64))
    assert np.array_equal(oracle.mx_fake_rows(X), X)
    p = _params()
    H, _, _ = oracle.expert_forward_mx(X, W1, None, np.zeros((64, 32)), None, p)
    assert np.array_equal(H, oracle.bf16_round(X @ W1.T))


def test_brute_force_blocks_forward_and_backward():
    X, W1, W2, dY = _tiny()
    m, d = X.shape
    F = W2.shape[1]
    p = _params()
    H16, A16, Y = oracle.expert_forward_mx(X, W1, None, W2, None, p)
    dX, dH16, dW1, db1, dW2, db2 = oracle.expert_backward_mx(X, H16, A16, dY, W1, W2, p)

    def dot_blocks(u_vecs, v_vecs):
        return sum(float(np.dot(_deq32(u), _deq32(v))) for u, v in zip(u_vecs, v_vecs))

    def row_blocks(M, i):                      # blocks along the row i of M
        return [M[i, 32 * j:32 * j + 32] for j in range(M.shape[1] // 32)]

    def col_blocks(M, c, rows=None):           # blocks down column c of M
        col = np.zeros(rows or M.shape[0])
        col[:M.shape[0]] = M[:, c]
        return [col[32 * j:32 * j + 32] for j in range(len(col) // 32)]

    rng = np.random.default_rng(1)
    for _ in range(12):
        r, f, c, g = rng.integers(m), rng.integers(F), rng.integers(d), rng.integers(2 * F)
        # FC1: K = d, X rows and W1 rows
        h = dot_blocks(row_blocks(X, r), row_blocks(W1, g))
        assert H16[r, g] == oracle.bf16_round(h)
        # FC2: K = F, A rows and W2 rows
        y = dot_blocks(row_blocks(A16, r), row_blocks(W2, c))
        assert abs(Y[r, c] - y) <= 1e-12 * max(1.0, abs(y))
        # FC1 dgrad: K = 2F, dH rows and W1 columns
        dx = dot_blocks(row_blocks(dH16, r), col_blocks(W1, c))
        assert abs(dX[r, c] - dx) <= 1e-12 * max(1.0, abs(dx))
        # FC2 wgrad: K = tokens, dY and A columns (group padded to 32 rows)
        mp = (m + 31) // 32 * 32
        w2 = dot_blocks(col_blocks(dY, c, mp), col_blocks(A16, f, mp))
        assert abs(dW2[c, f] - w2) <= 1e-12 * max(1.0, abs(w2))
        w1 = dot_blocks(col_blocks(dH16, g, mp), col_blocks(X, c, mp))
        assert abs(dW1[g, c] - w1) <= 1e-12 * max(1.0, abs(w1))
    # FC2 dgrad feeds the dGLU: K = d, dY rows and W2 columns
    dA = np.array([[dot_blocks(row_blocks(dY, r), col_blocks(W2, f)) for f in range(F)]
                   for r in range(m)])
    dG, dL = oracle.glu_backward(dA, H16[:, :F], H16[:, F:], p)
    assert np.allclose(dH16, oracle.bf16_round(np.concatenate([dG, dL], 1)), rtol=0, atol=1e-12)
    assert np.allclose(db2, dY.sum(0)) and np.allclose(db1, dH16.sum(0))


@pytest.mark.parametrize("act", ["swiglu", "geglu"])
def test_close_to_unquantized_oracle(act):
    """Quantization noise only: the MXFP8 results track the exact ones
    (relative Frobenius error of a few percent; a swapped or transposed
    operand would give an error of order one)."""
    X, W1, W2, dY = _tiny(seed=2, m=96, d=128, F=64)
    p = _params(act=act)
    Hm, Am, Ym = oracle.expert_forward_mx(X, W1, None, W2, None, p)
    H, A, Y = oracle.expert_forward(X, W1, None, W2, None, p)
    ref_b = oracle.expert_backward(X, H, A, dY, W1, W2, p)
    got_b = oracle.expert_backward_mx(X, Hm, Am, dY, W1, W2, p)
    for name, g, r in [("H", Hm, H), ("A", Am, A), ("Y", Ym, Y)] + list(
            zip(["dX", "dH", "dW1", "db1", "dW2", "db2"], got_b, ref_b)):
        err = np.linalg.norm(g - r) / np.linalg.norm(r)
        assert err < 0.1, (name, err)


def test_nongated_close_to_unquantized_oracle():
    """Non-gated squared ReLU (FC1 F wide): the same wiring check."""
    rng = np.random.default_rng(4)
    m, d, F = 96, 128, 64
    X = _bf(rng.standard_normal((m, d)))
    W1 = _bf(rng.standard_normal((F, d)) * 0.1)
    W2 = _bf(rng.standard_normal((d, F)) * 0.1)
    dY = _bf(rng.standard_normal((m, d)))
    p = _params(act="srelu")           # no clamp: its gradient jump is not noise
    Hm, Am, Ym = oracle.expert_forward_mx(X, W1, None, W2, None, p)
    H, A, Y = oracle.expert_forward(X, W1, None, W2, None, p)
    assert Hm.shape == (m, F) and Am.shape == (m, F)
    ref_b = oracle.expert_backward(X, H, A, dY, W1, W2, p)
    got_b = oracle.expert_backward_mx(X, Hm, Am, dY, W1, W2, p)
    for name, g, r in [("H", Hm, H), ("A", Am, A), ("Y", Ym, Y)] + list(
            zip(["dX", "dH", "dW1", "db1", "dW2", "db2"], got_b, ref_b)):
        err = np.linalg.norm(g - r) / np.linalg.norm(r)
        assert err < 0.1, (name, err)
