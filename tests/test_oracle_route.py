"""Pins of the oracle's routing, offsets and permutation.

Routing: brute force over every k-subset of experts, hand-derived tie cases,
and scipy's softmax.  Offsets/permutation: invariants that any correct
stable counting sort satisfies, and permute followed by unpermute being the
identity."""
import itertools
import os

import numpy as np
import pytest
from scipy.special import softmax

import oracle
from tests.conftest import read_golden

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def brute_topk(score_row, k):
    """The unique k-subset S in which every member beats every non-member
    (larger score, or equal score and lower index), listed by that order."""
    E = len(score_row)

    def beats(i, j):
        return score_row[i] > score_row[j] or (score_row[i] == score_row[j] and i < j)

    winners = []
    for S in itertools.combinations(range(E), k):
        rest = [j for j in range(E) if j not in S]
        if all(beats(i, j) for i in S for j in rest):
            winners.append(S)
    assert len(winners) == 1
    S = list(winners[0])
    # order inside S by the same relation (selection sort)
    out = []
    while S:
        best = S[0]
        for i in S[1:]:
            if beats(i, best):
                best = i
        out.append(best)
        S.remove(best)
    return out


@pytest.mark.parametrize("seed", range(6))
def test_topk_matches_brute_force_with_ties(seed):
    rng = np.random.default_rng(seed)
    T, E, k = 40, 7, 3
    # values on a coarse grid so that exact ties are frequent
    logits = rng.integers(-3, 4, size=(T, E)).astype(np.float32) * np.float32(0.5)
    bias = (rng.integers(-2, 3, size=E).astype(np.float32) * np.float32(0.25)
            if seed % 2 else None)
    idx, w, counts = oracle.route(logits, bias, k)
    score = logits + (bias if bias is not None else np.float32(0))
    for t in range(T):
        assert list(idx[t]) == brute_topk(list(score[t]), k)


def test_golden_tie_cases(golden_dir):
    for row in read_golden(os.path.join(golden_dir, "route_ties.txt")):
        logits = np.array([[float(v) for v in row[0].split()]], dtype=np.float32)
        bias = None if row[1] == "-" else np.array([float(v) for v in row[1].split()], dtype=np.float32)
        want_idx = [int(v) for v in row[2].split()]
        want_w = [float(v) for v in row[3].split()]
        idx, w, _ = oracle.route(logits, bias, len(want_idx))
        assert list(idx[0]) == want_idx
        np.testing.assert_allclose(w[0], want_w, rtol=1e-14)


def test_weights_are_renormalised_full_softmax():
    rng = np.random.default_rng(1)
    T, E, k = 64, 16, 4
    logits = rng.standard_normal((T, E)).astype(np.float32)
    idx, w, _ = oracle.route(logits, None, k)
    full = softmax(logits.astype(np.float64), axis=1)
    sel = np.take_along_axis(full, idx, axis=1)
    np.testing.assert_allclose(w, sel / sel.sum(axis=1, keepdims=True), rtol=1e-13)
    np.testing.assert_allclose(w.sum(axis=1), 1.0, rtol=1e-14)
    # k == E: the weights are the plain softmax in score order
    idx2, w2, _ = oracle.route(logits, None, E)
    np.testing.assert_allclose(w2, np.take_along_axis(full, idx2, axis=1), rtol=1e-13)


def test_counts_offsets_and_permutation_invariants():
    rng = np.random.default_rng(2)
    T, E, k, align = 300, 9, 3, 32
    logits = rng.standard_normal((T, E)).astype(np.float32)
    bias = (rng.standard_normal(E) * 2).astype(np.float32)
    idx, w, counts = oracle.route(logits, bias, k)
    assert counts.sum() == T * k
    for t in range(T):
        assert len(set(idx[t])) == k                      # distinct experts
    offsets, padded, tiles = oracle.group_offsets(counts, align=align, tile_m=128)
    assert offsets[0] == 0 and offsets[E] == T * k
    assert np.all(np.diff(offsets) == counts)
    assert np.all(padded % align == 0)
    assert np.all(np.diff(padded) >= counts) and np.all(np.diff(padded) - counts < align)
    assert np.all(np.diff(tiles) == -(-counts // 128))
    row_src, row_of = oracle.permute_index(idx, E, padded)
    assert row_src.shape[0] == padded[E]
    for t in range(T):
        for s in range(k):
            j = row_of[t, s]
            assert row_src[j] == t
            e = idx[t, s]
            assert padded[e] <= j < padded[e] + counts[e]
    for e in range(E):
        grp = row_src[padded[e]:padded[e] + counts[e]]
        assert np.all(np.diff(grp) > 0)                    # ascending tokens
        assert np.all(row_src[padded[e] + counts[e]:padded[e + 1]] == -1)
    # every (token, slot) owns a distinct row
    assert len(set(row_of.reshape(-1).tolist())) == T * k


def test_permute_then_unpermute_is_identity():
    rng = np.random.default_rng(3)
    T, E, d = 50, 5, 12
    x = rng.standard_normal((T, d))
    logits = rng.standard_normal((T, E)).astype(np.float32)
    idx, w, counts = oracle.route(logits, None, 1)
    _, padded, _ = oracle.group_offsets(counts, align=8)
    row_src, row_of = oracle.permute_index(idx, E, padded)
    x_perm = oracle.gather_rows(x, row_src)
    assert np.all(x_perm[row_src < 0] == 0)
    back = oracle.combine(x_perm, row_of, np.ones((T, 1)))
    assert np.array_equal(back, x)                          # bitwise
    # k > 1 with the renormalised weights and identity experts
    idx, w, counts = oracle.route(logits, None, 3)
    _, padded, _ = oracle.group_offsets(counts, align=8)
    row_src, row_of = oracle.permute_index(idx, E, padded)
    back = oracle.combine(oracle.gather_rows(x, row_src), row_of, w)
    np.testing.assert_allclose(back, x, rtol=1e-14, atol=1e-15)
