"""Pins of the indexer top-k oracle against closed forms, a hand-derived rounding case and brute
force over all k-subsets."""

import itertools

import numpy as np
import pytest

import oracle


def test_integer_scores_equal_the_exact_dot_product():
    # small integers: every product and partial sum is exact in fp32, so the score is the exact
    # integer dot product (a dropped term, a wrong index or a transposed operand changes it)
    rng = np.random.default_rng(1)
    q = rng.integers(-8, 9, size=64)
    K = rng.integers(-8, 9, size=(200, 64))
    got = oracle.index_scores(q.astype(np.float64), K.astype(np.float64))
    want = K.astype(np.int64) @ q.astype(np.int64)
    assert got.dtype == np.float32
    assert np.array_equal(got.astype(np.int64), want)


def test_scores_round_in_index_order():
    # q = (1, 1, 1), k = (2^24, 1, -2^24): in index order 2^24 + 1 rounds (to even) to 2^24 and the
    # last term cancels it, so the fp32 score is 0 although the exact dot product is 1; summed in
    # the opposite order it would be 1.
    q = np.array([1.0, 1.0, 1.0])
    K = np.array([[2.0 ** 24, 1.0, -(2.0 ** 24)], [-(2.0 ** 24), 1.0, 2.0 ** 24]])
    got = oracle.index_scores(q, K)
    # second row: -2^24 + 1 = -(2^24 - 1) is exact in fp32, so that order keeps the 1
    assert got[0] == 0.0 and got[1] == 1.0
    K2 = np.array([[1.0, 2.0 ** 24, -(2.0 ** 24)]])
    assert oracle.index_scores(q, K2)[0] == 0.0          # (1 + 2^24) -> 2^24, then -> 0
    K3 = np.array([[2.0 ** 24, -(2.0 ** 24), 1.0]])
    assert oracle.index_scores(q, K3)[0] == 1.0          # cancellation first keeps the 1


def _brute_force_topk(scores, k):
    # among all k-subsets, the best one by its descending score profile, then by its ascending
    # index list (equal scores: lower indices preferred)
    best = None
    for sub in itertools.combinations(range(len(scores)), k):
        prof = tuple(sorted((-float(scores[j]) for j in sub)))
        key = (prof, sub)
        if best is None or key < best[0]:
            best = (key, sub)
    return np.array(best[1], dtype=np.int32)


@pytest.mark.parametrize("seed", range(12))
def test_topk_matches_brute_force_with_ties(seed):
    rng = np.random.default_rng(seed)
    n = int(rng.integers(1, 10))
    k = int(rng.integers(1, n + 1))
    scores = rng.integers(-3, 4, size=n).astype(np.float32)    # many ties
    got = oracle.topk_ascending(scores, k)
    assert np.array_equal(got, _brute_force_topk(scores, k))


def test_topk_special_cases():
    s = np.array([5.0, 1.0, 5.0, 3.0, 5.0], dtype=np.float32)
    assert oracle.topk_ascending(s, 5).tolist() == [0, 1, 2, 3, 4]      # k = n: everything
    assert oracle.topk_ascending(s, 2).tolist() == [0, 2]               # ties: lower indices
    assert oracle.topk_ascending(np.zeros(6, np.float32), 3).tolist() == [0, 1, 2]
    assert oracle.topk_ascending(np.array([-0.0, 0.0], np.float32), 1).tolist() == [0]
    with pytest.raises(ValueError):
        oracle.topk_ascending(s, 6)


def test_select_uses_only_the_complete_blocks():
    rng = np.random.default_rng(5)
    q = rng.integers(-4, 5, size=8).astype(np.float64)
    K = rng.integers(-4, 5, size=(30, 8)).astype(np.float64)
    K[25:] = 100.0                       # entries past L // 4 must never be chosen
    sel = oracle.indexer_select(q, K, L=4 * 25 + 3, k=5)
    assert sel.max() < 25
    want = oracle.topk_ascending((K[:25].astype(np.int64) @ q.astype(np.int64)).astype(np.float32), 5)
    assert np.array_equal(sel, want)
