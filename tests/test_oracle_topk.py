"""Pins the oracle's top-k to a full stable sort (numpy), including ties and short rows."""
import numpy as np
import pytest

import oracle


def _ref(scores, kvlen, k):
    out = np.full((scores.shape[0], k), -1, np.int32)
    for t, n in enumerate(kvlen):
        s = scores[t, :n]
        order = np.lexsort((np.arange(n), -s))  # by -score, then index
        sel = np.sort(order[:min(k, n)])
        out[t, :len(sel)] = sel
    return out


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_matches_stable_sort(seed):
    rng = np.random.default_rng(seed)
    T, ld, k = 20, 700, 64
    scores = rng.standard_normal((T, ld))
    scores[::3] = np.round(scores[::3] * 4) / 4  # many exact ties
    kvlen = rng.integers(0, ld + 1, size=T).astype(np.int32)
    kvlen[:4] = [0, 1, k, k + 1]
    got = oracle.topk(scores, kvlen, k)
    assert np.array_equal(got, _ref(scores, kvlen, k))


def test_ties_take_lowest_index_and_signed_zero():
    scores = np.array([[0.0, -0.0, 1.0, 0.0, -0.0, 1.0]])
    got = oracle.topk(scores, np.array([6], np.int32), 3)
    assert got.tolist() == [[0, 2, 5]]


def test_nan_ranks_last():
    scores = np.array([[np.nan, -np.inf, 3.0, np.nan]])
    assert oracle.topk(scores, np.array([4], np.int32), 2).tolist() == [[1, 2]]
    assert oracle.topk(scores, np.array([4], np.int32), 3).tolist() == [[0, 1, 2]]
