"""Pins of the oracle's exact top-k: brute force with Python's sorted() on
small inputs full of ties, and the special cases the pages fix (every token
kept when at most 2048 are visible)."""
import numpy as np
import pytest

import oracle


def brute(scores, n, k):
    order = sorted(range(n), key=lambda s: (-scores[s], s))[:k]
    out = sorted(order) + [-1] * (k - min(k, n))
    return np.array(out, np.int32)


@pytest.mark.parametrize("n,k,levels", [(0, 5, 3), (1, 5, 3), (5, 5, 2), (100, 7, 4),
                                         (3000, 2048, 50), (5000, 2048, 5), (4097, 2048, 4096),
                                         (6000, 1, 10)])
def test_matches_brute_force(n, k, levels):
    rng = np.random.default_rng(n * 31 + k)
    scores = rng.integers(-levels, levels, size=max(n, 1)).astype(np.float64) / 4
    got = oracle.topk_row(scores, n, k)
    assert np.array_equal(got, brute(scores.tolist(), n, k))


def test_all_tokens_kept_when_at_most_k_visible():
    rng = np.random.default_rng(1)
    for n in [1, 63, 64, 65, 2047, 2048]:
        s = rng.standard_normal(n)
        got = oracle.topk_row(s, n, 2048)
        assert np.array_equal(got[:n], np.arange(n)) and (got[n:] == -1).all()


def test_all_equal_scores_pick_lowest_positions():
    s = np.full(10000, 3.25)
    got = oracle.topk_row(s, 10000, 2048)
    assert np.array_equal(got, np.arange(2048))


def test_signed_zeros_tie():
    s = np.array([-0.0, 0.0, -0.0, 1.0, -1.0])
    assert np.array_equal(oracle.topk_row(s, 5, 3), np.array([0, 1, 3]))


def test_ascending_unique_and_above_threshold():
    rng = np.random.default_rng(5)
    s = rng.standard_normal(50000)
    got = oracle.topk_row(s, 50000, 2048)
    assert (np.diff(got) > 0).all()
    tau = np.sort(s)[::-1][2047]
    assert (s[got] >= tau).all() and (s >= tau).sum() == 2048


def test_rows_use_their_own_visible_counts():
    rng = np.random.default_rng(8)
    S = rng.standard_normal((3, 3000))
    nv = np.array([3000, 2049, 10])
    got = oracle.topk(S, nv, 2048)
    for r in range(3):
        assert np.array_equal(got[r], oracle.topk_row(S[r], nv[r], 2048))


def test_nan_is_rejected():
    with pytest.raises(RuntimeError, match="NaN"):
        oracle.topk_row(np.array([1.0, np.nan]), 2, 1)
