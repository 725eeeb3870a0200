"""Pins for the oracle's top-k selection (CPU only).

The C oracle (qsort with a comparator) is checked against routes written
independently here: Python's sorted() on explicit tuple keys, numpy's
lexsort, and properties any correct selection has.  Each test names the
mistake it is there to catch.
"""

import math

import numpy as np
import pytest

import oracle


def python_topk(row, n, k):
    """The definition written out: (NaN last, larger score first, smaller
    position first), the first min(k, n) positions, listed ascending."""
    def key(j):
        s = float(row[j])
        return (math.isnan(s), 0.0 if math.isnan(s) else -s, j)
    return sorted(sorted(range(n), key=key)[:min(k, n)])


def special_scores(rng, n):
    """Scores with many ties, zeros of both signs, infinities and NaNs."""
    s = rng.integers(-4, 5, n).astype(np.float32)
    s[rng.random(n) < 0.1] = -0.0
    s[rng.random(n) < 0.05] = np.inf
    s[rng.random(n) < 0.05] = -np.inf
    s[rng.random(n) < 0.05] = np.nan
    return s


@pytest.fixture(scope="module")
def lib():
    oracle.build()
    return oracle.load()


@pytest.mark.parametrize("seed", range(6))
def test_matches_python_sorted_with_ties_and_specials(lib, seed):
    # catches: a wrong tie direction, NaN ranked above -inf, -0 ranked below +0
    rng = np.random.default_rng(100 + seed)
    R, ld, k, k_max = 5, 90, 17, 20
    scores = np.stack([special_scores(rng, ld) for _ in range(R)])
    n_valid = np.array([90, 0, 1, 17, 40], np.int32)
    idx, n_sel, bad = oracle.topk(scores, n_valid, k, k_max)
    assert not bad.any()
    for r in range(R):
        want = python_topk(scores[r], n_valid[r], k)
        assert n_sel[r] == len(want)
        assert list(idx[r, :n_sel[r]]) == want
        assert (idx[r, n_sel[r]:] == -1).all()


def test_matches_numpy_lexsort_on_a_prefill_row_set(lib):
    # catches: reading past n_valid, a row stride mistake
    rng = np.random.default_rng(7)
    R, ld, k = 64, 4096, 640
    scores = rng.standard_normal((R, ld), dtype=np.float32)
    n_valid = rng.integers(1, ld + 1, R).astype(np.int32)
    scores[:, ::7] = np.float32(0.5)        # plenty of exact ties
    idx, n_sel, _ = oracle.topk(scores, n_valid, k)
    for r in range(R):
        n = n_valid[r]
        order = np.sort(np.lexsort((np.arange(n), -scores[r, :n]))[:min(k, n)])
        assert n_sel[r] == min(k, n)
        assert np.array_equal(idx[r, :n_sel[r]], order)


def test_selection_properties(lib):
    # catches: a duplicated or missing pick, picks not listed ascending, a
    # pick below a candidate left out
    rng = np.random.default_rng(8)
    ld, k = 2048, 300
    scores = rng.standard_normal((3, ld), dtype=np.float32)
    idx, n_sel, _ = oracle.topk(scores, np.full(3, ld, np.int32), k)
    for r in range(3):
        sel = idx[r, :k]
        assert len(set(sel.tolist())) == k and sel.min() >= 0 and sel.max() < ld
        assert (np.diff(sel) > 0).all()
        rest = np.setdiff1d(np.arange(ld), sel)
        assert scores[r, sel].min() >= scores[r, rest].max()


def test_all_equal_scores_pick_the_first_positions(lib):
    # catches: ties broken by anything but the position
    scores = np.full((2, 50), 3.0, np.float32)
    idx, n_sel, _ = oracle.topk(scores, np.array([50, 20], np.int32), 10, 12)
    assert list(idx[0]) == list(range(10)) + [-1, -1]
    assert list(idx[1]) == list(range(10)) + [-1, -1]


def test_fewer_candidates_than_k_take_all_in_order(lib):
    # catches: n_sel not clipped to n_valid
    scores = np.array([[0.5, -1.0, 2.0, np.nan, 2.0, 0.0]], np.float32)
    idx, n_sel, _ = oracle.topk(scores, np.array([6], np.int32), 10)
    assert n_sel[0] == 6
    assert list(idx[0, :6]) == [0, 1, 2, 3, 4, 5]
    assert (idx[0, 6:] == -1).all()


def test_nan_only_when_numbers_run_out(lib):
    # catches: NaN compared as a number
    scores = np.array([[np.nan, -np.inf, np.nan, -np.inf]], np.float32)
    idx, n_sel, _ = oracle.topk(scores, np.array([4], np.int32), 3)
    assert list(idx[0]) == [0, 1, 3]
    idx, n_sel, _ = oracle.topk(scores, np.array([4], np.int32), 2)
    assert list(idx[0]) == [1, 3]


def test_bad_n_valid_selects_nothing(lib):
    scores = np.zeros((3, 8), np.float32)
    idx, n_sel, bad = oracle.topk(scores, np.array([9, -1, 8], np.int32), 4)
    assert list(bad) == [1, 1, 0]
    assert list(n_sel) == [0, 0, 4]
    assert (idx[:2] == -1).all()
    assert list(idx[2]) == [0, 1, 2, 3]


def test_rejects_bad_arguments(lib):
    with pytest.raises(ValueError):
        oracle.topk(np.zeros((1, 4), np.float32), [4], 0)
    with pytest.raises(ValueError):
        oracle.topk(np.zeros((1, 4), np.float32), [4], 5, 4)
