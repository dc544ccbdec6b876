"""Pins for the oracle's top-k list builder (CPU only): closed forms (equal
scores, increasing scores, short candidate lists), agreement with a second
selection routine (heapq.nlargest over (score, -position)), the ordering
property of the chosen set, and the -0.0 / +0.0 tie."""
import heapq

import numpy as np
import pytest

from oracle import topk


def test_equal_scores_take_the_lowest_positions():
    s = np.full((2, 100), 0.5)
    out = topk.topk_select(s, 10)
    assert (out == np.arange(10)).all()


def test_increasing_scores_take_the_last_positions():
    s = np.arange(300, dtype=np.float64)[None, :]
    out = topk.topk_select(s, 16)
    assert out[0].tolist() == list(range(284, 300))


def test_short_lists_are_padded():
    s = np.random.default_rng(0).standard_normal((3, 50))
    out = topk.topk_select(s, 64, lengths=[50, 7, 0])
    assert out[0, :50].tolist() == list(range(50)) and (out[0, 50:] == -1).all()
    assert out[1, :7].tolist() == list(range(7)) and (out[1, 7:] == -1).all()
    assert (out[2] == -1).all()
    # lengths beyond the row are clamped
    assert (topk.topk_select(s, 64, lengths=[99, 99, 99])[:, :50] == np.arange(50)).all()


@pytest.mark.parametrize("seed", [1, 2, 3])
def test_agrees_with_heapq(seed):
    rng = np.random.default_rng(seed)
    s = np.round(rng.standard_normal((4, 3000)), 1)  # many ties
    out = topk.topk_select(s, 200)
    for t in range(4):
        want = sorted(p for _, p in heapq.nlargest(200, ((s[t, p], -p) for p in range(3000))))
        want = sorted(-q for q in want)
        assert out[t].tolist() == want


def test_chosen_scores_dominate_the_rest():
    rng = np.random.default_rng(9)
    s = rng.standard_normal((2, 5000))
    out = topk.topk_select(s, 128)
    for t in range(2):
        chosen = np.zeros(5000, dtype=bool)
        chosen[out[t]] = True
        assert s[t, chosen].min() > s[t, ~chosen].max()
        assert (np.diff(out[t]) > 0).all()


def test_negative_zero_ties_with_positive_zero():
    s = np.array([[-1.0, 0.0, -0.0, 0.0, -2.0]])
    assert topk.topk_select(s, 2)[0].tolist() == [1, 2]
    s = np.array([[-0.0, 0.0]])
    assert topk.topk_select(s, 1)[0].tolist() == [0]
