"""Pins of the oracle's argmax (the greedy-token step after the lm_head
matvec; "Gemma4 raw-Metal loop on A19", "The parked levers" table, argmax
row: first-max tie-break).  Checked against hand cases and numpy's argmax,
which also returns the first occurrence of the maximum."""
import numpy as np
import pytest

import oracle


@pytest.mark.parametrize("y,idx", [
    ([1.0], 0),
    ([-3.0, -1.0, -2.0], 1),
    ([2.0, 5.0, 5.0, 1.0], 1),                 # tie: the first one
    ([5.0, 2.0, 5.0], 0),
    ([-0.0, 0.0, -1.0], 0),                    # -0 equals +0: the first
    ([0.0, -0.0], 0),
    ([float("nan"), 1.0, float("nan"), 3.0], 3),
    ([float("-inf"), float("-inf")], 0),
    ([1.0, float("inf"), float("inf")], 1),
])
def test_argmax_hand_cases(y, idx):
    i, v = oracle.argmax(np.array(y, np.float32))
    assert i == idx
    assert v == np.float32(y[idx])


def test_argmax_none():
    assert oracle.argmax(np.array([], np.float32))[0] == -1
    assert oracle.argmax(np.array([float("nan")] * 3, np.float32))[0] == -1


def test_argmax_matches_numpy_first_occurrence():
    rng = np.random.default_rng(5)
    for n in (1, 2, 7, 1000, 100003):
        # few distinct values: many ties
        y = rng.integers(-5, 6, size=n).astype(np.float32) * np.float32(0.25)
        i, v = oracle.argmax(y)
        assert i == int(np.argmax(y)) and v == y.max()
