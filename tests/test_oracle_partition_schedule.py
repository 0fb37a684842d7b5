"""Pins of the oracle's partition and schedule model.

The partition is pinned to hand-worked cases (tests/golden) and to the
identical-layer property the review states (Transformer layers are identical,
so cells balance exactly); the schedule simulation is pinned to the review's
printed bubble values and its closed form.
"""
import json
import os
from fractions import Fraction

import numpy as np
import pytest

from oracle import partition as op
from oracle import schedule as osch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_partition_hand_worked_cases():
    cases = json.load(open(os.path.join(GOLDEN, "partition_examples.json")))["cases"]
    for c in cases:
        bounds, _ = op.partition(c["costs"], c["K"])
        assert bounds == c["bounds"], c


@pytest.mark.parametrize("L,K", [(8, 4), (24, 8), (12, 3), (12, 12), (9, 1)])
def test_partition_identical_layers_split_evenly(L, K):
    bounds, var = op.partition([7] * L, K)
    assert var == 0
    assert bounds == [i * (L // K) for i in range(K + 1)]


def test_variance_equals_sum_of_squares_ordering():
    """Minimising the variance orders cuts exactly as minimising sum S_k^2."""
    rng = np.random.default_rng(0)
    for _ in range(20):
        costs = [int(c) for c in rng.integers(1, 50, size=7)]
        K = int(rng.integers(1, 8))
        from itertools import combinations
        keys = []
        for cuts in combinations(range(1, 7), K - 1):
            b = [0, *cuts, 7]
            s = op.cell_sums(costs, b)
            keys.append((op.variance(s), sum(x * x for x in s), b))
        by_var = min(keys, key=lambda t: (t[0], t[2]))
        by_sq = min(keys, key=lambda t: (t[1], t[2]))
        assert by_var[2] == by_sq[2]


def test_bubble_printed_values():
    g = json.load(open(os.path.join(GOLDEN, "bubble_examples.json")))
    for e in g["exact"]:
        sim = osch.simulate(e["K"], e["M"], 1, 1)
        assert sim["bubble"] == Fraction(e["num"], e["den"])
    for e in g["printed_percent"]:
        sim = osch.simulate(e["K"], e["M"], 1, 2)
        assert round(float(sim["bubble"]) * 100, 1) == e["percent"]
    for a in g["approx"]:
        for K in a["K_values"]:
            M = K if a["rule"] == "M=K" else 4 * K
            assert abs(float(osch.simulate(K, M, 1, 1)["bubble"]) - a["value"]) <= a["abs_tol"]


@pytest.mark.parametrize("K", [1, 2, 3, 4, 8])
@pytest.mark.parametrize("M", [1, 2, 4, 7, 32])
def test_simulation_equals_closed_form(K, M):
    for tf, tb in [(1, 1), (1, 2), (Fraction(3, 7), Fraction(5, 3))]:
        sim = osch.simulate(K, M, tf, tb)
        assert sim["bubble"] == osch.bubble_closed_form(K, M)
        assert sim["makespan"] == (M + K - 1) * (Fraction(tf) + Fraction(tb))


def test_simulation_unequal_cells_hand_worked():
    # K=2, M=2, cell times f=(1,3), b=(1,3):
    # F00 0-1, F01 1-4, F10 1-2, F11 4-7; B01 7-10, B11 10-13; B00 10-11, B10 13-14
    sim = osch.simulate(2, 2, [1, 3], [1, 3])
    assert sim["makespan"] == 14
    assert sim["busy"] == [4, 12]
    assert sim["bubble"] == 1 - Fraction(16, 28)
