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


@pytest.mark.parametrize("K,M", [(1, 4), (4, 1), (4, 16), (8, 32), (3, 7), (5, 2)])
@pytest.mark.parametrize("tf,tb", [(1, 2), (1, 1), (3, 5)])
def test_one_f_one_b_clock_closed_form(K, M, tf, tb):
    """With equal cells the interleaved order takes (M+K-1)(t_f+t_b), as GPipe
    does: the same bubble (K-1)/(M+K-1)."""
    sim = osch.simulate_1f1b(K, M, tf, tb)
    assert sim["makespan"] == (M + K - 1) * (tf + tb)
    assert sim["bubble"] == Fraction(K - 1, M + K - 1)


def test_one_f_one_b_clock_hand_worked():
    """K = 2, M = 3, t_f = (1, 2), t_b = (2, 3).  Cell 0: F0 F1 F2 B0 B1 B2,
    cell 1: F0 F1 B0 F2 B1 B2.  Cell 0 forwards in [0,1] [1,2] [2,3]; cell 1:
    F0 [1,3], F1 [3,5], B0 [5,8], F2 [8,10], B1 [10,13], B2 [13,16]; cell 0's
    backwards wait for cell 1's: B0 [8,10], B1 [13,15], B2 [16,18].  Makespan
    18, busy 3(1+2) + 3(2+3) = 24 of 2 x 18, bubble 1/3."""
    assert osch.one_f_one_b_sequence(2, 3, 0) == [("F", 0), ("F", 1), ("F", 2), ("B", 0), ("B", 1), ("B", 2)]
    assert osch.one_f_one_b_sequence(2, 3, 1) == [("F", 0), ("F", 1), ("B", 0), ("F", 2), ("B", 1), ("B", 2)]
    sim = osch.simulate_1f1b(2, 3, [1, 2], [2, 3])
    assert sim["makespan"] == 18 and sim["bubble"] == Fraction(1, 3)
