"""Brute-force variance-minimising partition of L layers into K cells.

TEST INFRASTRUCTURE ONLY (see the package docstring).

GPipe technical review (zzz0906.github.io), "Algorithm: minimal interface":
GPipe cuts the sequence of L layers into K cells of consecutive layers and
balances them by minimising the variance of the cells' estimated costs, the
cost of a cell being the sum of its layers' cost estimates c_i.

Readings taken where the review is silent:
  * every cell holds at least one layer (so 1 <= K <= L);
  * "variance" is the population variance of the K cell sums; since the sum of
    all costs is fixed, minimising it is the same as minimising sum_k S_k^2,
    which is integer-exact;
  * among several optimal cuts the lexicographically smallest bounds vector
    (b_0 = 0 < b_1 < ... < b_K = L) is returned.

This is the definition written out: every one of the C(L-1, K-1) cut sets is
evaluated, in lexicographic order, with exact rational variance.
"""
from __future__ import annotations

from fractions import Fraction
from itertools import combinations


def cell_sums(costs, bounds):
    return [sum(costs[bounds[k]:bounds[k + 1]]) for k in range(len(bounds) - 1)]


def variance(sums):
    """Population variance of the cell sums, exact."""
    k = len(sums)
    mean = Fraction(sum(sums), k)
    return sum((Fraction(s) - mean) ** 2 for s in sums) / k


def partition(costs, K):
    """Bounds [0, b_1, ..., L] of the minimum-variance contiguous K-way cut."""
    L = len(costs)
    if not 1 <= K <= L:
        raise ValueError("need 1 <= K <= L")
    best, best_bounds = None, None
    for cuts in combinations(range(1, L), K - 1):
        bounds = [0, *cuts, L]
        v = variance(cell_sums(costs, bounds))
        if best is None or v < best:
            best, best_bounds = v, bounds
    return best_bounds, best
