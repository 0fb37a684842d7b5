"""Discrete-event simulation of the GPipe clock and its bubble fraction.

TEST INFRASTRUCTURE ONLY (see the package docstring).

GPipe technical review (zzz0906.github.io), "Pipeline flow" (the K = 4,
M = 8 walk-through of the paper's Figure 2c) and "Bubble overhead analysis":

  phase 1  micro-batch m enters cell 0; cell k forwards m once it has
           finished m-1 and cell k-1 has handed it m;
  phase 2  backward runs from the last cell to the first; every cell
           re-computes its forward before differentiating;
  phase 3  one update after all M micro-batches.

Reading taken: the figure's order, all forwards before any backward; cell k
starts backward of micro-batch m once it finished its forwards, its backward
of m-1 (micro-batches in ascending order) and cell k+1 handed it the
gradient of m.  (The review's prose says cell K-1 starts backward "after
micro-batch 1 has passed all cells", which would interleave forward and
backward on that cell; the figure and the bubble formula
(K-1)/(M+K-1) both describe the all-forward-then-all-backward order.)

simulate_1f1b takes the same rules for the one-forward-one-backward order
(the review's "Historical impact" section: PipeDream-2BW interleaves forward
and backward to lower the activation peak); its warm-up reading: cell k runs
min(M, K+1-k) forwards before its first backward.

The bubble fraction is the idle share of the K cells' time between the first
forward's start and the last backward's end.  Times are kept as exact
rationals.
"""
from __future__ import annotations

import sys
from fractions import Fraction


def simulate(K, M, t_f, t_b):
    """Simulate one GPipe step.

    t_f, t_b: per-cell forward/backward durations (sequences of length K, or
    scalars).  Returns dict(makespan, busy[K], bubble) with exact Fractions.
    """
    if K < 1 or M < 1:
        raise ValueError("need K >= 1 and M >= 1")
    tf = [Fraction(t_f)] * K if not hasattr(t_f, "__len__") else [Fraction(x) for x in t_f]
    tb = [Fraction(t_b)] * K if not hasattr(t_b, "__len__") else [Fraction(x) for x in t_b]
    f_end = [[Fraction(0)] * K for _ in range(M)]
    for m in range(M):
        for k in range(K):
            start = Fraction(0)
            if m > 0:
                start = max(start, f_end[m - 1][k])
            if k > 0:
                start = max(start, f_end[m][k - 1])
            f_end[m][k] = start + tf[k]
    b_end = [[Fraction(0)] * K for _ in range(M)]
    for m in range(M):
        for k in reversed(range(K)):
            start = f_end[M - 1][k]
            if m > 0:
                start = max(start, b_end[m - 1][k])
            if k < K - 1:
                start = max(start, b_end[m][k + 1])
            b_end[m][k] = start + tb[k]
    makespan = max(b_end[m][0] for m in range(M))
    busy = [M * (tf[k] + tb[k]) for k in range(K)]
    bubble = 1 - Fraction(sum(busy)) / (K * makespan)
    return dict(makespan=makespan, busy=busy, bubble=bubble)


def bubble_closed_form(K, M):
    """The review's bubble fraction (K-1)/(M+K-1) for equal cells."""
    return Fraction(K - 1, M + K - 1)


def one_f_one_b_sequence(K, M, k):
    """Cell k's operations in the one-forward-one-backward order, as
    ("F" | "B", m): min(M, K+1-k) forwards (the head counts as the stage after
    the last cell), then a backward and a forward in turn, backwards in
    ascending micro-batch order, then the remaining backwards."""
    warm = min(M, K + 1 - k)
    seq = [("F", m) for m in range(warm)]
    nxt = warm
    for m in range(M):
        seq.append(("B", m))
        if nxt < M:
            seq.append(("F", nxt))
            nxt += 1
    return seq


def simulate_1f1b(K, M, t_f, t_b):
    """Clock of the one-forward-one-backward order with the same rules as
    ``simulate``: a cell runs its operations in its order, each one as soon as
    the cell is free and its producer has finished (the forward of m on cell
    k-1; for a backward, the backward of m on cell k+1, or for the last cell
    the head, which takes no time and follows the last cell's forward).
    Finish times are computed by memoised recursion over each operation's two
    predecessors.  Returns dict(makespan, busy[K], bubble) as exact Fractions.
    """
    if K < 1 or M < 1:
        raise ValueError("need K >= 1 and M >= 1")
    tf = [Fraction(t_f)] * K if not hasattr(t_f, "__len__") else [Fraction(x) for x in t_f]
    tb = [Fraction(t_b)] * K if not hasattr(t_b, "__len__") else [Fraction(x) for x in t_b]
    seqs = [one_f_one_b_sequence(K, M, k) for k in range(K)]
    prev = {}
    for k, seq in enumerate(seqs):
        for i, op in enumerate(seq):
            prev[(k,) + op] = (k,) + seq[i - 1] if i else None
    memo = {}

    def finish(k, kind, m):
        key = (k, kind, m)
        if key in memo:
            return memo[key]
        start = Fraction(0)
        p = prev[key]
        if p is not None:
            start = max(start, finish(*p))
        if kind == "F":
            if k > 0:
                start = max(start, finish(k - 1, "F", m))
            end = start + tf[k]
        else:
            start = max(start, finish(K - 1, "F", m) if k == K - 1 else finish(k + 1, "B", m))
            end = start + tb[k]
        memo[key] = end
        return end

    sys.setrecursionlimit(max(sys.getrecursionlimit(), 20 * K * M + 1000))
    makespan = max(finish(k, "B", M - 1) for k in range(K))
    busy = [M * (tf[k] + tb[k]) for k in range(K)]
    bubble = 1 - Fraction(sum(busy)) / (K * makespan)
    return dict(makespan=makespan, busy=busy, bubble=bubble)
