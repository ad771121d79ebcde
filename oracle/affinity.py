"""Expert co-activation and affinity-aware placement, by definition.

Test infrastructure only (see oracle/__init__.py).

Source: SGLang/H20 article "SGLang collaboration: best practices for deploying
DeepSeek-R1 on H20-96G", section "Expert Affinity EPLB": track which experts
are selected together in each token's top-k, build an expert affinity
matrix, and adjust the placement afterwards so that experts that are often
co-activated sit on the same node (a further ~5% over plain balancing).

Readings (the article gives no algorithm):
  * affinity A[a][b] = number of tokens whose top-k holds both a and b
    (a != b), over logical expert ids; symmetric, zero diagonal;
  * objective: the co-activation kept inside sets, sum over sets of
    A[a][b] for a < b in the same set, to be maximised;
  * constraint: every set total stays within a load bound, the larger of
    the balanced optimum and (1 + slack) x the mean set total;
  * quality figure: the mean number of distinct sets a token's experts
    span (the number of destinations its dispatch needs).
"""
from __future__ import annotations

import itertools

import numpy as np


def coactivation(logical_ids) -> np.ndarray:
    """A[a][b] for a token-by-k table of logical expert ids, by its definition."""
    ids = np.asarray(logical_ids, dtype=np.int64)
    E = int(ids.max()) + 1 if ids.size else 0
    return coactivation_n(ids, E)


def coactivation_n(logical_ids, num_experts: int) -> np.ndarray:
    ids = np.asarray(logical_ids, dtype=np.int64)
    A = np.zeros((num_experts, num_experts), dtype=np.int64)
    for row in ids:
        for a, b in itertools.combinations(row.tolist(), 2):
            if a != b:
                A[a, b] += 1
                A[b, a] += 1
    return A


def set_of_logical(log2phys, num_experts: int, num_sets: int) -> np.ndarray:
    m = num_experts // num_sets
    return np.asarray(log2phys, dtype=np.int64) // m


def intra_affinity(A, set_of) -> int:
    """Co-activation kept inside sets: sum of A[a][b], a < b, same set."""
    A = np.asarray(A)
    s = np.asarray(set_of)
    same = s[:, None] == s[None, :]
    return int(np.triu(A * same, k=1).sum())


def total_affinity(A) -> int:
    return int(np.triu(np.asarray(A), k=1).sum())


def mean_sets_per_token(logical_ids, set_of) -> float:
    ids = np.asarray(logical_ids, dtype=np.int64)
    s = np.asarray(set_of)[ids]
    return float(np.mean([len(set(r.tolist())) for r in s]))


def load_bound(counts, num_sets: int, balanced_max: int, slack: float) -> int:
    mean = float(np.sum(counts)) / num_sets
    return max(int(balanced_max), int(np.floor((1.0 + slack) * mean)))


def optimum_affinity(counts, A, num_sets: int, bound: int) -> int:
    """Largest intra-set affinity over all equal-size partitions whose set
    totals are all <= bound (exhaustive; tiny expert counts only)."""
    counts = [int(c) for c in counts]
    A = np.asarray(A)
    E = len(counts)
    m = E // num_sets
    best = [-1]

    def rec(remaining, acc):
        if not remaining:
            best[0] = max(best[0], acc)
            return
        first, rest = remaining[0], remaining[1:]
        for combo in itertools.combinations(rest, m - 1):
            members = (first,) + combo
            if sum(counts[e] for e in members) > bound:
                continue
            gain = sum(int(A[a, b]) for a, b in itertools.combinations(members, 2))
            left = [r for r in rest if r not in combo]
            rec(left, acc + gain)

    rec(list(range(E)), 0)
    return best[0]
