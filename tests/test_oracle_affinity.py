"""Pins of the oracle's co-activation matrix and affinity optimum (CPU only)."""
import itertools

import numpy as np

from oracle import affinity, balance


def test_coactivation_closed_forms():
    rng = np.random.default_rng(0)
    E, k, T = 12, 4, 200
    ids = np.array([rng.choice(E, k, replace=False) for _ in range(T)])
    A = affinity.coactivation_n(ids, E)
    assert np.array_equal(A, A.T) and np.all(np.diag(A) == 0)
    counts = np.bincount(ids.reshape(-1), minlength=E)
    # every selection of expert a pairs it with the other k-1 experts of its token
    assert np.array_equal(A.sum(axis=1), (k - 1) * counts)
    assert affinity.total_affinity(A) == T * k * (k - 1) // 2
    # one token: exactly its pairs
    one = affinity.coactivation_n(np.array([[3, 7, 1]]), 8)
    assert one[3, 7] == one[7, 1] == one[1, 3] == 1 and one.sum() == 6


def test_intra_affinity_and_sets_per_token():
    A = np.zeros((4, 4), np.int64)
    A[0, 1] = A[1, 0] = 5
    A[2, 3] = A[3, 2] = 2
    A[0, 2] = A[2, 0] = 1
    assert affinity.intra_affinity(A, [0, 0, 1, 1]) == 7
    assert affinity.intra_affinity(A, [0, 1, 0, 1]) == 1
    ids = np.array([[0, 1], [2, 3], [0, 2]])
    assert affinity.mean_sets_per_token(ids, [0, 0, 1, 1]) == (1 + 1 + 2) / 3


def _brute(counts, A, S, bound):
    E = len(counts)
    m = E // S
    best = -1
    for perm in itertools.permutations(range(E)):
        sets = [perm[s * m:(s + 1) * m] for s in range(S)]
        if any(sum(counts[e] for e in st) > bound for st in sets):
            continue
        best = max(best, sum(int(A[a, b]) for st in sets for a, b in itertools.combinations(st, 2)))
    return best


def test_optimum_against_brute_force():
    rng = np.random.default_rng(1)
    for E, S in [(6, 2), (6, 3), (8, 2), (8, 4)]:
        for _ in range(2):
            counts = rng.integers(1, 30, size=E)
            A = rng.integers(0, 9, size=(E, E))
            A = np.triu(A, 1)
            A = A + A.T
            bal = balance.optimum_max_load(counts.tolist(), S)
            bound = affinity.load_bound(counts, S, bal, 0.05)
            assert affinity.optimum_affinity(counts, A, S, bound) == _brute(counts.tolist(), A, S, bound)
