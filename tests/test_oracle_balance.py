"""Pins of the oracle's balanced partition (CPU only): its optimum against a
brute force over every assignment order, and closed forms."""
import itertools
import json
import os

import numpy as np
import pytest

from oracle import balance

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "pages_facts.json")


def _brute(counts, num_sets):
    """Every ordering of the experts, cut into consecutive sets."""
    E = len(counts)
    m = E // num_sets
    best = None
    for perm in itertools.permutations(range(E)):
        loads = [sum(counts[e] for e in perm[s * m:(s + 1) * m]) for s in range(num_sets)]
        best = max(loads) if best is None else min(best, max(loads))
    return best


@pytest.mark.parametrize("E,S", [(4, 2), (6, 2), (6, 3), (8, 2), (8, 4)])
def test_optimum_against_brute_force(E, S):
    rng = np.random.default_rng(E * 10 + S)
    for _ in range(3):
        counts = rng.integers(0, 50, size=E).tolist()
        assert balance.optimum_max_load(counts, S) == _brute(counts, S)


def test_closed_forms():
    assert balance.optimum_max_load([5] * 12, 4) == 15
    # one heavy expert: it shares its set with the lightest ones
    counts = [100, 1, 2, 3, 4, 5, 6, 7]
    assert balance.optimum_max_load(counts, 4) == 101
    assert balance.optimum_max_load(list(range(12)), 3) == 22   # sum 66 splits evenly


def test_loads_and_imbalance():
    counts = np.array([4, 0, 2, 2, 1, 3])
    l2p = np.array([5, 4, 3, 2, 1, 0])
    assert list(balance.set_loads(counts, l2p, 3)) == [4, 4, 4]
    assert balance.imbalance([4, 4, 4]) == 1.0
    assert list(balance.contiguous_loads(counts, 3)) == [4, 4, 4]
    assert balance.imbalance([6, 2]) == 1.5


def test_pages_set_structure():
    facts = json.load(open(GOLDEN))
    assert facts["balanced_sets"]["value"] * facts["balanced_set_size"]["value"] == \
        facts["routed_experts_per_block"]["value"]
    assert facts["experts_per_gpu"]["value"] * facts["ep_degree_per_node"]["value"] == \
        facts["routed_experts_per_block"]["value"]
