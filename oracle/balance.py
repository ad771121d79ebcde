"""Balanced partition of experts into equal-size sets, by exhaustive search.

Test infrastructure only (see oracle/__init__.py).

Source: Moreh report "21K output tokens/s DeepSeek inference on MI300X with
Expert Parallelism", section "Load balancing across GPUs": measure each
expert's activation frequency, group the 256 experts into 8 sets of 32 whose
total frequencies are as even as possible (a variant of balanced number
partitioning), and reorder the experts so each set is contiguous.  Splitting
into 8 contiguous chunks without balancing gave up to 2x imbalance; the
balanced grouping brought it within 5%.

Reading: the objective is the largest set total (minimised); the imbalance
figure is max set total / mean set total.  The exhaustive search below is
the definition of the optimum, usable for tiny expert counts only.
"""
from __future__ import annotations

import numpy as np


def set_loads(counts, log2phys, num_sets):
    """Total count per set when set s holds physical ids [s*m, (s+1)*m)."""
    counts = np.asarray(counts, dtype=np.int64)
    E = len(counts)
    m = E // num_sets
    loads = np.zeros(num_sets, dtype=np.int64)
    for e in range(E):
        loads[int(log2phys[e]) // m] += counts[e]
    return loads


def imbalance(loads) -> float:
    loads = np.asarray(loads, dtype=np.float64)
    mean = loads.mean()
    return float(loads.max() / mean) if mean > 0 else 1.0


def contiguous_loads(counts, num_sets):
    """Loads of the naive split: experts [s*m, (s+1)*m) on set s."""
    counts = np.asarray(counts, dtype=np.int64)
    return counts.reshape(num_sets, -1).sum(axis=1)


def optimum_max_load(counts, num_sets) -> int:
    """Smallest possible largest set total over all equal-size partitions.

    Enumerates every partition: the lowest unassigned expert opens a new set,
    which is filled with every combination of the remaining experts.
    """
    counts = [int(c) for c in counts]
    E = len(counts)
    assert E % num_sets == 0
    m = E // num_sets
    best = [None]

    def rec(remaining, cur_max):
        if best[0] is not None and cur_max >= best[0]:
            return
        if not remaining:
            best[0] = cur_max
            return
        first, rest = remaining[0], remaining[1:]
        for combo in _combinations(rest, m - 1):
            load = counts[first] + sum(counts[c] for c in combo)
            left = [r for r in rest if r not in combo]
            rec(left, max(cur_max, load))

    rec(list(range(E)), 0)
    return best[0]


def _combinations(items, r):
    if r == 0:
        yield ()
        return
    for i in range(len(items) - r + 1):
        for tail in _combinations(items[i + 1:], r - 1):
            yield (items[i],) + tail
