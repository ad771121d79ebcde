"""Pins of the oracle's dispatch permutation (CPU only): the row of every slot
by its counting definition, round trips, offsets as a prefix sum."""
import numpy as np
import pytest

from oracle import permute


@pytest.mark.parametrize("T,k,E,S", [(1, 1, 1, 0), (5, 2, 4, 1), (37, 8, 32, 1), (64, 4, 16, 2)])
def test_permute_definition(T, k, E, S):
    rng = np.random.default_rng(T * k)
    ids = rng.integers(0, E, size=(T, k)).astype(np.int32)
    if T > 4:
        ids[: T // 2] = 0                     # one popular expert
        ids[:, 0] = np.minimum(ids[:, 0], E - 1)
    off, src, ros = permute.permute(ids, E, S)
    R = T * k
    assert off.shape == (E + S + 1,) and src.shape == (R + S * T,) and ros.shape == (T, k)
    counts = np.array([(ids == e).sum() for e in range(E)])
    assert off[0] == 0 and np.array_equal(np.diff(off)[:E], counts)
    assert np.all(np.diff(off)[E:] == T) and off[-1] == R + S * T
    # the row of slot i is its expert's first row plus the number of earlier
    # slots with the same expert (counting definition)
    flat = ids.reshape(-1)
    for i in range(R):
        e = flat[i]
        assert ros.reshape(-1)[i] == off[e] + np.count_nonzero(flat[:i] == e)
    # round trips
    assert np.array_equal(src[ros.reshape(-1)], np.arange(R))
    assert np.array_equal(np.sort(src[:R]), np.arange(R))
    for s in range(S):
        rows = off[E + s] + np.arange(T)
        assert np.array_equal(src[rows], R + s * T + np.arange(T))
        assert np.array_equal(permute.token_of_slot(src[rows], T, k), np.arange(T))
    assert np.array_equal(permute.token_of_slot(src[ros.reshape(-1)], T, k), np.repeat(np.arange(T), k))


def test_all_tokens_to_one_expert_and_empty_experts():
    T, k, E = 9, 1, 6
    ids = np.full((T, k), 4, np.int32)
    off, src, ros = permute.permute(ids, E, 1)
    assert list(off) == [0, 0, 0, 0, 0, 9, 9, 18]
    assert np.array_equal(ros[:, 0], np.arange(T))
