"""The periodic re-balancing policy on the CPU (no device counts needed):
when ExpertRebalancer.step re-balances."""
import pytest

import moe_expert_layer_07_gb300 as moe


def test_every_n_batches():
    due = [moe.rebalance_due(b, 4, None, 1, lambda: pytest.fail("not read")) for b in range(1, 9)]
    assert due == [False, False, False, True, True, True, True, True]


def test_imbalance_bound_read_only_on_check_batches():
    reads = []

    def imb():
        reads.append(1)
        return 1.3

    assert not moe.rebalance_due(1, None, 1.2, 2, imb) and not reads
    assert moe.rebalance_due(2, None, 1.2, 2, imb) and len(reads) == 1
    assert not moe.rebalance_due(2, None, 1.5, 2, imb)            # within the bound
    assert moe.rebalance_due(3, 3, 1.5, 2, imb)                    # the period wins


def test_neither_rule_never_fires():
    assert not any(moe.rebalance_due(b, None, None, 1, lambda: 9.0) for b in range(1, 50))
