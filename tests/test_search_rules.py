"""The pattern search's host-side choice rules (dynamic_sparse_attention_slash_gb300
/search.py) agree with the oracle's rules (MInference 1.0 overview, section 2.1)
on random FLOPs / recall tables, ties included."""
import numpy as np
import pytest

from oracle import msa_oracle as O
from dynamic_sparse_attention_slash_gb300 import search


@pytest.mark.parametrize("seed", range(50))
def test_rules_match_oracle(seed):
    rng = np.random.default_rng(seed)
    flops = [float(x) for x in rng.integers(1, 6, size=rng.integers(1, 7))]
    budget = float(rng.integers(0, 7))
    assert search.choose_setting(flops, budget) == O.choose_setting(flops, budget)
    rec = [float(x) for x in rng.integers(0, 4, size=rng.integers(1, 4)) / 3]
    assert search.choose_pattern(rec) == O.choose_pattern(rec)


def test_assignment_groups_one_call_per_pattern_setting():
    from dynamic_sparse_attention_slash_gb300.search import assignment_groups
    a = {(0, 0): ("vs", (64, 32)), (0, 1): ("bs", 4), (0, 2): ("vs", (64, 32)),
         (0, 3): ("st", (1, 4)), (1, 0): ("vs", [64, 32]), (1, 1): ("bs", 4),
         (1, 2): ("vs", (64, 32)), (1, 3): ("st", (1, 4))}
    g = sorted(assignment_groups(a, 4))
    assert g == [("bs", 4, [1]), ("st", (1, 4), [3]), ("vs", (64, 32), [0, 2])]


def test_assignment_groups_rejects_inconsistent_or_partial_maps():
    import pytest
    from dynamic_sparse_attention_slash_gb300.search import assignment_groups
    with pytest.raises(ValueError):  # head 0 differs between batch entries
        assignment_groups({(0, 0): ("bs", 4), (1, 0): ("bs", 8)}, 1)
    with pytest.raises(ValueError):  # head 1 unassigned
        assignment_groups({(0, 0): ("bs", 4)}, 2)
    with pytest.raises(ValueError):  # unknown pattern
        assignment_groups({(0, 0): ("xx", 4)}, 1)
