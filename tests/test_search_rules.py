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
