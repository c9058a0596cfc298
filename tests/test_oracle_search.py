"""Pins for the oracle's kernel-aware pattern search (MInference 1.0 overview,
section 2.1 "Kernel-Aware Optimal Sparse Pattern Search": candidates of each
pattern share a FLOPs target measured as the kernel computes it; one reference
example picks, per head, the pattern and setting with the best recall of the
attention output).

The recall (the dense attention mass a mask keeps) is tied to the row
normalisers of the KV-selection oracle by the identity
recall_i = exp(lse_M,i - lse_dense,i), to a closed form with zero keys, to
monotonicity under mask inclusion; the choice rules to brute-force enumeration.
The last test plants mistakes and checks the pins catch each one.
"""
import itertools

import numpy as np
import pytest

from oracle import msa_oracle as O

D = 128


def rand_qk(N, seed):
    rng = np.random.default_rng(seed)
    return rng.standard_normal((N, D)), rng.standard_normal((N, D))


def random_block_mask(N, seed, density=0.4):
    rng = np.random.default_rng(seed)
    allow = rng.random((N // 64, N)) < density
    for m in range(N // 64):
        allow[m, m * 64:(m + 1) * 64] = True
    return lambda m: allow[m]


def test_recall_equals_normaliser_ratio():
    N = 256
    q, k = rand_qk(N, 1)
    mask = random_block_mask(N, 2)
    scale = O.default_scale(D)
    rows = np.arange(N)
    dense = lambda m: np.ones(N, dtype=bool)
    got = O.mass_recall(q, k, rows, mask, scale)
    ref = np.exp(O.row_lse(q, k, rows, mask, scale) - O.row_lse(q, k, rows, dense, scale))
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(O.mass_recall(q, k, rows, dense, scale), 1.0, rtol=0, atol=1e-13)


def test_recall_zero_keys_closed_form():
    N = 192
    q, _ = rand_qk(N, 3)
    k = np.zeros((N, D))
    mask = random_block_mask(N, 4, density=0.3)
    got = O.mass_recall(q, k, np.arange(N), mask, O.default_scale(D))
    ref = [mask(i // 64)[: i + 1].sum() / (i + 1) for i in range(N)]
    np.testing.assert_allclose(got, ref, rtol=1e-13, atol=1e-15)


def test_recall_grows_with_the_mask():
    N = 256
    q, k = rand_qk(N, 5)
    small = random_block_mask(N, 6, density=0.2)
    extra = random_block_mask(N, 7, density=0.2)
    union = lambda m: small(m) | extra(m)
    rows = np.arange(N)
    a = O.mass_recall(q, k, rows, small, O.default_scale(D))
    b = O.mass_recall(q, k, rows, union, O.default_scale(D))
    assert (b >= a - 1e-15).all() and (b > a).any()


def test_mask_nnz_matches_enumeration():
    N = 192
    mask = random_block_mask(N, 8)
    ref = sum(int(mask(i // 64)[j]) for i in range(N) for j in range(i + 1))
    assert O.mask_nnz(mask, N) == ref
    assert O.mask_nnz(lambda m: np.ones(N, dtype=bool), N) == N * (N + 1) // 2


@pytest.mark.parametrize("seed", range(20))
def test_choice_rules_brute_force(seed):
    rng = np.random.default_rng(seed)
    flops = rng.integers(1, 9, size=rng.integers(1, 6)).astype(float)
    budget = float(rng.integers(0, 10))
    fit = [i for i, f in enumerate(flops) if f <= budget]
    if fit:
        ref = min(fit, key=lambda i: (-flops[i], i))
    else:
        ref = min(range(len(flops)), key=lambda i: (flops[i], i))
    assert O.choose_setting(flops, budget) == ref
    rec = rng.integers(0, 3, size=3) / 2
    assert O.choose_pattern(rec) == min(range(3), key=lambda i: (-rec[i], i))


def test_search_tie_goes_to_the_earlier_pattern():
    """Attention confined to each query's own 64-token block: block-sparse and
    streaming both keep all of it at the same cost (recall 1), and the tie
    goes to the earlier pattern in the order vertical-slash, block-sparse,
    streaming."""
    N = 512
    rng = np.random.default_rng(9)
    q = rng.standard_normal((N, D)) * 0.1
    k = rng.standard_normal((N, D)) * 0.1
    u = rng.standard_normal((N // 64 + 1, D))
    for m in range(N // 64):
        q[m * 64:(m + 1) * 64] += 2.0 * u[m]
        k[m * 64:(m + 1) * 64] += 2.0 * u[m]
    cands = {"bs": [2, 4], "st": [(0, 2), (0, 4)]}
    budget = 4 * D * O.mask_nnz(O.pattern_masks(q, k, "st", (0, 2), O.default_scale(D)), N)
    best, setting, recs = O.pattern_search_head(q, k, cands, budget)
    assert recs["bs"]["setting"] == 0 and recs["st"]["setting"] == 0
    assert recs["bs"]["recall"] == recs["st"]["recall"] > 1 - 1e-9
    assert (best, setting) == ("bs", 2)


def search_inputs():
    """Diffuse attention (block-local structure of norm 3 plus a shared sink
    direction on the first 8 keys) where the three patterns keep different
    dense mass at similar cost."""
    N = 512
    rng = np.random.default_rng(21)
    q = rng.standard_normal((N, D))
    k = rng.standard_normal((N, D))
    u = rng.standard_normal((N // 64, D))
    u = 3 * u / np.linalg.norm(u, axis=1, keepdims=True)
    for m in range(N // 64):
        q[m * 64:(m + 1) * 64] += u[m]
        k[m * 64:(m + 1) * 64] += u[m]
    s = rng.standard_normal(D)
    s = 4 * s / np.linalg.norm(s)
    q += s
    k[:8] += s
    return q, k


SEARCH_CANDS = {"vs": [(4, 8), (8, 16), (12, 20)], "bs": [1, 2, 3], "st": [(0, 1), (1, 1), (1, 2)]}
SEARCH_BUDGET = 36e6  # between the second and third settings' kernel FLOPs of every pattern


def test_search_head_against_pinned_parts():
    """pattern_search_head end to end against its pinned parts: each pattern's
    masks (pattern_masks), kernel FLOPs (4 d mask_nnz), the setting the budget
    admits (choose_setting), its recall (mass_recall over every row of that
    setting's own mask) and the winning pattern (choose_pattern).  The inputs
    make the budget pick a non-zero setting in every pattern and give the
    three patterns different recalls, so a search that scores the wrong mask or
    returns the wrong setting changes the result."""
    q, k = search_inputs()
    N = q.shape[0]
    scale = O.default_scale(D)
    best, setting, recs = O.pattern_search_head(q, k, SEARCH_CANDS, SEARCH_BUDGET)
    rows = np.arange(N)
    ref = {}
    for p in ("vs", "bs", "st"):
        masks = [O.pattern_masks(q, k, p, st, scale) for st in SEARCH_CANDS[p]]
        flops = [4 * D * O.mask_nnz(mk, N) for mk in masks]
        i = O.choose_setting(flops, SEARCH_BUDGET)
        ref[p] = (i, flops, float(O.mass_recall(q, k, rows, masks[i], scale).mean()))
        assert recs[p]["setting"] == i and recs[p]["flops"] == flops
        assert recs[p]["recall"] == ref[p][2]
    assert all(ref[p][0] == 2 for p in ref), "the budget must admit the third setting"
    recalls = [ref[p][2] for p in ("vs", "bs", "st")]
    assert len(set(recalls)) == 3, "the patterns' recalls must differ"
    want = ("vs", "bs", "st")[O.choose_pattern(recalls)]
    assert (best, setting) == (want, SEARCH_CANDS[want][ref[want][0]])
    assert (best, setting) == ("bs", 3)


# ---------------------------------------------------------------- planted mistakes
def _recall_sparse_softmax(q, k, rows, block_mask, scale):
    """Normalises over the masked keys (always 1): a plausible slip."""
    return np.ones(len(rows))


def _setting_cheapest_fit(flops, budget):
    flops = np.asarray(flops, float)
    fit = np.nonzero(flops <= budget)[0]
    return int(fit[np.argmin(flops[fit])]) if fit.size else int(np.argmin(flops))


def _search_recall_first_mask(q, k, candidates, budget_flops, rows=None, scale=None):
    """Scores every pattern's recall on its first candidate's mask instead of
    the chosen one: a plausible indexing slip."""
    N, d = q.shape
    scale = O.default_scale(d) if scale is None else scale
    rows = np.arange(N) if rows is None else np.asarray(rows)
    order = [p for p in ("vs", "bs", "st") if candidates.get(p)]
    recs = {}
    for p in order:
        masks = [O.pattern_masks(q, k, p, st, scale) for st in candidates[p]]
        flops = [4 * d * O.mask_nnz(mk, N) for mk in masks]
        i = O.choose_setting(flops, budget_flops)
        rec = float(O.mass_recall(q, k, rows, masks[0], scale).mean())
        recs[p] = {"setting": i, "flops": flops, "recall": rec}
    best = order[O.choose_pattern([recs[p]["recall"] for p in order])]
    return best, candidates[best][recs[best]["setting"]], recs


def _search_first_setting(q, k, candidates, budget_flops, rows=None, scale=None):
    """Returns the winning pattern's first setting instead of the chosen one."""
    best, _, recs = _ORIG_SEARCH(q, k, candidates, budget_flops, rows, scale)
    return best, candidates[best][0], recs


_ORIG_SEARCH = O.pattern_search_head

PINS = [test_recall_equals_normaliser_ratio, test_recall_zero_keys_closed_form,
        test_recall_grows_with_the_mask, test_search_head_against_pinned_parts] + [
            lambda s=s: test_choice_rules_brute_force(s) for s in range(20)]


@pytest.mark.parametrize("name,fn", [("mass_recall", _recall_sparse_softmax),
                                     ("choose_setting", _setting_cheapest_fit),
                                     ("pattern_search_head", _search_recall_first_mask),
                                     ("pattern_search_head", _search_first_setting)])
def test_planted_mistakes_are_caught(monkeypatch, name, fn):
    monkeypatch.setattr(O, name, fn)
    caught = 0
    for t in PINS:
        try:
            t()
        except AssertionError:
            caught += 1
    assert caught > 0, f"no pin catches {fn.__name__}"
