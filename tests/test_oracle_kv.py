"""Pins for the oracle's KV selection ("How KV sparsity achieves 1.5x
acceleration for vLLM", Novita AI blog, section "2. Attention modification":
the attention pass exports each row's max and running sum; the score of key j
is the sum of its softmax probabilities over the rows of the instruction window
[n - alpha, n]; each head keeps the top-scoring keys).

Each test ties row_lse / kv_score to something other than their own formula:
the probability matrix that attend_blocks produces with identity values, the
vertical score of the estimate (an independent code path over the same
window), closed forms, and invariants.  The last test plants mistakes in the
oracle and checks that these pins catch every one.
"""
import math

import numpy as np
import pytest

from oracle import msa_oracle as O

D = 128


def rand_qk(N, seed, d=D):
    rng = np.random.default_rng(seed)
    return rng.standard_normal((N, d)), rng.standard_normal((N, d))


def random_block_mask(N, seed, density=0.4):
    """A mask per 64-row block that always admits the block's own keys."""
    rng = np.random.default_rng(seed)
    NB = N // O.BLOCK
    allow = rng.random((NB, N)) < density
    for m in range(NB):
        allow[m, m * O.BLOCK:(m + 1) * O.BLOCK] = True
    return lambda m: allow[m]


def test_score_is_column_sum_of_attention_probabilities():
    """N = d = 128 with v_j = e_j makes attend_blocks return the probability
    matrix P itself; the window score is the column sum of P over the window."""
    N, window = 128, 40
    q, k = rand_qk(N, 1)
    mask = random_block_mask(N, 2)
    P, _ = O.attend_blocks(q, k, np.eye(N), mask, O.default_scale(D))
    rec = O.kv_select_head(q, k, mask, window, 10)
    np.testing.assert_allclose(rec["score"], P[N - window:].sum(0), rtol=1e-12, atol=1e-15)
    # the exported normaliser reproduces every admitted probability
    z = q @ k.T * O.default_scale(D)
    for i in range(N):
        keys = np.nonzero(mask(i // O.BLOCK)[: i + 1])[0]
        np.testing.assert_allclose(np.exp(z[i, keys] - rec["lse"][i]), P[i, keys],
                                   rtol=1e-12, atol=1e-15)


def test_dense_window_score_equals_vertical_estimate():
    """With the all-ones mask and window = last_q the score is the estimate's
    vertical score: the column sum of the causal softmax of the last rows."""
    N = 320
    q, k = rand_qk(N, 3)
    v_score, _, _ = O.estimate_vs(q, k, 64, O.default_scale(D))
    rec = O.kv_select_head(q, k, lambda m: np.ones(N, dtype=bool), 64, 32)
    np.testing.assert_allclose(rec["score"], v_score, rtol=1e-11, atol=1e-14)


@pytest.mark.parametrize("window", [1, 64, 100, 256])
def test_scores_sum_to_the_window_rows(window):
    """Every non-empty window row's probabilities sum to 1."""
    N = 256
    q, k = rand_qk(N, 4)
    mask = random_block_mask(N, 5)
    rec = O.kv_select_head(q, k, mask, window, 8)
    assert abs(rec["score"].sum() - window) < 1e-10
    assert (rec["score"] >= 0).all()
    # no key after the last window row, no key outside every window row's set
    win = np.arange(N - window, N)
    reach = np.zeros(N, dtype=bool)
    for i in win:
        reach[: i + 1] |= mask(i // O.BLOCK)[: i + 1]
    assert (rec["score"][~reach] == 0).all()


def test_zero_keys_closed_form():
    """K = 0: every logit is 0, so lse_i = ln |J_i| and S_j = sum 1/|J_i|."""
    N, window = 192, 70
    q, _ = rand_qk(N, 6)
    k = np.zeros((N, D))
    mask = random_block_mask(N, 7, density=0.3)
    rec = O.kv_select_head(q, k, mask, window, 5)
    S = np.zeros(N)
    for i in range(N):
        keys = np.nonzero(mask(i // O.BLOCK)[: i + 1])[0]
        assert rec["lse"][i] == pytest.approx(math.log(keys.size), abs=1e-12)
        if i >= N - window:
            S[keys] += 1.0 / keys.size
    np.testing.assert_allclose(rec["score"], S, rtol=1e-12, atol=1e-15)


def test_empty_rows_have_minus_infinite_normaliser():
    N = 128
    q, k = rand_qk(N, 8)
    allow = np.zeros((2, N), dtype=bool)
    allow[1, 100:] = True          # rows 64..99 of block 1 see no key <= row
    rec = O.kv_select_head(q, k, lambda m: allow[m], 64, 4)
    assert np.isneginf(rec["lse"][:100]).all()
    assert np.isfinite(rec["lse"][100:]).all()
    assert abs(rec["score"].sum() - 28) < 1e-12   # rows 100..127 only


def test_keep_is_the_topk_of_the_score():
    N = 256
    q, k = rand_qk(N, 9)
    rec = O.kv_select_head(q, k, lambda m: np.ones(N, dtype=bool), 64, 20)
    order = sorted(range(N), key=lambda j: (-rec["score"][j], j))
    assert list(rec["keep"]) == sorted(order[:20])


def test_lse_matches_scalar_brute_force():
    N = 128
    q, k = rand_qk(N, 10)
    mask = random_block_mask(N, 11)
    scale = O.default_scale(D)
    rec = O.kv_select_head(q, k, mask, 16, 4)
    for i in (0, 1, 63, 64, 97, 127):
        keys = [j for j in range(i + 1) if mask(i // 64)[j]]
        zs = [scale * sum(q[i, c] * k[j, c] for c in range(D)) for j in keys]
        ref = math.log(sum(math.exp(z) for z in zs))
        assert rec["lse"][i] == pytest.approx(ref, rel=1e-12, abs=1e-12)


# ---------------------------------------------------------------- planted mistakes
def _score_window_off_by_one(q, k, window_lse, block_mask, window, scale):
    """Uses rows [N - window - 1, N - 1) with the normalisers of the true window."""
    N = q.shape[0]
    S = np.zeros(N)
    for r, i in enumerate(range(N - window - 1, N - 1)):
        if not np.isfinite(window_lse[r]):
            continue
        keys = np.nonzero(np.asarray(block_mask(i // 64))[: i + 1])[0]
        S[keys] += np.exp((k[keys] @ q[i]) * scale - window_lse[r])
    return S


def _score_no_causal(q, k, window_lse, block_mask, window, scale):
    N = q.shape[0]
    S = np.zeros(N)
    for r, i in enumerate(range(N - window, N)):
        if not np.isfinite(window_lse[r]):
            continue
        keys = np.nonzero(np.asarray(block_mask(i // 64)))[0]
        S[keys] += np.exp((k[keys] @ q[i]) * scale - window_lse[r])
    return S


def _lse_dense(q, k, rows, block_mask, scale):
    """Normaliser of dense causal attention whatever the mask."""
    out = np.empty(len(rows))
    for r, i in enumerate(rows):
        z = (k[: i + 1] @ q[i]) * scale
        out[r] = z.max() + np.log(np.exp(z - z.max()).sum())
    return out


PIN_TESTS = [
    test_score_is_column_sum_of_attention_probabilities,
    test_dense_window_score_equals_vertical_estimate,
    lambda: test_scores_sum_to_the_window_rows(100),
    test_zero_keys_closed_form,
    test_empty_rows_have_minus_infinite_normaliser,
]


@pytest.mark.parametrize("name,fn", [("kv_score", _score_window_off_by_one),
                                     ("kv_score", _score_no_causal),
                                     ("row_lse", _lse_dense)])
def test_planted_mistakes_are_caught(monkeypatch, name, fn):
    monkeypatch.setattr(O, name, fn)
    caught = 0
    for t in PIN_TESTS:
        try:
            t()
        except (AssertionError, ValueError, IndexError):
            caught += 1
    assert caught > 0, f"no pin catches the planted {fn.__name__}"
