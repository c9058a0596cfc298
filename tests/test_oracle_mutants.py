"""Plants plausible mistakes in the oracle (on the CPU) and checks that the pins
catch each one: a pin suite that passes a broken oracle pins nothing."""
import numpy as np
import pytest

from oracle import msa_oracle as O
from tests import test_oracle_attend as TA
from tests import test_oracle_bs_st as TB
from tests import test_oracle_vs as TV


def _estimate_noncausal(q, k, last_q, scale):
    N = q.shape[0]
    L = min(last_q, N)
    z = (q[N - L:] @ k.T) * scale
    A = np.exp(z - z.max(1, keepdims=True))
    A /= A.sum(1, keepdims=True)
    s = np.zeros(N)
    for r, i in enumerate(range(N - L, N)):
        s[: i + 1] += A[r, i::-1]
    return A.sum(0), s, A


def _estimate_reversed_diagonal(q, k, last_q, scale):
    v, s, A = O.__dict__["_orig_estimate"](q, k, last_q, scale)
    return v, s[::-1].copy(), A


def _estimate_no_scale(q, k, last_q, scale):
    return O.__dict__["_orig_estimate"](q, k, last_q, 1.0)


def _estimate_shifted_window(q, k, last_q, scale):
    """Uses rows [N-L-1, N-1) instead of the last L rows."""
    N = q.shape[0]
    v, s, A = O.__dict__["_orig_estimate"](q[:N - 1], k[:N - 1], last_q, scale)
    return np.append(v, 0.0), np.append(s, 0.0), np.pad(A, ((0, 0), (0, 1)))


def _topk_ties_high(scores, k):
    scores = np.asarray(scores, dtype=np.float64)
    k = int(min(max(k, 0), scores.size))
    order = np.argsort(-scores[::-1], kind="stable")
    return np.sort(scores.size - 1 - order[:k])


def _tiles_no_carry(slash_idx, N):
    NB = N // 64
    act = np.zeros((NB, NB), dtype=bool)
    for o in slash_idx:
        for m in range(NB):
            n = m - o // 64
            if n >= 0:
                act[m, n] = True
    return act


def _blocks_no_diag(q, k, topk, scale=None):
    N, d = q.shape
    scale = O.default_scale(d) if scale is None else scale
    S = O.block_scores(q, k, scale)
    sel = [O.topk_indices(S[m, :m + 1], topk) for m in range(S.shape[0])]
    return sel, S


def _stream_window_off_by_one(m, init_num, local_window_num):
    sink = set(range(0, min(init_num, m + 1)))
    local = set(range(max(0, m - local_window_num), m + 1))
    return np.array(sorted(sink | local), dtype=np.int64)


def _attend_rows_no_causal(q, k, v, rows, allowed_keys, scale):
    rows = list(rows)
    out = np.zeros((len(rows), q.shape[1]))
    counts = np.zeros(len(rows), dtype=np.int64)
    for r, i in enumerate(rows):
        J = np.asarray(allowed_keys(i))
        if J.dtype == bool:
            J = np.nonzero(J)[0]
        counts[r] = J.size
        if J.size:
            z = (k[J] @ q[i]) * scale
            p = np.exp(z - z.max())
            out[r] = (p / p.sum()) @ v[J]
    return out, counts


def _run_all(tests):
    failures = 0
    for fn, args in tests:
        try:
            fn(*args)
        except (AssertionError, ValueError, TypeError, IndexError):
            failures += 1
    return failures


ESTIMATE_PINS = [(TV.test_estimate_zero_keys_closed_form, ()),
                 (TV.test_estimate_scale_closed_form, ()),
                 (TV.test_estimate_matches_torch_softmax_and_trace, ()),
                 (TV.test_estimate_invariants, (300, 64))]


@pytest.mark.parametrize("mutant", [_estimate_noncausal, _estimate_reversed_diagonal,
                                    _estimate_no_scale, _estimate_shifted_window])
def test_estimate_mutants_are_caught(monkeypatch, mutant):
    monkeypatch.setitem(O.__dict__, "_orig_estimate", O.estimate_vs)
    monkeypatch.setattr(O, "estimate_vs", mutant)
    assert _run_all(ESTIMATE_PINS) >= 1


def test_topk_mutant_is_caught(monkeypatch):
    monkeypatch.setattr(O, "topk_indices", _topk_ties_high)
    assert _run_all([(TV.test_topk_ties_prefer_lower_index, ()),
                     (TV.test_topk_brute_force, (0,))]) >= 1


def test_tile_mutant_is_caught(monkeypatch):
    monkeypatch.setattr(O, "vs_active_tiles", _tiles_no_carry)
    assert _run_all([(TV.test_tiles_three_derivations_agree, (256, 0)),
                     (TV.test_golden_tiny_vs_format, ())]) >= 1


def test_block_mutant_is_caught(monkeypatch):
    monkeypatch.setattr(O, "block_sparse_blocks", _blocks_no_diag)
    assert _run_all([(TB.test_block_selection_brute_force, (3,)),
                     (TB.test_diagonal_block_kept_even_when_it_scores_lowest, ())]) >= 1


def test_streaming_mutant_is_caught(monkeypatch):
    monkeypatch.setattr(O, "streaming_blocks", _stream_window_off_by_one)
    assert _run_all([(TB.test_streaming_blocks_closed_form, ()),
                     (TB.test_streaming_nnz_matches_mask_popcount, ())]) >= 1


def test_attend_mutant_is_caught(monkeypatch):
    monkeypatch.setattr(O, "attend_rows", _attend_rows_no_causal)
    assert _run_all([(TA.test_page_formula_with_large_c_matches_exclusion, ()),
                     (TA.test_single_key_rows_copy_the_value, ()),
                     (TA.test_attend_rows_and_blocks_agree, ())]) >= 1
