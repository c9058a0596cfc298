"""Pins for the oracle's vertical-slash head (MInference 1.0 overview,
section 2.2, "Vertical-Slash Head": estimate A-hat from the last queries,
choose vertical and slash lines, convert them to a sparse format, run
block-sparse attention over it).

Pins: closed forms for the estimate (zero keys, one-dimensional logits),
torch.softmax and numpy.trace as independent library routines, line-score
invariants, brute-force sorting for top-k, three derivations of the sparse
format (interval scan, enumeration of every (row, offset) pair, and the
tile-distance set), a hand-worked golden case, and reductions to dense
attention.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import msa_oracle as O

D = 128
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rand_qk(N, seed):
    rng = np.random.default_rng(seed)
    return rng.standard_normal((N, D)), rng.standard_normal((N, D))


# ----------------------------------------------------------------------------- estimate
def test_estimate_zero_keys_closed_form():
    """K = 0: A-hat[i, j] = 1/(i+1) over j <= i, so
    v[j] = sum_{i >= max(j, N-L)} 1/(i+1) and s[o] = sum_{i >= max(o, N-L)} 1/(i+1)."""
    N, L = 200, 64
    q, _ = rand_qk(N, 1)
    k = np.zeros((N, D))
    v, s, A = O.estimate_vs(q, k, L, 0.1)
    for j in range(N):
        expect = sum(1.0 / (i + 1) for i in range(max(j, N - L), N))
        assert abs(v[j] - expect) < 1e-12
        assert abs(s[j] - expect) < 1e-12  # same closed form with o in place of j


def test_estimate_scale_closed_form():
    """One query row whose logits are scale * a * j: A-hat is a geometric softmax."""
    N = 50
    a = 3.0
    q = np.zeros((N, D)); q[-1, 0] = a
    k = np.zeros((N, D)); k[:, 0] = np.arange(N) / 10.0
    scale = 1 / math.sqrt(D)
    v, s, _ = O.estimate_vs(q, k, 1, scale)
    w = [math.exp(scale * a * j / 10.0) for j in range(N)]
    tot = sum(w)
    for j in range(N):
        assert abs(v[j] - w[j] / tot) < 1e-13
        assert abs(s[N - 1 - j] - w[j] / tot) < 1e-13  # offset o = (N-1) - j


def test_estimate_matches_torch_softmax_and_trace():
    N, L = 192, 64
    q, k = rand_qk(N, 2)
    scale = 1 / math.sqrt(D)
    v, s, A = O.estimate_vs(q, k, L, scale)
    rows = torch.arange(N - L, N)
    z = torch.from_numpy(q[N - L:] @ k.T * scale)
    z = torch.where(torch.arange(N)[None, :] <= rows[:, None], z, torch.tensor(-math.inf, dtype=torch.float64))
    A_ref = torch.softmax(z, dim=-1).numpy()
    np.testing.assert_allclose(A, A_ref, rtol=1e-12, atol=1e-15)
    # diagonal o through the L x N window: column j = (N - L + r) - o, i.e. offset N-L-o
    for o in range(N):
        assert abs(s[o] - np.trace(A_ref, offset=N - L - o)) < 1e-12
    # column sums by scalar loops
    for j in [0, 1, 77, N - L - 1, N - L, N - 2, N - 1]:
        assert abs(v[j] - sum(A_ref[r, j] for r in range(L))) < 1e-12


@pytest.mark.parametrize("N,L", [(64, 64), (300, 64), (40, 64), (256, 16)])
def test_estimate_invariants(N, L):
    q, k = rand_qk(N, 3)
    v, s, A = O.estimate_vs(q, k, L, 1 / math.sqrt(D))
    Lc = min(L, N)
    assert A.shape == (Lc, N)
    assert abs(v.sum() - Lc) < 1e-10  # each estimate row sums to 1
    assert abs(s.sum() - Lc) < 1e-10
    assert abs(s[0] - sum(A[r, N - Lc + r] for r in range(Lc))) < 1e-12  # main diagonal
    assert (v >= 0).all() and (s >= 0).all()
    # keys / offsets no estimate row can reach score exactly 0
    assert (s[N:] == 0).all()


# ----------------------------------------------------------------------------- top-k
def brute_topk(scores, k):
    order = sorted(range(len(scores)), key=lambda j: (-scores[j], j))
    return sorted(order[:min(k, len(scores))])


@pytest.mark.parametrize("seed", range(5))
def test_topk_brute_force(seed):
    rng = np.random.default_rng(seed)
    n = int(rng.integers(1, 400))
    s = rng.random(n)
    s[rng.integers(0, n, n // 3)] = 0.5  # plant ties
    for k in [0, 1, 7, n // 2, n - 1, n, n + 5]:
        assert O.topk_indices(s, k).tolist() == brute_topk(s.tolist(), k)


def test_topk_ties_prefer_lower_index():
    s = np.array([1.0, 2.0, 2.0, 1.0, 2.0, 0.0])
    assert O.topk_indices(s, 2).tolist() == [1, 2]
    assert O.topk_indices(s, 4).tolist() == [0, 1, 2, 4]
    assert O.topk_indices(np.zeros(10), 3).tolist() == [0, 1, 2]


# ----------------------------------------------------------------------------- sparse format
def enumerate_tiles(S, N):
    """Every (row i, offset o) pair with i - o >= 0 marks key i - o; a tile is
    active iff it holds a marked key of one of its rows (rows of the sequence
    padded to a multiple of 64)."""
    NB = (N + 63) // 64
    act = np.zeros((NB, NB), dtype=bool)
    for o in S:
        for i in range(o, NB * 64):
            act[i // 64, (i - o) // 64] = True
    return act


def distance_set_tiles(S, N):
    """Tile distances t = m - n: {o // 64} and {o // 64 + 1 if o % 64 != 0}."""
    NB = (N + 63) // 64
    Dset = set()
    for o in S:
        Dset.add(o // 64)
        if o % 64:
            Dset.add(o // 64 + 1)
    act = np.zeros((NB, NB), dtype=bool)
    for m in range(NB):
        for n in range(m + 1):
            act[m, n] = (m - n) in Dset
    return act


@pytest.mark.parametrize("N,seed", [(256, 0), (256, 1), (192, 2), (320, 3), (128, 4),
                                    (200, 5), (77, 6), (130, 7), (1, 8), (63, 9)])
def test_tiles_three_derivations_agree(N, seed):
    rng = np.random.default_rng(seed)
    S = np.sort(rng.choice(N, size=min(N, int(rng.integers(1, 12))), replace=False))
    a = O.vs_active_tiles(S, N)
    np.testing.assert_array_equal(a, enumerate_tiles(S, N))
    np.testing.assert_array_equal(a, distance_set_tiles(S, N))
    assert not np.triu(a, 1).any()  # causal


def test_tiles_special_cases():
    N = 512
    only_diag = O.vs_active_tiles(np.array([0]), N)
    np.testing.assert_array_equal(only_diag, np.eye(8, dtype=bool))
    assert not O.vs_active_tiles(np.array([], dtype=np.int64), N).any()
    # offsets 64 and 128 hit exactly one tile diagonal each
    a = O.vs_active_tiles(np.array([64, 128]), N)
    np.testing.assert_array_equal(a, np.eye(8, k=-1, dtype=bool) | np.eye(8, k=-2, dtype=bool))


def test_columns_brute_force():
    N = 320
    rng = np.random.default_rng(5)
    S = np.array([0, 70, 200])
    V = np.sort(rng.choice(N, 40, replace=False))
    act = O.vs_active_tiles(S, N)
    cols = O.vs_columns(V, act, N)
    for m in range(5):
        expect = [j for j in V if j <= 64 * m + 63 and not act[m, j // 64]]
        assert cols[m].tolist() == expect


def test_golden_tiny_vs_format():
    """Hand-worked case (derivation in the fixture)."""
    with open(os.path.join(GOLDEN, "vs_format_tiny.json")) as f:
        g = json.load(f)
    N = g["N"]
    act = O.vs_active_tiles(np.array(g["slash"]), N)
    for m, tiles in enumerate(g["active_tiles"]):
        assert np.nonzero(act[m])[0].tolist() == tiles
    cols = O.vs_columns(np.array(g["vertical"]), act, N)
    assert [c.tolist() for c in cols] == g["columns"]
    rng = np.random.default_rng(0)
    q, k, v = (rng.standard_normal((N, D)) for _ in range(3))
    _, counts = O.attend_blocks(q, k, v, O.vs_block_mask(act, cols, N), 0.1)
    assert int(counts.sum()) == g["nnz"]


# ----------------------------------------------------------------------------- end to end
def test_vertical_topk_covering_all_keys_is_dense():
    N = 320
    rng = np.random.default_rng(6)
    q, k, v = (rng.standard_normal((N, D)) for _ in range(3))
    out, idx = O.vertical_slash_head(q, k, v, vertical_topk=N + 10, slash=3)
    np.testing.assert_allclose(out, O.dense_causal(q, k, v, 1 / math.sqrt(D)), rtol=1e-12,
                               atol=1e-13)
    assert idx["nnz"] == N * (N + 1) // 2


def test_slash_covering_all_offsets_is_dense():
    N = 256
    rng = np.random.default_rng(7)
    q, k, v = (rng.standard_normal((N, D)) for _ in range(3))
    out, idx = O.vertical_slash_head(q, k, v, vertical_topk=1, slash=N)
    assert idx["active"][np.tril_indices(4)].all()
    np.testing.assert_allclose(out, O.dense_causal(q, k, v, 1 / math.sqrt(D)), rtol=1e-12,
                               atol=1e-13)


def test_gqa_head_mapping():
    """Query head h reads KV head h // (Hq / Hkv)."""
    rng = np.random.default_rng(8)
    B, Hq, Hkv, N = 1, 4, 2, 128
    q = rng.standard_normal((B, Hq, N, D))
    k = rng.standard_normal((B, Hkv, N, D))
    v = rng.standard_normal((B, Hkv, N, D))
    out, _ = O.vertical_slash_sparse_attention(q, k, v, 16, 32, heads=[1, 2])
    for t, h in enumerate([1, 2]):
        ref, _ = O.vertical_slash_head(q[0, h], k[0, h // 2], v[0, h // 2], 16, 32)
        np.testing.assert_array_equal(out[0, t], ref)


def test_row_block_mask_agrees_with_full_format():
    N = 640
    rng = np.random.default_rng(9)
    S = np.sort(rng.choice(N, 7, replace=False))
    V = np.sort(rng.choice(N, 25, replace=False))
    act = O.vs_active_tiles(S, N)
    full = O.vs_block_mask(act, O.vs_columns(V, act, N), N)
    lazy = O.vs_row_block_mask(S, V, N)
    for m in range(N // 64):
        np.testing.assert_array_equal(full(m), lazy(m))
        np.testing.assert_array_equal(O.vs_active_tiles(S, N, [m])[0], act[m])
