"""Pins for the oracle's block-sparse head (MInference 1.0 overview, section
2.2, "Block-Sparse Head": mean-pool Q and K, block-level weights, top-k block
index) and streaming head (the page's kernel listing: streaming_forward with
init_num sink blocks and local_window_num local blocks).
"""
import math

import numpy as np
import pytest

from oracle import msa_oracle as O

D = 128


def test_pool_constant_and_ramp_closed_forms():
    N = 256
    a = np.random.default_rng(0).standard_normal(D)
    np.testing.assert_allclose(O.mean_pool(np.tile(a, (N, 1)), N), np.tile(a, (4, 1)), rtol=1e-14,
                               atol=1e-14)
    w = np.random.default_rng(1).standard_normal(D)
    ramp = np.arange(N)[:, None] * w[None, :]
    pooled = O.mean_pool(ramp, N)
    for m in range(4):
        np.testing.assert_allclose(pooled[m], (64 * m + 31.5) * w, rtol=1e-13, atol=1e-12)


def test_block_scores_closed_form():
    """Rows of block m of Q equal a_m, rows of block n of K equal b_n, so the
    pooled score is scale * a_m . b_n."""
    N = 192
    rng = np.random.default_rng(2)
    a = rng.standard_normal((3, D)); b = rng.standard_normal((3, D))
    q = np.repeat(a, 64, axis=0); k = np.repeat(b, 64, axis=0)
    S = O.block_scores(q, k, 0.5)
    for m in range(3):
        for n in range(3):
            assert abs(S[m, n] - 0.5 * sum(a[m, c] * b[n, c] for c in range(D))) < 1e-11


def brute_blocks(S, topk):
    sel = []
    for m in range(S.shape[0]):
        order = sorted(range(m), key=lambda n: (-S[m, n], n))[:max(topk - 1, 0)]
        sel.append(sorted(order + [m]))
    return sel


@pytest.mark.parametrize("topk", [1, 2, 3, 5, 8, 100])
def test_block_selection_brute_force(topk):
    N = 512
    rng = np.random.default_rng(3)
    q, k = rng.standard_normal((N, D)), rng.standard_normal((N, D))
    sel, S = O.block_sparse_blocks(q, k, topk)
    assert [s.tolist() for s in sel] == brute_blocks(S, topk)
    for m, s in enumerate(sel):
        assert len(s) == min(topk, m + 1) and m in s.tolist()


def test_row_restricted_selection_brute_force():
    """Selecting for a few row blocks scores exactly those rows: brute force on
    the pooled means, in the order the rows are given (ragged last block)."""
    N, topk = 700, 4
    rng = np.random.default_rng(6)
    q, k = rng.standard_normal((N, D)), rng.standard_normal((N, D))
    rows = [10, 0, 3, 7]
    sel, S = O.block_sparse_blocks(q, k, topk, row_blocks=rows)
    NB = (N + 63) // 64
    kp = np.stack([k[64 * n:min(N, 64 * n + 64)].mean(0) for n in range(NB)])
    for r, m in enumerate(rows):
        qm = q[64 * m:min(N, 64 * m + 64)].mean(0)
        want = (kp @ qm) / np.sqrt(D)
        np.testing.assert_allclose(S[r], want, rtol=1e-12, atol=1e-12)
        order = sorted(range(m), key=lambda n: (-want[n], n))[:topk - 1]
        assert sel[r].tolist() == sorted(order + [m])


def test_diagonal_block_kept_even_when_it_scores_lowest():
    N = 256
    rng = np.random.default_rng(4)
    base = rng.standard_normal(D)
    q = np.tile(base, (N, 1))
    k = np.tile(base, (N, 1))
    k[192:] = -base  # block 3 scores lowest for row block 3
    sel, S = O.block_sparse_blocks(q, k, 2)
    assert S[3, 3] < S[3, :3].min()
    assert sel[3].tolist() == [0, 3]  # tie among 0..2 -> lowest block


def test_softmax_ranking_gives_same_blocks():
    """The page ranks softmax-normalised block weights; softmax is monotone per
    row, so ranking raw pooled scores gives the same set."""
    N = 640
    rng = np.random.default_rng(5)
    q, k = rng.standard_normal((N, D)), rng.standard_normal((N, D))
    sel, S = O.block_sparse_blocks(q, k, 4)
    for m in range(1, S.shape[0]):
        row = S[m, :m + 1]
        p = np.exp(row - row.max()); p /= p.sum()
        earlier = O.topk_indices(p[:m], 3)
        assert sorted(earlier.tolist() + [m]) == sel[m].tolist()


def test_block_topk_covering_everything_is_dense():
    N = 320
    rng = np.random.default_rng(6)
    q, k, v = (rng.standard_normal((N, D)) for _ in range(3))
    out, rec = O.block_sparse_head(q, k, v, topk=5)
    np.testing.assert_allclose(out, O.dense_causal(q, k, v, 1 / math.sqrt(D)), rtol=1e-12,
                               atol=1e-13)
    assert rec["nnz"] == N * (N + 1) // 2


def test_streaming_blocks_closed_form():
    assert O.streaming_blocks(0, 1, 2).tolist() == [0]
    assert O.streaming_blocks(1, 1, 2).tolist() == [0, 1]
    assert O.streaming_blocks(5, 1, 2).tolist() == [0, 4, 5]
    assert O.streaming_blocks(5, 2, 3).tolist() == [0, 1, 3, 4, 5]
    assert O.streaming_blocks(3, 2, 3).tolist() == [0, 1, 2, 3]  # overlap, no repeats
    assert O.streaming_blocks(7, 0, 1).tolist() == [7]
    for m in range(10):  # init + local >= m + 1 covers every block
        assert O.streaming_blocks(m, 3, 8).tolist() == list(range(m + 1))


def test_streaming_wide_window_is_dense():
    N = 384
    rng = np.random.default_rng(7)
    q, k, v = (rng.standard_normal((N, D)) for _ in range(3))
    out, rec = O.streaming_head(q, k, v, init_num=0, local_window_num=6)
    np.testing.assert_allclose(out, O.dense_causal(q, k, v, 1 / math.sqrt(D)), rtol=1e-12,
                               atol=1e-13)


def test_streaming_nnz_matches_mask_popcount():
    N = 1024
    rng = np.random.default_rng(8)
    q, k, v = (rng.standard_normal((N, D)) for _ in range(3))
    out, rec = O.streaming_head(q, k, v, init_num=1, local_window_num=3)
    assert rec["nnz"] == O.nnz_from_blocks(rec["blocks"], N)
    # closed form: every row block has its diagonal tile (2080 pairs) plus a
    # full 4096-pair tile for each other block among {0} and {m-2, m-1}
    expect = 0
    for m in range(16):
        blocks = set([0]) | set(range(max(0, m - 2), m + 1))
        expect += 2080 + 4096 * (len(blocks) - 1)
    assert rec["nnz"] == expect


def test_golden_tiny_block_sparse_and_streaming():
    """Hand-worked cases (derivations in the fixture): block choice, admitted
    pairs and closed-form output rows of the block-sparse head; block lists and
    admitted pairs of the streaming head."""
    import json
    import os
    with open(os.path.join(os.path.dirname(__file__), "golden", "bs_st_tiny.json")) as f:
        g = json.load(f)
    bs = g["block_sparse"]
    N = bs["N"]
    q, k, v = np.zeros((N, D)), np.zeros((N, D)), np.zeros((N, D))
    for m in range(N // 64):
        q[64 * m:64 * (m + 1), :2] = bs["a"][m]
        k[64 * m:64 * (m + 1), :2] = bs["b"][m]
        v[64 * m:64 * (m + 1), :] = bs["c"][m]
    for case in bs["cases"]:
        out, info = O.block_sparse_head(q, k, v, case["topk"])
        assert [s.tolist() for s in info["blocks"]] == case["blocks"]
        assert info["nnz"] == case["nnz"]
        for row, val in case["rows"].items():
            np.testing.assert_allclose(out[int(row)], val, rtol=0, atol=2e-10)
    st = g["streaming"]
    N = st["N"]
    rng = np.random.default_rng(9)
    q, k, v = (rng.standard_normal((N, D)) for _ in range(3))
    for case in st["cases"]:
        _, info = O.streaming_head(q, k, v, case["init_num"], case["local_window_num"])
        assert [s.tolist() for s in info["blocks"]] == case["blocks"]
        assert info["nnz"] == case["nnz"]
