"""Pins for the oracle's hierarchical pruning head (InfiniteHiP summary page,
section "modular hierarchical token pruning algorithm": chunks of the key
sequence are represented by their highest-scoring token, only the best chunks
go on to the next stage, and stacked stages refine the block-sparse mask for
the current query block).

Each pin ties the oracle to something other than itself: keep-all stages give
dense causal attention (torch SDPA); one stage of single blocks equals a
brute-force scalar-loop ranking of block maxima; with keep counts that cover
the final one, stacking stages cannot change the result (a theorem, proved in
the docstring below); zero keys tie every score and give a closed-form set;
hand-built cases fix the representative (the maximum token, not the mean),
the forced own chunk and the narrowing of candidates between stages.  The
last test plants mistakes and checks the pins catch each.
"""

import numpy as np
import pytest
import torch

from oracle import msa_oracle as O

D = 128
SCALE = O.default_scale(D)

def rand_qk(N, seed, block=0.0):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((N, D))
    k = rng.standard_normal((N, D))
    if block:
        nb = (N + 63) // 64
        u = rng.standard_normal((nb, D))
        u = block * u / np.linalg.norm(u, axis=1, keepdims=True)
        rows = np.repeat(u, 64, axis=0)[:N]
        q += rows
        k += rows
    return q, k

@pytest.mark.parametrize("N", [640, 700])
def test_keep_all_is_dense_causal(N):
    q, k = rand_qk(N, 1)
    v = np.random.default_rng(2).standard_normal((N, D))
    NB = (N + 63) // 64
    stages = [(4, NB), (2, NB), (1, NB)]
    sel, _ = O.hierarchical_blocks(q, k, stages)
    for m in range(NB):
        np.testing.assert_array_equal(sel[m], np.arange(m + 1))
    out, _ = O.hierarchical_head(q, k, v, stages)
    ref = torch.nn.functional.scaled_dot_product_attention(
        *(torch.from_numpy(x)[None, None] for x in (q, k, v)), is_causal=True)[0, 0].numpy()
    np.testing.assert_allclose(out, ref, rtol=1e-10, atol=1e-12)

def brute_block_max(q, k, m, n):
    """max over the keys j of block n (j <= 64m + 63, j < N) of scale * Qhat_m . k_j,
    with the pooled query and every dot product written out as scalar loops."""
    N = q.shape[0]
    rows = range(m * 64, min(N, m * 64 + 64))
    qhat = [sum(q[i, c] for i in rows) / len(rows) for c in range(D)]
    best = -np.inf
    for j in range(n * 64, min(N, n * 64 + 64, m * 64 + 64)):
        best = max(best, SCALE * sum(qhat[c] * k[j, c] for c in range(D)))
    return best

@pytest.mark.parametrize("keep", [1, 3, 5])
def test_single_stage_is_brute_force_block_max_ranking(keep):
    N = 576
    q, k = rand_qk(N, 3, block=2.0)
    sel, _ = O.hierarchical_blocks(q, k, [(1, keep)])
    for m in (0, 1, 4, 8):
        r = [brute_block_max(q, k, m, n) for n in range(m)]
        others = sorted(range(m), key=lambda n: (-r[n], n))[:keep - 1]
        np.testing.assert_array_equal(sel[m], sorted(others + [m]), err_msg=f"m{m}")

@pytest.mark.parametrize("seed", range(4))
def test_covering_stages_equal_one_stage(seed):
    """Theorem: if every stage keeps at least as many chunks as the last stage
    keeps blocks (keep_s >= keep_S), and scores have no ties, multi-stage
    pruning keeps exactly the blocks one stage of single blocks keeps.  Proof:
    let b != m be among the keep_S - 1 best other blocks by block maximum.  If
    some stage dropped b's chunk X, then keep_s - 1 >= keep_S - 1 other chunks
    beat X's maximum, each through a block (not m's chunk, so not m) whose
    maximum beats b's: b would not be among the keep_S - 1 best.  So every
    such b survives to the last stage, where it is again among the best."""
    N = 1280
    q, k = rand_qk(N, 10 + seed, block=1.5)
    one, _ = O.hierarchical_blocks(q, k, [(1, 6)])
    for stages in ([(4, 6), (1, 6)], [(8, 7), (2, 6), (1, 6)], [(2, 9), (1, 6)]):
        multi, _ = O.hierarchical_blocks(q, k, stages)
        for m in range(len(one)):
            np.testing.assert_array_equal(multi[m], one[m], err_msg=f"{stages} m{m}")

def test_stages_narrow_the_candidates():
    """Query block 7 with stages [(4, 1), (1, 2)]: the first stage keeps only
    the chunk of blocks 4..7, so the final pair is block 7 and the best of
    blocks 4..6, although block 0 holds the best token of all."""
    N = 512
    q = np.zeros((N, D))
    k = np.zeros((N, D))
    q[:, 0] = 1.0
    k[10, 0] = 9.0        # block 0: the best token
    k[64 * 5 + 3, 0] = 4.0  # block 5: the best token of chunk 1 besides block 7's
    k[64 * 6 + 1, 0] = 2.0
    sel, kept = O.hierarchical_blocks(q, k, [(4, 1), (1, 2)])
    np.testing.assert_array_equal(kept[7][0], [1])
    np.testing.assert_array_equal(sel[7], [5, 7])
    # one stage of single blocks would take block 0
    one, _ = O.hierarchical_blocks(q, k, [(1, 2)])
    np.testing.assert_array_equal(one[7], [0, 7])

def test_representative_is_the_best_token_not_the_mean():
    """Chunk 0 (blocks 0-1) holds one strong token among very weak ones; chunk
    1 (blocks 2-3) holds uniformly good tokens with a higher mean.  Query block
    5 (own chunk 2) keeps one other chunk: chunk 0, by its best token."""
    N = 384
    q = np.zeros((N, D))
    k = np.zeros((N, D))
    q[:, 0] = 1.0
    k[:128, 0] = -5.0
    k[77, 0] = 10.0
    k[128:256, 0] = 6.0
    sel, kept = O.hierarchical_blocks(q, k, [(2, 2), (1, 6)])
    np.testing.assert_array_equal(kept[5][0], [0, 2])
    np.testing.assert_array_equal(sel[5], [0, 1, 4, 5])

def zero_key_sets(NB, stages):
    """Closed form with every score equal: each stage keeps the own chunk and
    the lowest-numbered other chunks that still hold candidates."""
    out = []
    for m in range(NB):
        cand = set(range(m + 1))
        for c, keep in stages:
            chunks = sorted({n // c for n in cand})
            kept = {m // c} | set([x for x in chunks if x != m // c][:keep - 1])
            cand = {n for n in cand if n // c in kept}
        out.append(sorted(cand))
    return out

def test_zero_keys_closed_form():
    N = 1024
    q = np.random.default_rng(4).standard_normal((N, D))
    k = np.zeros((N, D))
    stages = [(4, 2), (1, 3)]
    sel, _ = O.hierarchical_blocks(q, k, stages)
    want = zero_key_sets(N // 64, stages)
    for m in range(N // 64):
        np.testing.assert_array_equal(sel[m], want[m])
    # written out for three blocks: chunk 0 is the lowest other chunk
    assert want[10] == [0, 1, 10] and want[2] == [0, 1, 2] and want[5] == [0, 1, 5]

def test_planted_token_is_kept_by_every_later_block():
    N = 1024
    q, k = rand_qk(N, 5)
    u = q.mean(0)
    k[300] += 40 * u / np.linalg.norm(u)  # block 4
    sel, _ = O.hierarchical_blocks(q, k, [(4, 2), (2, 2), (1, 2)])
    for m in range(4, N // 64):
        assert 4 in sel[m], m

def test_kept_counts():
    N = 2048
    q, k = rand_qk(N, 6, block=2.0)
    stages = [(8, 3), (2, 4), (1, 5)]
    sel, kept = O.hierarchical_blocks(q, k, stages)
    for m, blocks in enumerate(sel):
        assert blocks[-1] == m and np.all(np.diff(blocks) > 0)
        for s, (c, keep) in enumerate(stages):
            assert m // c in kept[m][s] and len(kept[m][s]) <= keep
        # the last stage keeps min(5, candidates left by the first two stages)
        left = [n for n in range(m + 1) if n // 8 in kept[m][0] and n // 2 in kept[m][1]]
        assert blocks.size == min(5, len(left)) and set(blocks) <= set(left)
        np.testing.assert_array_equal(kept[m][2], blocks)

# ---------------------------------------------------------------- planted mistakes
def _mutant(score_rule="max", force_own=True, narrow=True, chunk_of_key=False):
    def blocks(q, k, stages, scale=None):
        stages = O.check_stages(stages)
        N, d = q.shape
        scale = O.default_scale(d) if scale is None else scale
        NB = (N + 63) // 64
        sel, kept_all = [], []
        for m in range(NB):
            t = O.hip_token_scores(q, k, m, scale)
            blk = np.arange(t.size) // 64
            cand = np.ones(t.size, dtype=bool)
            per = []
            for c, keep in stages:
                chunk = (np.arange(t.size) // c) if chunk_of_key else blk // c
                own = m // c
                live = np.unique(chunk[cand] if narrow else chunk)
                pool = cand if narrow else np.ones_like(cand)
                agg = np.max if score_rule == "max" else np.mean
                score = {int(x): float(agg(t[pool & (chunk == x)])) for x in live}
                if force_own:
                    others = sorted((x for x in score if x != own), key=lambda x: (-score[x], x))
                    kept = sorted(others[:keep - 1] + [own])
                else:
                    kept = sorted(sorted(score, key=lambda x: (-score[x], x))[:keep])
                per.append(np.array(kept))
                cand &= np.isin(chunk, kept)
            sel.append(np.unique(blk[cand]).astype(np.int64))
            kept_all.append(per)
        return sel, kept_all
    return blocks

PINS = [lambda: test_keep_all_is_dense_causal(640)] + \
       [lambda kp=kp: test_single_stage_is_brute_force_block_max_ranking(kp) for kp in (1, 3, 5)] + \
       [lambda s=s: test_covering_stages_equal_one_stage(s) for s in range(2)] + \
       [test_stages_narrow_the_candidates, test_representative_is_the_best_token_not_the_mean,
        test_zero_keys_closed_form, test_planted_token_is_kept_by_every_later_block,
        test_kept_counts]

@pytest.mark.parametrize("name,fn", [
    ("mean representative", _mutant(score_rule="mean")),
    ("own chunk not forced", _mutant(force_own=False)),
    ("candidates not narrowed", _mutant(narrow=False)),
    ("chunks counted in tokens", _mutant(chunk_of_key=True)),
])
def test_planted_mistakes_are_caught(monkeypatch, name, fn):
    monkeypatch.setattr(O, "hierarchical_blocks", fn)
    caught = 0
    for t in PINS:
        try:
            t()
        except AssertionError:
            caught += 1
    assert caught > 0, f"no pin catches: {name}"
