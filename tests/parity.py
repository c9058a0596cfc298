"""Helpers shared by the GPU parity tests: run the CUDA path through the C ABI
with index export, and compare it with the oracle under the stated rules.

Rules (the method's stated parity tolerances):
* index sets are compared exactly; a top-k set may differ from the oracle's
  only by elements whose oracle score lies within 1e-5 (relative) of the
  oracle's k-th score, and then the downstream format and outputs are checked
  against the oracle run on the GPU's own sets;
* bf16 outputs: max |diff| <= 1e-2 and mean |diff| <= 1e-3 against the fp64
  oracle given identical indices, where the 1e-2 bound covers the arithmetic
  before the final bf16 cast: each element may differ by 1e-2 plus half a bf16
  ulp of the oracle value (the cast alone moves a value in [4, 8) by up to
  1.56e-2, so no bf16 output can meet a bare 1e-2 there).
"""
from __future__ import annotations

import numpy as np
import torch

from oracle import msa_oracle as O
from dynamic_sparse_attention_slash_gb300 import msa

MAX_TOL = 1e-2
MEAN_TOL = 1e-3
TIE_REL = 1e-5


def to_np(t):
    return t.detach().to("cpu", torch.float64).numpy()


def run_vs(q, k, v, vertical_topk, slash, last_q=64, heads=None, scale=None):
    """CUDA vertical-slash call with index export; returns (out, export dict of numpy)."""
    B, Hq, N, _ = q.shape
    heads_l = list(range(Hq)) if heads is None else list(heads)
    U = B * len(heads_l)
    kv, ks = min(vertical_topk, N), min(slash, N)
    dev = q.device
    ex = vs_export_buffers(U, N, kv, ks, dev)
    out = msa.msa_vertical_slash(q, k, v, vertical_topk, slash, last_q=last_q, heads=heads,
                                 export=ex, scale=scale)
    torch.cuda.synchronize()
    return out, {name: t.cpu().numpy() for name, t in ex.items()}


def vs_export_buffers(U, N, kv, ks, dev):
    """Device buffers for every vertical-slash export of U units (sizes as in
    include/msa.h)."""
    NB, NQ = (N + 63) // 64, (N + 127) // 128
    return {
        "v_score": torch.empty(U, N, dtype=torch.float32, device=dev),
        "s_score": torch.empty(U, N, dtype=torch.float32, device=dev),
        "vertical": torch.empty(U, kv, dtype=torch.int32, device=dev),
        "slash": torch.empty(U, ks, dtype=torch.int32, device=dev),
        "tile_dist": torch.empty(U, (NB + 32) // 32, dtype=torch.int32, device=dev),
        "col_count": torch.empty(U, NB, dtype=torch.int32, device=dev),
        "col_chunks": torch.empty(U, NQ, ((kv + 127) // 128 + 31) // 32, dtype=torch.int32,
                                  device=dev),
    }


def vs_block_columns(V, S, N, m):
    """Columns of row block m (the oracle's format rule), from the chosen sets."""
    act = O.vs_active_tiles(S, N, [m])[0]
    last_row = min(N, (m + 1) * 64) - 1
    c = V[V <= last_row]
    return c[~act[c // 64]]


def check_vs_columns(ex, u, V, S, N, blocks, what):
    """The exported column format of unit u, compared exactly with the oracle's
    columns on row blocks `blocks`: the per-row-block count, and every
    128-position chunk of the vertical list that the block's query tile
    needs (the chunk words of a query tile are checked when both of its row
    blocks are in `blocks`, or when its second block is past the sequence)."""
    NB = (N + 63) // 64
    words = np.asarray(ex["col_chunks"][u], dtype=np.int64) & 0xFFFFFFFF
    cols = {m: vs_block_columns(V, S, N, m) for m in blocks}
    for m in blocks:
        assert int(ex["col_count"][u, m]) == cols[m].size, (
            f"{what}: row block {m} has {int(ex['col_count'][u, m])} columns, oracle {cols[m].size}")
    for p in sorted({m // 2 for m in blocks}):
        pair = [m for m in (2 * p, 2 * p + 1) if m < NB]
        if not all(m in cols for m in pair):
            continue
        want = np.zeros(words.shape[1], dtype=np.int64)
        for m in pair:
            for c in np.unique(np.searchsorted(V, cols[m]) // 128):
                want[c // 32] |= 1 << int(c % 32)
        np.testing.assert_array_equal(words[p], want, err_msg=f"{what}: chunk mask of query tile {p}")


def run_bs(q, k, v, topk, heads=None):
    B, Hq, N, _ = q.shape
    heads_l = list(range(Hq)) if heads is None else list(heads)
    U = B * len(heads_l)
    NB = (N + 63) // 64
    kb = min(topk, NB)
    dev = q.device
    ex = {
        "block_count": torch.empty(U, NB, dtype=torch.int32, device=dev),
        "block_ids": torch.empty(U, NB, kb, dtype=torch.int32, device=dev),
    }
    out = msa.msa_block_sparse(q, k, v, topk, heads=heads, export=ex)
    torch.cuda.synchronize()
    return out, {name: t.cpu().numpy() for name, t in ex.items()}


def run_hip(q, k, v, stages, heads=None, kv_select=None):
    """CUDA hierarchical-head call with block export; returns (out, export dict of numpy)."""
    B, Hq, N, _ = q.shape
    U = B * (Hq if heads is None else len(heads))
    NB = (N + 63) // 64
    kb = min(int(stages[-1][1]), NB)
    ex = {"block_count": torch.empty(U, NB, dtype=torch.int32, device=q.device),
          "block_ids": torch.empty(U, NB, kb, dtype=torch.int32, device=q.device)}
    out = msa.msa_hierarchical(q, k, v, stages, heads=heads, export=ex, kv_select=kv_select)
    torch.cuda.synchronize()
    return out, {name: t.cpu().numpy() for name, t in ex.items()}


def check_hip_blocks(counts, ids, qn, kn, stages, row_blocks, what):
    """Kept blocks of one hierarchical head (counts [NB], ids [NB][kb] from the
    GPU) against the oracle on `row_blocks`.  Exact, except for a row block
    where some stage's cut is a near-tie in the oracle's own chunk scores (the
    last kept and the first dropped other chunk within 1e-5 relative): there
    the GPU may keep either chunk, so only the structure of its set is checked.
    Returns ({m: GPU blocks} for the attention check, number of near-tie rows)."""
    sel, _, scores = O.hierarchical_blocks(qn, kn, stages, row_blocks=row_blocks, with_scores=True)
    keep_last = int(stages[-1][1])
    got_sel, near = {}, 0
    for i, m in enumerate(row_blocks):
        cnt = int(counts[m])
        got = np.asarray(ids[m, :cnt], dtype=np.int64)
        assert cnt >= 1 and got[-1] == m and np.all(np.diff(got) > 0), f"{what} m{m}: {got}"
        assert cnt <= keep_last, f"{what} m{m}: {cnt} blocks"
        tie = False
        for st, (c, keep) in enumerate(stages):
            others = sorted((val for x, val in scores[i][st].items() if x != m // c), reverse=True)
            if keep >= 2 and len(others) >= keep:
                a, b = others[keep - 2], others[keep - 1]
                tie |= abs(a - b) <= TIE_REL * max(abs(a), 1e-30)
        if tie:
            near += 1
        else:
            np.testing.assert_array_equal(got, sel[i], err_msg=f"{what} m{m}")
        got_sel[m] = got
    return got_sel, near


def check_topk(gpu_set, oracle_scores, k, what):
    """Exact set equality, except near-ties at the k-th score (see module doc)."""
    ref = O.topk_indices(oracle_scores, k)
    got = np.asarray(gpu_set, dtype=np.int64)
    assert np.all(np.diff(got) > 0), f"{what}: GPU set not strictly ascending"
    if np.array_equal(got, ref):
        return 0
    assert got.size == ref.size, f"{what}: size {got.size} != {ref.size}"
    kth = np.sort(oracle_scores)[::-1][min(k, oracle_scores.size) - 1]
    diff = np.setxor1d(got, ref)
    tol = TIE_REL * max(abs(kth), 1e-30)
    bad = diff[np.abs(oracle_scores[diff] - kth) > tol]
    assert bad.size == 0, (f"{what}: {diff.size} differing indices, {bad.size} not near-ties; "
                           f"e.g. {bad[:5]} scores {oracle_scores[bad[:5]]} vs kth {kth}")
    return int(diff.size)


def dist_bits_to_active(words, NB):
    """Expand the exported tile-distance bitset into the [NB, NB] active-tile matrix."""
    words = np.asarray(words, dtype=np.int64) & 0xFFFFFFFF
    bits = np.array([(words[t >> 5] >> (t & 31)) & 1 for t in range(NB)], dtype=bool)
    act = np.zeros((NB, NB), dtype=bool)
    for m in range(NB):
        act[m, :m + 1] = bits[m - np.arange(m + 1)]
    return act


def half_ulp_bf16(x):
    """Half the bf16 spacing at |x| (8 significant bits)."""
    a = np.abs(np.asarray(x, dtype=np.float64))
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -126)))
    return np.exp2(e - 8)


def compare_out(got, ref, what):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    d = np.abs(got - ref)
    excess = d - (MAX_TOL + half_ulp_bf16(ref))
    mx, mean = float(d.max()), float(d.mean())
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    at = np.unravel_index(int(excess.argmax()), d.shape)
    assert excess.max() <= 0 and mean <= MEAN_TOL, (
        f"{what}: |d| {d[at]:.3e} at {tuple(int(x) for x in at)} (ref {ref[at]:.5f}, "
        f"got {got[at]:.5f}) exceeds 1e-2 + half ulp; max|d| {mx:.3e} mean|d| {mean:.3e}")
    return mx, mean
