"""Kernel-aware work counts: the (query, key) pairs a call's attention kernel
computes, from the index data the call itself built (exported through
msa_index_export).  Host-side bookkeeping for the benchmark and the pattern
search; the attention FLOPs of a head are 4 * d * pairs (2 for Q K^T and 2 for
P V per pair and head dimension).
"""
from __future__ import annotations

import numpy as np


def vs_pairs(tile_dist_words, vertical, N: int) -> int:
    """Admitted (i, j) pairs, j <= i, of one vertical-slash head: active 64x64
    tiles (the diagonal one triangular) plus the uncovered vertical columns."""
    NB = N // 64
    words = np.asarray(tile_dist_words, dtype=np.int64) & 0xFFFFFFFF
    t = np.arange(NB)
    bits = ((words[t >> 5] >> (t & 31)) & 1).astype(np.int64)
    cum = np.cumsum(bits)  # cum[m] = #{t in D, t <= m}
    diag = int(bits[0])
    total = int(((cum - diag) * 4096).sum()) + diag * 2080 * NB
    V = np.asarray(vertical, dtype=np.int64)
    mj = V // 64
    # row blocks m > mj whose distance m - mj is not in D contribute 64 rows
    upto = NB - 1 - mj
    in_d = np.where(upto >= 1, cum[np.maximum(upto, 0)] - diag, 0)
    total += int((64 * (upto - in_d)).sum())
    if not diag:  # the key's own row block: rows j..64*mj+63
        total += int((64 * (mj + 1) - V).sum())
    return total


def bs_pairs(block_count) -> int:
    c = np.asarray(block_count, dtype=np.int64)
    return int(((c - 1) * 4096 + 2080).sum())


def st_pairs(N: int, init_num: int, local: int) -> int:
    total = 0
    for m in range(N // 64):
        blocks = set(range(min(init_num, m + 1))) | set(range(max(0, m - local + 1), m + 1))
        total += 2080 + 4096 * (len(blocks) - 1)
    return total
