"""Kernel-aware work counts: the (query, key) pairs a call's attention kernel
computes, from the index data the call itself built (exported through
msa_index_export).  Host-side bookkeeping for the benchmark and the pattern
search; the attention FLOPs of a head are 4 * d * pairs (2 for Q K^T and 2 for
P V per pair and head dimension).
"""
from __future__ import annotations

import numpy as np


def _rows(N: int) -> np.ndarray:
    """Real rows of each 64-row block (only the last one can be partial)."""
    NB = (N + 63) // 64
    r = np.full(NB, 64, dtype=np.int64)
    r[-1] = N - 64 * (NB - 1)
    return r


def vs_pairs(tile_dist_words, vertical, N: int) -> int:
    """Admitted (i, j) pairs, j <= i, of one vertical-slash head: active 64x64
    tiles (the diagonal one triangular) plus the uncovered vertical columns.
    A partial last row block has fewer rows; its tiles follow the padded-block
    rule, and keys past N are never admitted (they lie after every row)."""
    NB = (N + 63) // 64
    rows = _rows(N)
    R = int(rows[-1])
    words = np.asarray(tile_dist_words, dtype=np.int64) & 0xFFFFFFFF
    t = np.arange(NB)
    bits = ((words[t >> 5] >> (t & 31)) & 1).astype(np.int64)
    cum = np.cumsum(bits)  # cum[m] = #{t in D, t <= m}
    diag = int(bits[0])
    # off-diagonal active tiles of row block m: (cum[m] - diag) full key blocks
    total = int(((cum - diag) * 64 * rows).sum()) + diag * int((rows * (rows + 1) // 2).sum())
    V = np.asarray(vertical, dtype=np.int64)
    mj = V // 64
    # row blocks m > mj whose distance m - mj is not in D contribute their rows
    upto = NB - 1 - mj
    has = upto >= 1
    in_d = np.where(has, cum[np.maximum(upto, 0)] - diag, 0)
    last_in_d = np.where(has, bits[np.maximum(upto, 0)], 0)
    rows_after = 64 * upto - (64 - R) * has                  # sum of rows(m), mj < m < NB
    rows_in_d = 64 * in_d - (64 - R) * last_in_d              # of those, with m - mj in D
    total += int((rows_after - rows_in_d).sum())
    if not diag:  # the key's own row block: rows j .. end of the block
        total += int((np.minimum(64 * (mj + 1), N) - V).sum())
    return total


def vs_exact_line_pairs(vertical, slash, N: int) -> int:
    """Pairs (i, j), j <= i < N, on the chosen lines themselves: j a chosen
    vertical column or i - j a chosen slash offset, without the expansion to
    64x64 tiles that the kernels compute (a diagnostic of the sparse format's
    overhead).  Column j covers rows j .. N-1 (N - j pairs), offset o covers
    rows o .. N-1 (N - o pairs), and a pair on both a column j and an offset o
    (j + o <= N - 1) is counted once."""
    V = np.sort(np.asarray(vertical, dtype=np.int64))
    S = np.asarray(slash, dtype=np.int64)
    both = int(np.searchsorted(V, N - S, side="left").sum())  # per o: columns j < N - o
    return int((N - V).sum() + (N - S).sum() - both)


def bs_pairs(block_count, N: int | None = None) -> int:
    """Pairs of a block-sparse head (or stacked heads) from its per-row-block
    kept-block counts [.., NB]: the diagonal block triangular, the others full.
    N (when not a multiple of 64) shortens the last row block."""
    c = np.asarray(block_count, dtype=np.int64)
    if N is None or N % 64 == 0:
        return int(((c - 1) * 4096 + 2080).sum())
    R = N - 64 * (c.shape[-1] - 1)
    rows = np.full(c.shape[-1], 64, dtype=np.int64)
    rows[-1] = R
    return int(((c - 1) * 64 * rows + rows * (rows + 1) // 2).sum())


def st_pairs(N: int, init_num: int, local: int) -> int:
    """Pairs of a streaming head: sinks plus the local window per row block."""
    rows = _rows(N)
    total = 0
    for m, r in enumerate(rows):
        blocks = set(range(min(init_num, m + 1))) | set(range(max(0, m - local + 1), m + 1))
        total += int(r * (r + 1) // 2 + 64 * r * (len(blocks) - 1))
    return total
