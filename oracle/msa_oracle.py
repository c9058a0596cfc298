"""CPU oracle for MInference-style dynamic sparse prefill attention (fp64, numpy).

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports this module:
only the tests, the package smoke check and the CPU-baseline leg of the
benchmark may call it.  It shares no code with the CUDA path.

Every function restates one step of the method in plain numpy, in float64,
from bf16 inputs converted exactly.  Sources, by page title and section:

* [MInf-1]  MInference 1.0 overview (developer.volcengine.com article),
            section 1 "Problem Formulation": A(M) = Softmax(Q K^T / sqrt(d) - c (1 - M)) V
            with a binary dynamic mask M, a scale of sqrt(d) and a constant c that
            drives masked entries to ~0 after the softmax.
* [MInf-2.2] same page, section 2.2 "Sparsity Indices Approximation and Dynamic
            Sparse Attention Calculation": the vertical-slash head (estimate A-hat
            from a matmul of the last queries with all keys, pick the vertical
            and slash index sets, convert them to a sparse format, run
            block-sparse attention) and the block-sparse head (mean-pool Q and
            K, block-level weights, top-k block index, sparse attention).
* [MInf-2.1] same page, section 2.1 "Kernel-Aware Optimal Sparse Pattern
            Search": candidates of each pattern share a FLOPs target measured
            as the kernel computes it; one reference example picks, per head,
            the pattern and setting with the best recall of the attention
            output.
* [MInf-API] same page, the "using only the kernel" listing: the entry points
            vertical_slash_sparse_attention(q,k,v,vertical_topk,slash),
            block_sparse_attention(q,k,v,topk) and
            streaming_forward(q,k,v,init_num,local_window_num).
* [HiP-prune] InfiniteHiP summary (dtcms.com page), section "modular
            hierarchical token pruning algorithm": the key sequence is split
            into fixed-length chunks, each chunk is represented by its token
            with the highest attention score, only the most important chunks
            go on to the next pruning module; stacked modules refine the
            block-sparse mask stage by stage for the current query block.
* [KV-1.5x] "How KV sparsity achieves 1.5x acceleration for vLLM" (Novita AI
            blog), section "Key Techniques / 2. Attention modification": the
            token score is a sum of softmax probabilities over a window of the
            last queries, computed from the row max and the row sum l that the
            attention pass exports; each head keeps its top-scoring tokens.

Readings where the pages are silent or garbled (the plainest completion in
each case):

* masked entries are excluded exactly (c -> infinity); a row with no allowed
  key outputs zeros;
* the estimate uses the last ``last_q`` (default 64) query rows with a causal
  softmax over every key j <= i;
* the vertical score of key j is the column sum of A-hat, the slash score of
  offset o = i - j is the sum of A-hat along that diagonal, o in [0, N);
* top-k orders by score descending, ties to the lower index, and returns the
  chosen indices in ascending order; k is clamped to the number of candidates;
* the sparse format expands every selected diagonal to the 64x64 key tiles it
  crosses and keeps vertical columns that no active tile of the row block
  already covers; for N not a multiple of 64 it is built over the sequence
  padded to the next multiple (MInference's block kernels work on padded
  blocks), so every row block counts 64 rows; block-sparse pooling averages
  the real rows of a partial block;
* the block-sparse head keeps the diagonal block plus the top-(topk-1) earlier
  blocks by pooled score; streaming keeps blocks [0, init_num) and the
  ``local_window_num`` blocks ending at the query's own block;
* the hierarchical pruning head scores a key token for query block m as the
  block's mean-pooled query against the key, scale * Qhat_m . k_j, over the
  causal candidates j <= 64m + 63; chunks are aligned groups of c 64-token
  blocks, c decreasing stage by stage down to 1, each dividing the previous;
  a chunk's score is its highest candidate token score; every stage keeps the
  chunk holding block m plus the keep-1 best other chunks (ties to the lower
  chunk), as the block-sparse head keeps its diagonal block;
* query head h reads KV head h // (Hq / Hkv);
* KV selection: the exported normaliser is lse = rowmax + ln(l); a window row's
  probabilities are those of the attention the call computed (zero outside
  its key set J_i); the score is per query head; no pooling of the score
  before its top-k (the page names none);
* pattern search: "recall of the attention output" is the dense attention
  mass a mask keeps, averaged over rows; per pattern the search uses the most
  expensive setting within the FLOPs budget; the best recall wins, ties to the
  earlier pattern.

Parity pins for every function live in tests/test_oracle_*.py.
"""
from __future__ import annotations

import numpy as np

BLOCK = 64


# ----------------------------------------------------------------------------- helpers
def as_f64(x) -> np.ndarray:
    """bf16/fp32 torch tensor or array -> float64 numpy array (exact widening)."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            return x.detach().to("cpu", torch.float64).numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.asarray(x, dtype=np.float64)


def default_scale(d: int) -> float:
    """1 / sqrt(d) [MInf-1]."""
    return 1.0 / np.sqrt(d)


# ----------------------------------------------------------------------------- attention given a mask
def attend_rows(q: np.ndarray, k: np.ndarray, v: np.ndarray, rows, allowed_keys, scale: float):
    """Masked softmax attention for selected query rows [MInf-1].

    q, k, v: [N, d] float64 for one query head and its KV head.
    rows: iterable of query indices i.
    allowed_keys(i) -> 1-D integer array (or boolean mask over [0, N)) of the keys
    the mask M admits for row i; keys j > i are removed here (causal).
    Returns out [len(rows), d] and the per-row key counts |J_i|.

    A masked entry gets weight exactly 0 (c -> infinity); a row with no admitted
    key outputs zeros.
    """
    rows = list(rows)
    N, d = q.shape
    out = np.zeros((len(rows), d), dtype=np.float64)
    counts = np.zeros(len(rows), dtype=np.int64)
    for r, i in enumerate(rows):
        J = np.asarray(allowed_keys(i))
        admit = np.zeros(i + 1, dtype=bool)
        if J.dtype == bool:
            admit[:] = J[:i + 1]
        else:
            admit[J[J <= i]] = True
        counts[r] = int(admit.sum())
        if counts[r] == 0:
            continue
        z = (k[:i + 1] @ q[i]) * scale
        z = np.where(admit, z, -np.inf)
        p = np.exp(z - z.max())
        p /= p.sum()
        out[r] = p @ v[:i + 1]
    return out, counts


def attend_blocks(q, k, v, block_mask, scale: float):
    """Masked softmax attention for all rows, mask given per 64-row block.

    block_mask(m) -> boolean [N] over keys admitted for every row of row block m
    (the causal cut j <= i is applied per row here).  Same arithmetic as
    attend_rows, evaluated 64 rows at a time.
    """
    N, d = q.shape
    out = np.zeros((N, d), dtype=np.float64)
    counts = np.zeros(N, dtype=np.int64)
    for m in range((N + BLOCK - 1) // BLOCK):
        r0, r1 = m * BLOCK, min(N, (m + 1) * BLOCK)
        allow = np.asarray(block_mask(m), dtype=bool)[:r1]
        idx = np.arange(r1)
        M = np.broadcast_to(allow, (r1 - r0, r1)) & (idx[None, :] <= np.arange(r0, r1)[:, None])
        counts[r0:r1] = M.sum(1)
        z = (q[r0:r1] @ k[:r1].T) * scale
        z = np.where(M, z, -np.inf)
        zmax = z.max(1, keepdims=True)
        zmax = np.where(np.isfinite(zmax), zmax, 0.0)
        p = np.exp(z - zmax)
        den = p.sum(1, keepdims=True)
        res = p @ v[:r1]
        out[r0:r1] = np.divide(res, den, out=np.zeros_like(res), where=den > 0)
    return out, counts


def dense_causal(q, k, v, scale: float):
    """Dense causal attention: the all-ones mask [MInf-1]."""
    N = q.shape[0]
    return attend_blocks(q, k, v, lambda m: np.ones(N, dtype=bool), scale)[0]


# ----------------------------------------------------------------------------- vertical-slash head
def estimate_vs(q, k, last_q: int, scale: float):
    """Estimated attention of the last queries and its line scores [MInf-2.2], [KV-1.5x].

    A-hat[r, j] = softmax over j <= i of scale * q_i . k_j, for the rows
    i = N - L + r, L = min(last_q, N).  Returns (v_score [N], s_score [N], A_hat [L, N]):
    v_score[j] = sum over rows of A-hat[r, j]            (vertical line j)
    s_score[o] = sum over rows of A-hat[r, i - o], i-o>=0 (slash line, offset o)
    """
    N = q.shape[0]
    L = min(last_q, N)
    rows = np.arange(N - L, N)
    z = (q[rows] @ k.T) * scale
    keys = np.arange(N)
    causal = keys[None, :] <= rows[:, None]
    z = np.where(causal, z, -np.inf)
    m = z.max(1, keepdims=True)
    e = np.exp(z - m)
    ell = e.sum(1, keepdims=True)
    A = e / ell
    v_score = A.sum(0)
    s_score = np.zeros(N, dtype=np.float64)
    for r, i in enumerate(rows):
        # keys j = i, i-1, ..., 0 lie on offsets o = 0, 1, ..., i
        s_score[: i + 1] += A[r, i::-1]
    return v_score, s_score, A


def topk_indices(scores, k: int) -> np.ndarray:
    """Top-k by score descending, ties to the lower index; returned ascending."""
    scores = np.asarray(scores, dtype=np.float64)
    k = int(min(max(k, 0), scores.size))
    order = np.argsort(-scores, kind="stable")
    return np.sort(order[:k]).astype(np.int64)


def vs_active_tiles(slash_idx, N: int, row_blocks=None) -> np.ndarray:
    """64x64 tiles crossed by the selected diagonals [MInf-2.2] (sparse format, tile part).

    Tile (m, n), n <= m, is active iff some selected offset o has a row
    i in [64m, 64m+63] with i - o inside key tile n, i.e. iff the key range
    [64m - o, 64m + 63 - o] (cut at 0) meets [64n, 64n + 63].
    Returns a boolean [NB, NB] matrix (row block m, key block n); with
    `row_blocks`, a [len(row_blocks), NB] matrix for those row blocks only.
    When N is not a multiple of 64 the format is built over the sequence
    padded to the next multiple (the last row block counts as 64 rows); the
    causal cut later removes the padded keys.
    """
    NB = (N + BLOCK - 1) // BLOCK
    S = np.asarray(slash_idx, dtype=np.int64)
    blocks = range(NB) if row_blocks is None else list(row_blocks)
    active = np.zeros((len(blocks), NB), dtype=bool)
    for r, m in enumerate(blocks):
        first_row = m * BLOCK
        last_row = (m + 1) * BLOCK - 1
        lo = first_row - S
        hi = last_row - S
        keep = hi >= 0
        lo = np.maximum(lo[keep], 0)
        hi = hi[keep]
        for n_lo, n_hi in zip(lo // BLOCK, hi // BLOCK):
            active[r, n_lo:n_hi + 1] = True
    return active


def vs_columns(vertical_idx, active: np.ndarray, N: int):
    """Column part of the sparse format [MInf-2.2]: per row block m, the selected
    vertical keys j <= last row of m whose key tile is not active for m; ascending."""
    V = np.asarray(vertical_idx, dtype=np.int64)
    NB = active.shape[0]
    cols = []
    for m in range(NB):
        last_row = min(N, (m + 1) * BLOCK) - 1
        c = V[V <= last_row]
        c = c[~active[m, c // BLOCK]]
        cols.append(c)
    return cols


def vs_row_block_mask(slash_idx, vertical_idx, N):
    """Keys admitted for row block m, built for that block alone from the chosen
    offsets and columns (same rule as vs_active_tiles + vs_columns; for long
    sequences where the full [NB, NB] tile matrix is not needed)."""
    V = np.asarray(vertical_idx, dtype=np.int64)

    def mask(m):
        act = vs_active_tiles(slash_idx, N, [m])[0]
        last_row = min(N, (m + 1) * BLOCK) - 1
        c = V[V <= last_row]
        c = c[~act[c // BLOCK]]
        allow = np.repeat(act, BLOCK)[:N].copy()
        allow[c] = True
        return allow
    return mask


def vs_block_mask(active, cols, N):
    """Keys admitted for row block m: active tiles plus the block's columns."""
    def mask(m):
        allow = np.repeat(active[m], BLOCK)[:N].copy()
        allow[cols[m]] = True
        return allow
    return mask


def vertical_slash_indices(q, k, vertical_topk: int, slash: int, last_q: int = 64,
                           scale: float | None = None):
    """Index construction of one vertical-slash head [MInf-2.2]."""
    N, d = q.shape
    scale = default_scale(d) if scale is None else scale
    v_score, s_score, _ = estimate_vs(q, k, last_q, scale)
    V = topk_indices(v_score, vertical_topk)
    S = topk_indices(s_score, slash)
    active = vs_active_tiles(S, N)
    cols = vs_columns(V, active, N)
    return {"v_score": v_score, "s_score": s_score, "vertical": V, "slash": S,
            "active": active, "columns": cols}


def vertical_slash_head(q, k, v, vertical_topk: int, slash: int, last_q: int = 64,
                        scale: float | None = None):
    """One vertical-slash head end to end: indices, then block-sparse attention."""
    N, d = q.shape
    scale = default_scale(d) if scale is None else scale
    idx = vertical_slash_indices(q, k, vertical_topk, slash, last_q, scale)
    out, counts = attend_blocks(q, k, v, vs_block_mask(idx["active"], idx["columns"], N), scale)
    idx["nnz"] = int(counts.sum())
    return out, idx


# ----------------------------------------------------------------------------- block-sparse head
def mean_pool(x, N: int):
    """Mean over each 64-row block [MInf-2.2] (block-sparse head, step 1)."""
    NB = (N + BLOCK - 1) // BLOCK
    return np.stack([x[m * BLOCK:min(N, (m + 1) * BLOCK)].mean(0) for m in range(NB)])


def block_scores(q, k, scale: float):
    """Pooled block logits scale * Qhat_m . Khat_n (before the row softmax) [MInf-2.2]."""
    N = q.shape[0]
    return (mean_pool(q, N) @ mean_pool(k, N).T) * scale


def block_sparse_blocks(q, k, topk: int, scale: float | None = None, row_blocks=None):
    """Selected key blocks per row block [MInf-2.2]: the diagonal block plus the
    top-(topk-1) earlier blocks by pooled score (ties to the lower block);
    min(topk, m+1) blocks, ascending.  With row_blocks given, only those row
    blocks are scored and selected: the lists and the score rows follow
    row_blocks' order (each score row is that row of the full score matrix)."""
    N, d = q.shape
    scale = default_scale(d) if scale is None else scale
    if row_blocks is None:
        S = block_scores(q, k, scale)
        rows = range(S.shape[0])
    else:
        rows = [int(m) for m in row_blocks]
        S = (mean_pool(q, N)[rows] @ mean_pool(k, N).T) * scale
    sel = []
    for r, m in enumerate(rows):
        earlier = topk_indices(S[r, :m], max(topk - 1, 0)) if m > 0 else np.zeros(0, np.int64)
        sel.append(np.sort(np.concatenate([earlier, [m]]).astype(np.int64)))
    return sel, S


def block_mask_from_blocks(sel, N):
    def mask(m):
        allow = np.zeros(((N + BLOCK - 1) // BLOCK) * BLOCK, dtype=bool)
        for n in sel[m]:
            allow[n * BLOCK:(n + 1) * BLOCK] = True
        return allow[:N]
    return mask


def block_sparse_head(q, k, v, topk: int, scale: float | None = None):
    N, d = q.shape
    scale = default_scale(d) if scale is None else scale
    sel, S = block_sparse_blocks(q, k, topk, scale)
    out, counts = attend_blocks(q, k, v, block_mask_from_blocks(sel, N), scale)
    return out, {"blocks": sel, "block_scores": S, "nnz": int(counts.sum())}


# ----------------------------------------------------------------------------- streaming head
def streaming_blocks(m: int, init_num: int, local_window_num: int) -> np.ndarray:
    """Key blocks of row block m for the streaming / A-shape head [MInf-API]:
    the sink blocks [0, init_num) and the local window [m - local + 1, m], cut at
    [0, m], without repeats, ascending."""
    sink = set(range(0, min(init_num, m + 1)))
    local = set(range(max(0, m - local_window_num + 1), m + 1))
    return np.array(sorted(sink | local), dtype=np.int64)


def streaming_head(q, k, v, init_num: int, local_window_num: int, scale: float | None = None):
    N, d = q.shape
    scale = default_scale(d) if scale is None else scale
    NB = (N + BLOCK - 1) // BLOCK
    sel = [streaming_blocks(m, init_num, local_window_num) for m in range(NB)]
    out, counts = attend_blocks(q, k, v, block_mask_from_blocks(sel, N), scale)
    return out, {"blocks": sel, "nnz": int(counts.sum())}


# ----------------------------------------------------------------------------- hierarchical pruning head
def check_stages(stages):
    """Stages [(chunk_blocks, keep), ...] of the hierarchical head: chunk sizes
    in 64-token blocks, decreasing, each dividing the one before, the last 1;
    keep >= 1 chunks per stage."""
    stages = [(int(c), int(kp)) for c, kp in stages]
    assert stages and stages[-1][0] == 1, "the last stage must select single blocks"
    for (c0, _), (c1, _) in zip(stages, stages[1:]):
        assert c0 > c1 and c0 % c1 == 0, "chunk sizes must decrease, each dividing the previous"
    assert all(c >= 1 and kp >= 1 for c, kp in stages)
    return stages


def hip_token_scores(q, k, m: int, scale: float) -> np.ndarray:
    """Attention score of every candidate key token for query block m
    [HiP-prune]: scale * Qhat_m . k_j for the keys j <= 64m + 63 (cut at N),
    Qhat_m the mean of the block's query rows."""
    N = q.shape[0]
    qhat = q[m * BLOCK:min(N, (m + 1) * BLOCK)].mean(0)
    return (k[:min(N, (m + 1) * BLOCK)] @ qhat) * scale


def hierarchical_blocks(q, k, stages, scale: float | None = None, row_blocks=None,
                        with_scores: bool = False):
    """Kept key blocks per query block after multi-stage pruning [HiP-prune].

    For query block m the candidates start as every key j <= 64m + 63.  Stage
    (c, keep) splits the candidate keys into chunks of c consecutive 64-token
    blocks (chunk x = blocks [x c, (x + 1) c)); a chunk's score is the score of
    its representative, the candidate token with the highest attention score
    (hip_token_scores); the chunk holding block m and the keep - 1 other
    chunks with the highest scores (ties to the lower chunk) stay, and the
    keys of every other chunk leave the candidates.  The last stage has c = 1:
    its kept blocks, ascending, are the block-sparse mask of m (at most
    min(keep_last, m + 1) blocks).  Returns (blocks per query block, the
    per-stage kept chunk lists [m][stage]), for every query block or for
    those in `row_blocks`; with_scores adds the per-stage chunk scores
    ({chunk: score} for every chunk holding a candidate) as a third item."""
    stages = check_stages(stages)
    N, d = q.shape
    scale = default_scale(d) if scale is None else scale
    NB = (N + BLOCK - 1) // BLOCK
    sel, kept_chunks, stage_scores = [], [], []
    for m in (range(NB) if row_blocks is None else row_blocks):
        t = hip_token_scores(q, k, m, scale)
        blk = np.arange(t.size) // BLOCK  # key block of every candidate key
        cand = np.ones(t.size, dtype=bool)
        per_stage, per_scores = [], []
        for c, keep in stages:
            chunk = blk // c
            own = m // c
            live = np.unique(chunk[cand])
            score = {int(x): float(t[cand & (chunk == x)].max()) for x in live}
            others = sorted((x for x in score if x != own), key=lambda x: (-score[x], x))
            kept = sorted(others[:keep - 1] + [own])
            per_stage.append(np.array(kept, dtype=np.int64))
            per_scores.append(score)
            cand &= np.isin(chunk, kept)
        sel.append(np.unique(blk[cand]).astype(np.int64))
        kept_chunks.append(per_stage)
        stage_scores.append(per_scores)
    if with_scores:
        return sel, kept_chunks, stage_scores
    return sel, kept_chunks


def hierarchical_head(q, k, v, stages, scale: float | None = None):
    """One hierarchical-pruning head end to end: kept blocks, then block-sparse
    attention over them [HiP-prune], [MInf-1]."""
    N, d = q.shape
    scale = default_scale(d) if scale is None else scale
    sel, kept = hierarchical_blocks(q, k, stages, scale)
    out, counts = attend_blocks(q, k, v, block_mask_from_blocks(sel, N), scale)
    return out, {"blocks": sel, "stage_chunks": kept, "nnz": int(counts.sum())}


# ----------------------------------------------------------------------------- multi-head entry points
def _kv_head(h: int, n_q: int, n_kv: int) -> int:
    return h // (n_q // n_kv)


def vertical_slash_sparse_attention(q, k, v, vertical_topk, slash, last_q=64, heads=None,
                                    scale=None):
    """[MInf-API] vertical_slash_sparse_attention on q [B,Hq,N,d], k/v [B,Hkv,N,d].

    Returns out [B, len(heads), N, d] float64 and the per-(b, h) index records.
    """
    q, k, v = as_f64(q), as_f64(k), as_f64(v)
    B, Hq, N, d = q.shape
    heads = list(range(Hq)) if heads is None else list(heads)
    out = np.zeros((B, len(heads), N, d))
    recs = {}
    for b in range(B):
        for t, h in enumerate(heads):
            g = _kv_head(h, Hq, k.shape[1])
            out[b, t], recs[(b, h)] = vertical_slash_head(q[b, h], k[b, g], v[b, g],
                                                          vertical_topk, slash, last_q, scale)
    return out, recs


def block_sparse_attention(q, k, v, topk, heads=None, scale=None):
    """[MInf-API] block_sparse_attention on q [B,Hq,N,d], k/v [B,Hkv,N,d]."""
    q, k, v = as_f64(q), as_f64(k), as_f64(v)
    B, Hq, N, d = q.shape
    heads = list(range(Hq)) if heads is None else list(heads)
    out = np.zeros((B, len(heads), N, d))
    recs = {}
    for b in range(B):
        for t, h in enumerate(heads):
            g = _kv_head(h, Hq, k.shape[1])
            out[b, t], recs[(b, h)] = block_sparse_head(q[b, h], k[b, g], v[b, g], topk, scale)
    return out, recs


def streaming_forward(q, k, v, init_num, local_window_num, heads=None, scale=None):
    """[MInf-API] streaming_forward on q [B,Hq,N,d], k/v [B,Hkv,N,d]."""
    q, k, v = as_f64(q), as_f64(k), as_f64(v)
    B, Hq, N, d = q.shape
    heads = list(range(Hq)) if heads is None else list(heads)
    out = np.zeros((B, len(heads), N, d))
    recs = {}
    for b in range(B):
        for t, h in enumerate(heads):
            g = _kv_head(h, Hq, k.shape[1])
            out[b, t], recs[(b, h)] = streaming_head(q[b, h], k[b, g], v[b, g], init_num,
                                                     local_window_num, scale)
    return out, recs


def hierarchical_sparse_attention(q, k, v, stages, heads=None, scale=None):
    """The hierarchical pruning head on q [B,Hq,N,d], k/v [B,Hkv,N,d] [HiP-prune]."""
    q, k, v = as_f64(q), as_f64(k), as_f64(v)
    B, Hq, N, d = q.shape
    heads = list(range(Hq)) if heads is None else list(heads)
    out = np.zeros((B, len(heads), N, d))
    recs = {}
    for b in range(B):
        for t, h in enumerate(heads):
            g = _kv_head(h, Hq, k.shape[1])
            out[b, t], recs[(b, h)] = hierarchical_head(q[b, h], k[b, g], v[b, g], stages, scale)
    return out, recs


# ----------------------------------------------------------------------------- KV selection
def row_lse(q, k, rows, block_mask, scale: float) -> np.ndarray:
    """Row normaliser of the masked causal attention [KV-1.5x] (the "rowmax / l"
    pair the attention pass exports, as one number):
    lse_i = ln sum_{j in J_i} exp(z_ij), z_ij = scale * q_i . k_j, where J_i is
    the set of keys j <= i that block_mask(i // 64) admits; -inf for an empty J_i.
    """
    out = np.full(len(rows), -np.inf)
    for r, i in enumerate(rows):
        allow = np.asarray(block_mask(i // BLOCK), dtype=bool)[: i + 1]
        if not allow.any():
            continue
        z = (k[: i + 1][allow] @ q[i]) * scale
        zmax = z.max()
        out[r] = zmax + np.log(np.exp(z - zmax).sum())
    return out


def kv_score(q, k, window_lse, block_mask, window: int, scale: float) -> np.ndarray:
    """Token score for keeping KV entries [KV-1.5x]: for the query rows of the
    instruction window i in [N - window, N),
        S_j = sum over window rows i with j in J_i of exp(z_ij - lse_i),
    i.e. the attention probability of key j in row i under the row normaliser of
    the attention pass, summed over the window ("kq" order on the page: one sum
    per key).  window_lse[r] is lse of row N - window + r.
    """
    N = q.shape[0]
    S = np.zeros(N, dtype=np.float64)
    for r, i in enumerate(range(N - window, N)):
        if not np.isfinite(window_lse[r]):
            continue
        allow = np.asarray(block_mask(i // BLOCK), dtype=bool)[: i + 1]
        keys = np.nonzero(allow)[0]
        z = (k[keys] @ q[i]) * scale
        S[keys] += np.exp(z - window_lse[r])
    return S


def kv_select_head(q, k, block_mask, window: int, keep_k: int, scale: float | None = None,
                   lse_rows=None):
    """KV selection of one head after its attention pass [KV-1.5x]: the row
    normalisers, the window score S and the keep set (the keep_k keys with the
    highest S, ties to the lower index, ascending; top-k as everywhere else).
    lse_rows: rows whose lse is returned (default: every row)."""
    N, d = q.shape
    scale = default_scale(d) if scale is None else scale
    rows = np.arange(N) if lse_rows is None else np.asarray(lse_rows)
    lse = row_lse(q, k, rows, block_mask, scale)
    win = np.arange(N - window, N)
    lse_w = row_lse(q, k, win, block_mask, scale)
    S = kv_score(q, k, lse_w, block_mask, window, scale)
    return {"lse": lse, "lse_rows": rows, "score": S, "keep": topk_indices(S, keep_k)}


# ----------------------------------------------------------------------------- pattern search
def mass_recall(q, k, rows, block_mask, scale: float) -> np.ndarray:
    """Recall of the dense attention that a mask keeps [MInf-2.1]: for each row i,
    sum over j in J_i of the dense causal softmax A_dense[i, j] (1 for the dense
    mask, 0 for a row whose J_i is empty).  Computed from the dense softmax
    itself, not from normalisers."""
    out = np.zeros(len(rows))
    for r, i in enumerate(rows):
        z = (k[: i + 1] @ q[i]) * scale
        a = np.exp(z - z.max())
        a /= a.sum()
        allow = np.asarray(block_mask(i // BLOCK), dtype=bool)[: i + 1]
        out[r] = a[allow].sum()
    return out


def choose_setting(flops, budget: float) -> int:
    """Index of the candidate setting of one pattern that the search uses at a
    FLOPs budget [MInf-2.1] ("candidates of similar cost"): the most expensive
    setting whose kernel FLOPs do not exceed the budget; if every setting
    exceeds it, the cheapest (ties to the earlier setting)."""
    flops = np.asarray(flops, dtype=np.float64)
    fit = np.nonzero(flops <= budget)[0]
    if fit.size:
        return int(fit[np.argmax(flops[fit])])  # argmax: first of equal maxima
    return int(np.argmin(flops))


def choose_pattern(recalls) -> int:
    """Pattern with the highest recall of the attention output [MInf-2.1]; ties
    go to the earlier pattern (vertical-slash, block-sparse, streaming)."""
    return int(np.argmax(np.asarray(recalls, dtype=np.float64)))


def mask_nnz(block_mask, N: int) -> int:
    """Admitted (i, j) pairs, j <= i, of a mask given per 64-row block."""
    total = 0
    for m in range((N + BLOCK - 1) // BLOCK):
        allow = np.asarray(block_mask(m), dtype=bool)[:N]
        c = np.cumsum(allow)
        r0, r1 = m * BLOCK, min(N, (m + 1) * BLOCK)
        total += int(c[r0:r1].sum())
    return total


def pattern_masks(q, k, pattern: str, setting, scale: float):
    """Block mask of one head under one candidate: ("vs", (vertical_topk, slash)),
    ("bs", topk) or ("st", (init_num, local_window_num))."""
    N = q.shape[0]
    if pattern == "vs":
        idx = vertical_slash_indices(q, k, setting[0], setting[1], 64, scale)
        return vs_block_mask(idx["active"], idx["columns"], N)
    if pattern == "bs":
        sel, _ = block_sparse_blocks(q, k, setting, scale)
        return block_mask_from_blocks(sel, N)
    NB = (N + BLOCK - 1) // BLOCK
    return block_mask_from_blocks([streaming_blocks(m, setting[0], setting[1]) for m in range(NB)], N)


def pattern_search_head(q, k, candidates, budget_flops: float, rows=None, scale=None):
    """Kernel-aware pattern search for one head [MInf-2.1].

    candidates: {"vs": [(vertical_topk, slash), ...], "bs": [topk, ...],
    "st": [(init_num, local_window_num), ...]}; FLOPs of a candidate are the
    kernel's 4 * d * (admitted causal pairs); recall is the mean of mass_recall
    over `rows` (default: every row).  Returns the chosen pattern, its setting,
    and the per-pattern (setting index, FLOPs, recall) records."""
    N, d = q.shape
    scale = default_scale(d) if scale is None else scale
    rows = np.arange(N) if rows is None else np.asarray(rows)
    order = [p for p in ("vs", "bs", "st") if candidates.get(p)]
    recs = {}
    for p in order:
        masks = [pattern_masks(q, k, p, st, scale) for st in candidates[p]]
        flops = [4 * d * mask_nnz(mk, N) for mk in masks]
        i = choose_setting(flops, budget_flops)
        rec = float(mass_recall(q, k, rows, masks[i], scale).mean())
        recs[p] = {"setting": i, "flops": flops, "recall": rec}
    best = order[choose_pattern([recs[p]["recall"] for p in order])]
    return best, candidates[best][recs[best]["setting"]], recs


# ----------------------------------------------------------------------------- counting
def nnz_from_blocks(sel, N: int) -> int:
    """Number of (i, j) pairs, j <= i, admitted by whole 64-key blocks per row block."""
    total = 0
    for m, blocks in enumerate(sel):
        r0, r1 = m * BLOCK, min(N, (m + 1) * BLOCK)
        for n in blocks:
            k0, k1 = n * BLOCK, min(N, (n + 1) * BLOCK)
            for i in range(r0, r1):
                total += max(0, min(k1, i + 1) - k0)
    return total
