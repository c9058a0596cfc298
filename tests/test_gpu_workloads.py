"""The named workloads at full size, called exactly as the benchmark calls them
(one call per head type on its head subset of shared q/k/v/out tensors).

Checked against the oracle: index data for every head (line scores, chosen
sets with the near-tie rule, the tile-distance set on sampled row blocks,
block selections for every row block), and outputs on seeded sampled query
rows computed one by one by the oracle from the GPU's own index sets.
"""
import math

import numpy as np
import pytest
import torch

from oracle import msa_oracle as O
from dynamic_sparse_attention_slash_gb300 import inputs, msa
from tests import parity as P

pytestmark = pytest.mark.gpu
D = 128


def run_step(w, q, k, v, heads):
    """One benchmark step with index export; returns (out, exports)."""
    B, N = w.batch, w.seq_len
    out = torch.zeros_like(q)
    ex = {}
    if heads["vs"]:
        U = B * len(heads["vs"])
        ex["vs"] = P.vs_export_buffers(U, N, min(w.vertical_topk, N), min(w.slash, N), q.device)
        msa.msa_vertical_slash(q, k, v, w.vertical_topk, w.slash, out, last_q=w.last_q,
                               heads=heads["vs"], export=ex["vs"])
    if heads["bs"]:
        U = B * len(heads["bs"])
        NB = (N + 63) // 64
        ex["bs"] = {"block_count": torch.empty(U, NB, dtype=torch.int32, device=q.device),
                    "block_ids": torch.empty(U, NB, min(w.block_topk, NB), dtype=torch.int32,
                                             device=q.device)}
        msa.msa_block_sparse(q, k, v, w.block_topk, out, heads=heads["bs"], export=ex["bs"])
    if heads["st"]:
        msa.msa_streaming(q, k, v, w.init_num, w.local_window_num, out, heads=heads["st"])
    if heads["hip"]:
        U = B * len(heads["hip"])
        NB = (N + 63) // 64
        kb = min(w.hip_stages[-1][1], NB)
        ex["hip"] = {"block_count": torch.empty(U, NB, dtype=torch.int32, device=q.device),
                     "block_ids": torch.empty(U, NB, kb, dtype=torch.int32, device=q.device)}
        msa.msa_hierarchical(q, k, v, w.hip_stages, out, heads=heads["hip"], export=ex["hip"])
    torch.cuda.synchronize()
    return out, {kind: {n: t.cpu().numpy() for n, t in d.items()} for kind, d in ex.items()}


def sample_rows(N, n, seed):
    rng = np.random.default_rng(seed)
    rows = set(rng.choice(N, size=n - 4, replace=False).tolist()) | {0, 63, N - 64, N - 1}
    return sorted(rows)


ROWS = {"vs_32k": 48, "bs_64k": 48, "mixed_128k": 32, "vs_1m": 16, "hip_64k": 32}


@pytest.mark.parametrize("name", ["vs_32k", "bs_64k", "mixed_128k", "vs_1m", "hip_64k"])
def test_workload_full_size(name):
    w, q, k, v, heads = inputs.make_workload(name, device="cuda")
    out, ex = run_step(w, q, k, v, heads)
    N, G = w.seq_len, w.n_q_heads // w.n_kv_heads
    scale = 1 / math.sqrt(D)
    rows = sample_rows(N, ROWS[name], w.seed)
    kind_of = {h: kind for kind in ("vs", "bs", "st", "hip") for h in heads[kind]}
    near_ties = 0
    for g in range(w.n_kv_heads):
        kn, vn = P.to_np(k[0, g]), P.to_np(v[0, g])
        for h in range(g * G, (g + 1) * G):
            kind = kind_of[h]
            q_rows = sorted(set(rows) | set(range(N - w.last_q, N)))
            qsel = P.to_np(q[0, h, q_rows])
            qn = np.zeros((N, D))
            qn[q_rows] = qsel
            if kind == "vs":
                u = heads["vs"].index(h)
                e = ex["vs"]
                vs_, ss_, _ = O.estimate_vs(qn, kn, w.last_q, scale)
                np.testing.assert_allclose(e["v_score"][u], vs_, rtol=1e-4, atol=1e-6 * vs_.max())
                np.testing.assert_allclose(e["s_score"][u], ss_, rtol=1e-4, atol=1e-6 * ss_.max())
                near_ties += P.check_topk(e["vertical"][u], vs_, w.vertical_topk, f"{name} h{h} vertical")
                near_ties += P.check_topk(e["slash"][u], ss_, w.slash, f"{name} h{h} slash")
                S, V = e["slash"][u].astype(np.int64), e["vertical"][u].astype(np.int64)
                blocks = sorted({i // 64 for i in rows})
                bits = P.dist_bits_to_active(e["tile_dist"][u], (N + 63) // 64) if N <= 131072 else None
                ref_act = O.vs_active_tiles(S, N, blocks)
                words = np.asarray(e["tile_dist"][u], dtype=np.int64) & 0xFFFFFFFF
                for r, m in enumerate(blocks):
                    t = m - np.arange(m + 1)
                    got = ((words[t >> 5] >> (t & 31)) & 1).astype(bool)
                    np.testing.assert_array_equal(got, ref_act[r, :m + 1], err_msg=f"h{h} m{m}")
                    if bits is not None:
                        np.testing.assert_array_equal(bits[m], ref_act[r])
                # the column part of the format, exactly, on the sampled row
                # blocks and their query tiles' partner blocks
                col_blocks = sorted({b_ for m in blocks for b_ in (m ^ 1, m) if b_ < (N + 63) // 64})
                P.check_vs_columns(e, u, V, S, N, col_blocks, f"{name} h{h}")
                mask = O.vs_row_block_mask(S, V, N)
            elif kind == "bs":
                u = heads["bs"].index(h)
                e = ex["bs"]
                # pooled scores need every row of q for this head
                qn = P.to_np(q[0, h])
                sel_ref, Sc = O.block_sparse_blocks(qn, kn, w.block_topk, scale)
                sel = []
                for m in range((N + 63) // 64):
                    cnt = int(e["block_count"][u, m])
                    assert cnt == min(w.block_topk, m + 1)
                    got = e["block_ids"][u, m, :cnt].astype(np.int64)
                    assert got[-1] == m
                    if m > 0:
                        near_ties += P.check_topk(got[:-1], Sc[m, :m], w.block_topk - 1,
                                                  f"{name} h{h} m{m}")
                    sel.append(got)
                mask = O.block_mask_from_blocks(sel, N)
            elif kind == "hip":
                u = heads["hip"].index(h)
                e = ex["hip"]
                qn = P.to_np(q[0, h])  # pooled queries need every row of q
                blocks = sorted({i // 64 for i in rows} | {0, (N + 63) // 64 - 1})
                sel, nt = P.check_hip_blocks(e["block_count"][u], e["block_ids"][u], qn, kn,
                                             w.hip_stages, blocks, f"{name} h{h}")
                near_ties += nt
                keys = lambda i, sel=sel: np.concatenate([np.arange(64 * n, min(N, 64 * n + 64))
                                                          for n in sel[i // 64]])
                mask = lambda m, keys=keys: np.isin(np.arange(N), keys(64 * m))
            else:
                sel = [O.streaming_blocks(m, w.init_num, w.local_window_num) for m in range((N + 63) // 64)]
                mask = O.block_mask_from_blocks(sel, N)
            ref, counts = O.attend_rows(qn, kn, vn, rows, lambda i: mask(i // 64), scale)
            assert (counts > 0).all(), "no sampled row may be empty under the planted inputs"
            got = P.to_np(out[0, h, rows])
            P.compare_out(got, ref, f"{name} {kind} h{h}")
    print(f"{name}: {near_ties} near-tie index differences")
