"""Every head type at the longest sequence the library takes, N = 2^21 tokens
(the library refuses anything longer).

One KV head shared by four query heads, with both plantings of the synthetic
recipe: head 0 vertical-slash with 6096 slash lines (sparse tiles: the
one-query-tile kernel), head 1 vertical-slash with 20000 slash lines (dense
tiles: the two-query-tile kernel), head 2 block-sparse top-100, head 3
streaming.  Checked against the oracle as the full-size workload tests do:
line scores and chosen sets (near-tie rule), the tile-distance set and the
column format on sampled row blocks, block selections on the sampled row
blocks, and outputs on seeded sampled rows computed one by one from the GPU's
own index sets.
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
N = 1 << 21
NB = N // 64


def sample_rows(n, seed):
    rng = np.random.default_rng(seed)
    rows = set(rng.choice(N, size=n - 4, replace=False).tolist()) | {0, 63, N - 64, N - 1}
    return sorted(rows)


def test_every_head_type_at_the_maximum_length():
    dev = torch.device("cuda")
    q, k, v = inputs.make_qkv(1, 4, 1, N, 1006, vs_planting=True, bs_planting=True, device=dev)
    out = torch.zeros_like(q)
    vs_cfg = {0: (1000, 6096), 1: (1000, 20000)}
    ex = {}
    for h, (kv, ks) in vs_cfg.items():
        ex[h] = P.vs_export_buffers(1, N, kv, ks, dev)
        msa.msa_vertical_slash(q, k, v, kv, ks, out, heads=[h], export=ex[h])
    exb = {"block_count": torch.empty(1, NB, dtype=torch.int32, device=dev),
           "block_ids": torch.empty(1, NB, 100, dtype=torch.int32, device=dev)}
    msa.msa_block_sparse(q, k, v, 100, out, heads=[2], export=exb)
    msa.msa_streaming(q, k, v, 1, 64, out, heads=[3])
    torch.cuda.synchronize()
    ex = {h: {n: t.cpu().numpy() for n, t in e.items()} for h, e in ex.items()}
    exb = {n: t.cpu().numpy() for n, t in exb.items()}

    scale = 1 / math.sqrt(D)
    rows = sample_rows(12, 1006)
    blocks = sorted({i // 64 for i in rows})
    kn, vn = P.to_np(k[0, 0]), P.to_np(v[0, 0])
    near_ties = 0
    for h in range(4):
        if h in vs_cfg:
            kv, ks = vs_cfg[h]
            e = ex[h]
            q_rows = sorted(set(rows) | set(range(N - 64, N)))
            qn = np.zeros((N, D))
            qn[q_rows] = P.to_np(q[0, h, q_rows])
            vs_, ss_, _ = O.estimate_vs(qn, kn, 64, scale)
            np.testing.assert_allclose(e["v_score"][0], vs_, rtol=1e-4, atol=1e-6 * vs_.max())
            np.testing.assert_allclose(e["s_score"][0], ss_, rtol=1e-4, atol=1e-6 * ss_.max())
            near_ties += P.check_topk(e["vertical"][0], vs_, kv, f"h{h} vertical")
            near_ties += P.check_topk(e["slash"][0], ss_, ks, f"h{h} slash")
            S, V = e["slash"][0].astype(np.int64), e["vertical"][0].astype(np.int64)
            ref_act = O.vs_active_tiles(S, N, blocks)
            words = np.asarray(e["tile_dist"][0], dtype=np.int64) & 0xFFFFFFFF
            for r, m in enumerate(blocks):
                t = m - np.arange(m + 1)
                got = ((words[t >> 5] >> (t & 31)) & 1).astype(bool)
                np.testing.assert_array_equal(got, ref_act[r, :m + 1], err_msg=f"h{h} m{m}")
            col_blocks = sorted({b for m in blocks for b in (m ^ 1, m) if b < NB})
            P.check_vs_columns(e, 0, V, S, N, col_blocks, f"h{h}")
            mask = O.vs_row_block_mask(S, V, N)
        elif h == 2:
            qn = P.to_np(q[0, h])  # pooled queries need every row of q
            _, Sc = O.block_sparse_blocks(qn, kn, 100, scale, row_blocks=blocks)
            sel = {}
            for r, m in enumerate(blocks):
                cnt = int(exb["block_count"][0, m])
                assert cnt == min(100, m + 1)
                got = exb["block_ids"][0, m, :cnt].astype(np.int64)
                assert got[-1] == m
                if m > 0:
                    near_ties += P.check_topk(got[:-1], Sc[r, :m], 99, f"bs m{m}")
                sel[m] = got
            mask = O.block_mask_from_blocks(sel, N)
        else:
            qn = np.zeros((N, D))
            qn[rows] = P.to_np(q[0, h, rows])
            sel = {m: O.streaming_blocks(m, 1, 64) for m in blocks}
            mask = O.block_mask_from_blocks(sel, N)
        ref, counts = O.attend_rows(qn, kn, vn, rows, lambda i: mask(i // 64), scale)
        assert (counts > 0).all()
        P.compare_out(P.to_np(out[0, h, rows]), ref, f"N=2^21 h{h}")
    print(f"N=2^21: {near_ties} near-tie index differences")
