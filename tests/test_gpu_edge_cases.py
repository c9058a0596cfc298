"""Degenerate cases of the method on the GPU, against the oracle, with exact
integer results and no near-tie allowance.

* Exact ties in the top-k (score descending, ties to the lower index; the
  MInference 1.0 overview, section 2.2, keeps "top-k" lines and blocks, and the
  tie rule is this library's stated reading).  With K = 0 every logit is 0, so
  every vertical score of a key before the estimate window, and every slash
  score of an offset every window row reaches, is the same sum of the same 64
  probabilities 1/(i+1), added in the same order: bit-identical on both sides.
  With every key row equal, every pooled key block is that row, so all
  block-sparse scores of a row block are bit-identical.  The chosen sets must
  then be exactly the lowest indices.
* Rows whose mask admits no key (the page's A(M) formula, section 1, leaves
  them undefined; this library writes zeros and lse = -inf).  The inputs make
  the estimate pick only very long diagonals and one late column, so the
  first 14 row blocks of 16 have no active tile and no column.
"""
import math

import numpy as np
import pytest
import torch

from oracle import msa_oracle as O
from dynamic_sparse_attention_slash_gb300 import msa
from tests import parity as P

pytestmark = pytest.mark.gpu
D = 128
SCALE = 1 / math.sqrt(D)


def test_vertical_slash_exact_ties_take_the_lowest_indices():
    N, kv, ks = 2048, 100, 150
    g = torch.Generator().manual_seed(7)
    q = torch.randn(1, 2, N, D, generator=g).to(torch.bfloat16).cuda()
    k = torch.zeros(1, 1, N, D, dtype=torch.bfloat16).cuda()
    v = torch.randn(1, 1, N, D, generator=g).to(torch.bfloat16).cuda()
    out, ex = P.run_vs(q, k, v, kv, ks)
    qn, kn, vn = P.to_np(q), P.to_np(k), P.to_np(v)
    for h in range(2):
        vs_, ss_, _ = O.estimate_vs(qn[0, h], kn[0, 0], 64, SCALE)
        # the tie is exact on both sides: every pre-window column, every
        # full-length diagonal
        assert np.unique(vs_[:N - 63]).size == 1 and np.unique(ss_[:N - 63]).size == 1
        assert np.unique(ex["v_score"][h, :N - 63]).size == 1
        assert np.unique(ex["s_score"][h, :N - 63]).size == 1
        V_ref, S_ref = O.topk_indices(vs_, kv), O.topk_indices(ss_, ks)
        np.testing.assert_array_equal(V_ref, np.arange(kv))
        np.testing.assert_array_equal(S_ref, np.arange(ks))
        np.testing.assert_array_equal(ex["vertical"][h], V_ref)
        np.testing.assert_array_equal(ex["slash"][h], S_ref)
        act = O.vs_active_tiles(S_ref, N)
        np.testing.assert_array_equal(P.dist_bits_to_active(ex["tile_dist"][h], N // 64), act)
        ref, _ = O.attend_blocks(qn[0, h], kn[0, 0], vn[0, 0],
                                 O.vs_block_mask(act, O.vs_columns(V_ref, act, N), N), SCALE)
        P.compare_out(P.to_np(out[0, h]), ref, f"vs ties h{h}")


def test_block_sparse_exact_ties_take_the_lowest_blocks():
    N, topk = 2048, 6
    g = torch.Generator().manual_seed(8)
    q = torch.randn(1, 2, N, D, generator=g)
    q += torch.randn(1, 2, N // 64, D, generator=g).repeat_interleave(64, dim=2)
    k = torch.randn(1, 1, 1, D, generator=g).expand(1, 1, N, D).contiguous()
    v = torch.randn(1, 1, N, D, generator=g)
    q, k, v = (t.to(torch.bfloat16).cuda() for t in (q, k, v))
    out, ex = P.run_bs(q, k, v, topk)
    qn, kn, vn = P.to_np(q), P.to_np(k), P.to_np(v)
    NB = N // 64
    for h in range(2):
        sel_ref, S = O.block_sparse_blocks(qn[0, h], kn[0, 0], topk, SCALE)
        for m in range(NB):
            assert np.unique(S[m, :m + 1]).size == 1, "pooled scores of a row block must tie"
            want = np.concatenate([np.arange(min(topk - 1, m)), [m]])
            np.testing.assert_array_equal(sel_ref[m], want)
            cnt = int(ex["block_count"][h, m])
            assert cnt == want.size
            np.testing.assert_array_equal(ex["block_ids"][h, m, :cnt], want, err_msg=f"h{h} m{m}")
        ref, _ = O.attend_blocks(qn[0, h], kn[0, 0], vn[0, 0], O.block_mask_from_blocks(sel_ref, N),
                                 SCALE)
        P.compare_out(P.to_np(out[0, h]), ref, f"bs ties h{h}")


def empty_row_inputs(N):
    """Every query is 8 e_0.  Keys 0..63 get 5.657 e_0 (weight about e^4 each
    for every window row) and key N - 128 gets 8.6 e_0 (about 8 times a band
    key's weight); all other keys are 0.  The single chosen column is then key
    N - 128, and the 16 chosen diagonals are those through the early band, at
    offsets near N - 64: their tiles lie at distances >= N/64 - 2."""
    q = torch.zeros(1, 1, N, D)
    k = torch.zeros(1, 1, N, D)
    q[..., 0] = 8.0
    k[0, 0, :64, 0] = 5.657
    k[0, 0, N - 128, 0] = 8.6
    v = torch.randn(1, 1, N, D, generator=torch.Generator().manual_seed(5))
    return [t.to(torch.bfloat16).cuda() for t in (q, k, v)]


def test_vertical_slash_empty_rows_are_zero_with_lse_minus_inf():
    N, kv, ks = 1024, 1, 16
    q, k, v = empty_row_inputs(N)
    U, NB = 1, N // 64
    ex = {"vertical": torch.empty(U, kv, dtype=torch.int32, device="cuda"),
          "slash": torch.empty(U, ks, dtype=torch.int32, device="cuda"),
          "tile_dist": torch.empty(U, (NB + 32) // 32, dtype=torch.int32, device="cuda")}
    kvb = msa.kv_select_buffers(q, 64, 8)
    out = torch.full_like(q, 3.0)
    msa.msa_vertical_slash(q, k, v, kv, ks, out, export=ex, kv_select=kvb)
    torch.cuda.synchronize()
    qn, kn, vn = P.to_np(q)[0, 0], P.to_np(k)[0, 0], P.to_np(v)[0, 0]
    ref, idx = O.vertical_slash_head(qn, kn, vn, kv, ks, scale=SCALE)
    vs_, ss_, _ = O.estimate_vs(qn, kn, 64, SCALE)
    P.check_topk(ex["vertical"][0].cpu().numpy(), vs_, kv, "empty-row vertical")
    P.check_topk(ex["slash"][0].cpu().numpy(), ss_, ks, "empty-row slash")
    np.testing.assert_array_equal(ex["vertical"][0].cpu().numpy(), idx["vertical"])
    np.testing.assert_array_equal(ex["slash"][0].cpu().numpy(), idx["slash"])
    empty = [m for m in range(NB) if not idx["active"][m].any() and idx["columns"][m].size == 0]
    assert empty == list(range(14)), f"the inputs must leave row blocks 0..13 empty, got {empty}"
    rows = np.arange(64 * len(empty))
    # the oracle's rule (c2) on its side
    assert (ref[rows] == 0).all()
    lse_ref = O.row_lse(qn, kn, np.arange(N),
                        O.vs_block_mask(idx["active"], idx["columns"], N), SCALE)
    assert np.isneginf(lse_ref[rows]).all() and np.isfinite(lse_ref[64 * 14:]).all()
    # and on the GPU's: zeros written over the 3.0 fill, lse = -inf
    got = P.to_np(out[0, 0])
    assert (got[rows] == 0).all(), "an empty row must be written as zeros"
    lse = kvb["lse"][0, 0].double().cpu().numpy()
    assert np.isneginf(lse[rows]).all()
    assert np.abs(lse[64 * 14:] - lse_ref[64 * 14:]).max() <= 1e-4
    P.compare_out(got, ref, "empty-row head")
