"""The hierarchical multi-stage pruning head on the GPU against the fp64
oracle (InfiniteHiP summary page, section on the modular hierarchical token
pruning algorithm), through the C ABI.

Kept blocks are compared exactly per row block (the near-tie rule applied at
every stage's cut, see tests/parity.py), outputs element-wise against the
oracle's attention over the GPU's own blocks.  Sizes span several 128-row
query tiles and a ragged tail; one case holds more block maxima than one slab,
so the index runs in two slabs of query blocks.
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
SCALE = 1 / math.sqrt(D)


def qkv(B, Hq, Hkv, N, seed):
    q, k, v = inputs.make_qkv(B, Hq, Hkv, N, seed, vs_planting=False, bs_planting=True, device="cpu")
    return q.cuda(), k.cuda(), v.cuda()


@pytest.mark.parametrize("N,stages", [
    (2048, [(4, 3), (1, 4)]),
    (2112, [(8, 2), (2, 3), (1, 5)]),
    (2048, [(1, 6)]),
    (640, [(16, 2), (4, 2), (1, 3)]),
    (4160, [(8, 4), (2, 6), (1, 7)]),
])
def test_hierarchical_matches_oracle(N, stages):
    q, k, v = qkv(1, 4, 2, N, 31)
    out, ex = P.run_hip(q, k, v, stages)
    qn, kn, vn = P.to_np(q), P.to_np(k), P.to_np(v)
    NB = (N + 63) // 64
    near = 0
    for h in range(4):
        g = h // 2
        sel, nt = P.check_hip_blocks(ex["block_count"][h], ex["block_ids"][h], qn[0, h], kn[0, g],
                                     stages, list(range(NB)), f"hip h{h}")
        near += nt
        ref, _ = O.attend_blocks(qn[0, h], kn[0, g], vn[0, g],
                                 O.block_mask_from_blocks([sel[m] for m in range(NB)], N), SCALE)
        P.compare_out(P.to_np(out[0, h]), ref, f"hip h{h}")
    assert near <= 2, f"{near} near-tie row blocks"


def test_hierarchical_keep_all_is_dense_causal():
    N = 1536
    q, k, v = qkv(1, 2, 1, N, 32)
    NB = N // 64
    out, ex = P.run_hip(q, k, v, [(4, NB), (1, NB)])
    qn, kn, vn = P.to_np(q), P.to_np(k), P.to_np(v)
    for h in range(2):
        for m in range(NB):
            np.testing.assert_array_equal(ex["block_ids"][h, m, :ex["block_count"][h, m]],
                                          np.arange(m + 1))
        P.compare_out(P.to_np(out[0, h]), O.dense_causal(qn[0, h], kn[0, 0], vn[0, 0], SCALE),
                      f"dense h{h}")


def test_hierarchical_zero_keys_take_the_lowest_chunks():
    """K = 0: every token score is exactly 0 on both sides, every stage's
    chunk scores tie, and the kept sets are the closed form (own chunk plus
    the lowest other chunks), with no near-tie allowance."""
    N, stages = 1024, [(4, 2), (1, 3)]
    g = torch.Generator().manual_seed(9)
    q = torch.randn(1, 1, N, D, generator=g).to(torch.bfloat16).cuda()
    k = torch.zeros(1, 1, N, D, dtype=torch.bfloat16).cuda()
    v = torch.randn(1, 1, N, D, generator=g).to(torch.bfloat16).cuda()
    out, ex = P.run_hip(q, k, v, stages)
    sel, _ = O.hierarchical_blocks(P.to_np(q)[0, 0], P.to_np(k)[0, 0], stages)
    for m in range(N // 64):
        np.testing.assert_array_equal(ex["block_ids"][0, m, :ex["block_count"][0, m]], sel[m])
    assert sel[10].tolist() == [0, 1, 10]
    ref, _ = O.attend_blocks(P.to_np(q)[0, 0], P.to_np(k)[0, 0], P.to_np(v)[0, 0],
                             O.block_mask_from_blocks(sel, N), SCALE)
    P.compare_out(P.to_np(out[0, 0]), ref, "hip zero keys")


def test_hierarchical_batch_head_subset_and_normalisers():
    """A batch of two, a head subset and a ragged length; the row normalisers
    (lse) the KV selection exports, against the oracle's over the GPU's blocks."""
    N, stages, heads = 1088, [(4, 3), (1, 4)], [3, 0]
    q, k, v = qkv(2, 4, 2, N, 33)
    NB = (N + 63) // 64
    U = 2 * len(heads)
    ex = {"block_count": torch.empty(U, NB, dtype=torch.int32, device="cuda"),
          "block_ids": torch.empty(U, NB, 4, dtype=torch.int32, device="cuda")}
    kvb = msa.kv_select_buffers(q, 64, 16)
    out = torch.full_like(q, 7.0)
    msa.msa_hierarchical(q, k, v, stages, out, heads=heads, export=ex, kv_select=kvb)
    torch.cuda.synchronize()
    qn, kn, vn = P.to_np(q), P.to_np(k), P.to_np(v)
    counts, ids = ex["block_count"].cpu().numpy(), ex["block_ids"].cpu().numpy()
    for b in range(2):
        for t, h in enumerate(heads):
            u, g = b * len(heads) + t, h // 2
            sel, _ = P.check_hip_blocks(counts[u], ids[u], qn[b, h], kn[b, g], stages,
                                        list(range(NB)), f"hip b{b} h{h}")
            mask = O.block_mask_from_blocks([sel[m] for m in range(NB)], N)
            ref, _ = O.attend_blocks(qn[b, h], kn[b, g], vn[b, g], mask, SCALE)
            P.compare_out(P.to_np(out[b, h]), ref, f"hip b{b} h{h}")
            lse_ref = O.row_lse(qn[b, h], kn[b, g], np.arange(N), mask, SCALE)
            lse = kvb["lse"][b, h].double().cpu().numpy()
            assert np.abs(lse - lse_ref).max() <= 1e-4
        for h in (1, 2):
            assert (out[b, h] == 7.0).all(), f"head {h} outside the subset was written"


def test_hierarchical_two_slabs():
    """12 heads at N = 262144: the block maxima of all 4096 query blocks would
    exceed one slab, so the index runs slab by slab (the second slab starts at
    query block 2688).  Kept blocks on sampled row blocks around the slab
    boundary and at both ends, outputs on sampled rows."""
    N, stages = 262144, [(16, 8), (4, 12), (1, 40)]
    q, k, v = qkv(1, 12, 4, N, 34)
    out, ex = P.run_hip(q, k, v, stages)
    NB = N // 64
    blocks = [0, 1, 63, 1000, 2687, 2688, 2689, 3000, NB - 2, NB - 1]
    rng = np.random.default_rng(34)
    rows = sorted(set(rng.integers(0, N, 24).tolist()) | {0, 64 * 2688, N - 1})
    near = 0
    for h in (0, 5, 11):
        g = h // 3
        qn, kn, vn = P.to_np(q[0, h]), P.to_np(k[0, g]), P.to_np(v[0, g])
        sel, nt = P.check_hip_blocks(ex["block_count"][h], ex["block_ids"][h], qn, kn, stages,
                                     sorted(set(blocks) | {i // 64 for i in rows}), f"slab h{h}")
        near += nt
        keys = lambda i: np.concatenate([np.arange(64 * n, 64 * n + 64) for n in sel[i // 64]])
        ref, _ = O.attend_rows(qn, kn, vn, rows, keys, SCALE)
        P.compare_out(P.to_np(out[0, h, rows]), ref, f"slab h{h}")
    assert near <= 2, f"{near} near-tie row blocks"


def test_hierarchical_long_single_stage_cta_selection():
    """One stage of single blocks over 2048 query blocks: the candidate lists
    would not fit eight warps' shared memory, so the selection runs one CTA
    per query block (the other path); kept blocks on sampled query blocks and
    outputs on sampled rows against the oracle."""
    N, stages = 131072, [(1, 20)]
    q, k, v = qkv(1, 2, 1, N, 35)
    out, ex = P.run_hip(q, k, v, stages)
    NB = N // 64
    rng = np.random.default_rng(35)
    rows = sorted(set(rng.integers(0, N, 16).tolist()) | {0, N - 1})
    blocks = sorted({0, 1, 19, 20, NB - 1} | {i // 64 for i in rows})
    near = 0
    for h in range(2):
        qn, kn, vn = P.to_np(q[0, h]), P.to_np(k[0, 0]), P.to_np(v[0, 0])
        sel, nt = P.check_hip_blocks(ex["block_count"][h], ex["block_ids"][h], qn, kn, stages,
                                     blocks, f"single-stage h{h}")
        near += nt
        keys = lambda i: np.concatenate([np.arange(64 * n, 64 * n + 64) for n in sel[i // 64]])
        ref, _ = O.attend_rows(qn, kn, vn, rows, keys, SCALE)
        P.compare_out(P.to_np(out[0, h, rows]), ref, f"single-stage h{h}")
    assert near <= 1, f"{near} near-tie row blocks"
