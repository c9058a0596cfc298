"""Kernel-aware pattern search on the GPU vs the oracle (MInference 1.0
overview, section 2.1 "Kernel-Aware Optimal Sparse Pattern Search").

For every head and every candidate the search's work count (from the GPU's
own index sets) must equal the oracle's pair count of the mask those sets
define, and its recall (mean kept dense-attention mass, from the exported row
normalisers) must match the oracle's recall computed from the dense softmax.
The assignment must be the oracle rules' choice on the oracle's recalls,
unless two candidates' recalls lie within twice the recall tolerance.

Recall tolerance: recall_i = exp(lse_M,i - lse_dense,i) with |d lse| <= 1e-4
for each normaliser, so the per-row relative error is at most e^(2e-4) - 1;
the mean keeps that bound: |d recall| <= 2.1e-4 * recall + 1e-6.
"""
import math

import numpy as np
import pytest
import torch

from oracle import msa_oracle as O
from dynamic_sparse_attention_slash_gb300 import inputs, msa, search

pytestmark = pytest.mark.gpu
D = 128
R_REL, R_ABS = 2.1e-4, 1e-6


def test_search_matches_oracle():
    N, Hq, Hkv = 2048, 4, 2
    q, k, v = inputs.make_qkv(1, Hq, Hkv, N, 31, vs_planting=True, bs_planting=True, device="cpu")
    q, k, v = q.cuda(), k.cuda(), v.cuda()
    cands = {"vs": [(64, 32), (128, 96), (256, 256)], "bs": [2, 4, 8],
             "st": [(1, 2), (1, 4), (1, 8)]}
    budget = 0.25 * 4 * D * N * (N + 1) / 2
    res = search.search(q, k, v, cands, budget)
    scale = 1 / math.sqrt(D)
    NB = (N + 63) // 64
    qn, kn = q[0].double().cpu().numpy(), k[0].double().cpu().numpy()
    # the GPU's index sets per candidate, for the oracle's masks
    for h in range(Hq):
        kh = kn[h // (Hq // Hkv)]
        rec = res["records"][(0, h)]
        oracle_recall = {}
        for p in ("vs", "bs", "st"):
            oracle_recall[p] = []
            for si, st in enumerate(cands[p]):
                if p == "vs":
                    ex = {"vertical": torch.empty(1, min(st[0], N), dtype=torch.int32, device="cuda"),
                          "slash": torch.empty(1, min(st[1], N), dtype=torch.int32, device="cuda")}
                    msa.msa_vertical_slash(q, k, v, st[0], st[1], heads=[h], export=ex)
                    torch.cuda.synchronize()
                    act = O.vs_active_tiles(ex["slash"][0].cpu().numpy(), N)
                    mask = O.vs_block_mask(act, O.vs_columns(ex["vertical"][0].cpu().numpy(),
                                                             act, N), N)
                elif p == "bs":
                    ex = {"block_count": torch.empty(1, NB, dtype=torch.int32, device="cuda"),
                          "block_ids": torch.empty(1, NB, min(st, NB), dtype=torch.int32,
                                                   device="cuda")}
                    msa.msa_block_sparse(q, k, v, st, heads=[h], export=ex)
                    torch.cuda.synchronize()
                    cnt, ids = ex["block_count"][0].cpu().numpy(), ex["block_ids"][0].cpu().numpy()
                    mask = O.block_mask_from_blocks([ids[m, :cnt[m]] for m in range(NB)], N)
                else:
                    mask = O.pattern_masks(qn[h], kh, "st", st, scale)
                assert rec[p]["flops"][si] == 4 * D * O.mask_nnz(mask, N), f"h{h} {p}{st} flops"
                r = float(O.mass_recall(qn[h], kh, np.arange(N), mask, scale).mean())
                got = rec[p]["recall"][si]
                assert abs(got - r) <= R_REL * r + R_ABS, f"h{h} {p}{st}: recall {got} vs {r}"
                oracle_recall[p].append(r)
        # the choice, from the (exact) FLOPs and the oracle's recalls
        best = []
        for p in ("vs", "bs", "st"):
            si = O.choose_setting(rec[p]["flops"], budget)
            assert si == rec[p]["setting"], f"h{h} {p}: setting"
            best.append(oracle_recall[p][si])
        want = ("vs", "bs", "st")[O.choose_pattern(best)]
        got_p, got_s = res["assignment"][(0, h)]
        if got_p != want:
            gap = abs(best[("vs", "bs", "st").index(got_p)] - max(best))
            assert gap <= 2 * (R_REL * max(best) + R_ABS), f"h{h}: chose {got_p}, oracle {want}"
        assert got_s == cands[got_p][rec[got_p]["setting"]]


def test_mass_recall_dense_is_one_and_subset_heads():
    N = 1024
    q, k, v = inputs.make_qkv(2, 4, 2, N, 32, vs_planting=True, device="cpu")
    q, k, v = q.cuda(), k.cuda(), v.cuda()
    ref = {"lse": torch.zeros(2, 4, N, device="cuda"), "window": 0, "keep_k": 0}
    msa.msa_streaming(q, k, v, 0, (N + 63) // 64, kv_select=ref)
    recall = torch.full((2, 4), 9.0, device="cuda")
    msa.mass_recall(ref["lse"], ref["lse"], recall, heads=[2, 0])
    torch.cuda.synchronize()
    r = recall.cpu()
    assert torch.allclose(r[:, [0, 2]], torch.ones(2, 2), atol=1e-6)
    assert bool((r[:, [1, 3]] == 9.0).all())
    # rows [row0, N) only
    cur = {"lse": torch.zeros(2, 4, N, device="cuda"), "window": 0, "keep_k": 0}
    msa.msa_streaming(q, k, v, 0, 2, kv_select=cur)
    msa.mass_recall(cur["lse"], ref["lse"], recall, row0=N - 64)
    torch.cuda.synchronize()
    qn, kn = q.double().cpu().numpy(), k.double().cpu().numpy()
    mask = O.block_mask_from_blocks([O.streaming_blocks(m, 0, 2) for m in range((N + 63) // 64)], N)
    for b in range(2):
        for h in range(4):
            ref_r = O.mass_recall(qn[b, h], kn[b, h // 2], np.arange(N - 64, N), mask,
                                  1 / math.sqrt(D)).mean()
            assert abs(float(recall[b, h]) - ref_r) <= R_REL * ref_r + R_ABS


def test_apply_assignment_matches_individual_calls():
    """The searched per-head patterns applied in one call give exactly the
    outputs of the three entry points called on their head groups."""
    N = 1024
    q, k, v = inputs.make_qkv(1, 4, 2, N, 33, vs_planting=True, bs_planting=True, device="cpu")
    q, k, v = q.cuda(), k.cuda(), v.cuda()
    a = {(0, 0): ("vs", (64, 96)), (0, 1): ("bs", 4), (0, 2): ("st", (1, 4)),
         (0, 3): ("vs", (64, 96))}
    out = search.apply_assignment(q, k, v, a)
    ref = torch.empty_like(q)
    msa.msa_vertical_slash(q, k, v, 64, 96, ref, heads=[0, 3])
    msa.msa_block_sparse(q, k, v, 4, ref, heads=[1])
    msa.msa_streaming(q, k, v, 1, 4, ref, heads=[2])
    torch.cuda.synchronize()
    assert torch.equal(out, ref)
    # and straight from a search result
    res = search.search(q, k, v, {"vs": [(64, 32)], "bs": [2, 4], "st": [(1, 2)]},
                        0.25 * 4 * D * N * (N + 1) / 2)
    out2 = search.apply_assignment(q, k, v, res["assignment"])
    torch.cuda.synchronize()
    assert torch.isfinite(out2.float()).all()
