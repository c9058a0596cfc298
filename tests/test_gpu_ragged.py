"""Sequence lengths that are not a multiple of 64 (and shorter than one block)
through the C ABI, against the oracle.

Reading (both sides): index formats treat the last block as a padded 64-token
block; the causal cut removes padded keys; padded rows are never written;
block-sparse pooling averages the real rows of a partial block.
"""
import math

import numpy as np
import pytest
import torch

from oracle import msa_oracle as O
from dynamic_sparse_attention_slash_gb300 import inputs, msa
from tests import parity as P
from tests.test_gpu_kv import check_keep, check_lse, check_score, oracle_kv
from tests.test_gpu_parity import check_vs_case

pytestmark = pytest.mark.gpu
D = 128


def qkv(B, Hq, Hkv, N, seed, vs=True, bs=False):
    q, k, v = inputs.make_qkv(B, Hq, Hkv, N, seed, vs_planting=vs, bs_planting=bs, device="cpu")
    return q.cuda(), k.cuda(), v.cuda()


@pytest.mark.parametrize("N,kv,ks", [(1, 1, 1), (37, 10, 5), (100, 30, 20), (1000, 120, 90),
                                     (1217, 200, 150), (4095, 300, 400)])
def test_vertical_slash_any_length(N, kv, ks):
    q, k, v = qkv(1, 2, 1, N, 41)
    out, _ = check_vs_case(q, k, v, kv, ks)
    # padded rows are not written: a fresh output keeps nothing past N (shape check)
    assert out.shape[2] == N


@pytest.mark.parametrize("N,topk", [(70, 2), (1000, 5), (1217, 8), (33, 1)])
def test_block_sparse_any_length(N, topk):
    q, k, v = qkv(1, 2, 2, N, 42, vs=False, bs=True)
    out, ex = P.run_bs(q, k, v, topk)
    qn, kn, vn = P.to_np(q), P.to_np(k), P.to_np(v)
    NB = (N + 63) // 64
    for h in range(2):
        sel, S = O.block_sparse_blocks(qn[0, h], kn[0, h], topk)
        gpu_sel = []
        for m in range(NB):
            cnt = int(ex["block_count"][h, m])
            assert cnt == min(topk, m + 1)
            got = ex["block_ids"][h, m, :cnt]
            assert got[-1] == m
            if m > 0:
                P.check_topk(got[:-1], S[m, :m], topk - 1, f"h{h} m{m}")
            gpu_sel.append(got.astype(np.int64))
        ref, _ = O.attend_blocks(qn[0, h], kn[0, h], vn[0, h], O.block_mask_from_blocks(gpu_sel, N),
                                 1 / math.sqrt(D))
        P.compare_out(P.to_np(out[0, h]), ref, f"bs N={N} h{h}")


@pytest.mark.parametrize("N,init,local", [(1, 1, 1), (100, 1, 1), (1217, 2, 3), (650, 0, 20)])
def test_streaming_and_dense_any_length(N, init, local):
    q, k, v = qkv(1, 2, 1, N, 43)
    out = msa.msa_streaming(q, k, v, init, local)
    dense = msa.msa_streaming(q, k, v, 0, (N + 63) // 64)
    torch.cuda.synchronize()
    ref, _ = O.streaming_forward(q.cpu(), k.cpu(), v.cpu(), init, local)
    P.compare_out(P.to_np(out[0]), ref[0], f"streaming N={N}")
    qn, kn, vn = P.to_np(q), P.to_np(k), P.to_np(v)
    for h in range(2):
        P.compare_out(P.to_np(dense[0, h]), O.dense_causal(qn[0, h], kn[0, 0], vn[0, 0],
                                                            1 / math.sqrt(D)), f"dense N={N}")


@pytest.mark.parametrize("N,window", [(100, 30), (1217, 256), (37, 37)])
def test_kv_select_any_length(N, window):
    q, k, v = qkv(1, 2, 1, N, 44)
    kv = msa.kv_select_buffers(q, window, 16)
    msa.msa_streaming(q, k, v, 1, 2, kv_select=kv)
    torch.cuda.synchronize()
    NB = (N + 63) // 64
    mask = O.block_mask_from_blocks([O.streaming_blocks(m, 1, 2) for m in range(NB)], N)
    for h in range(2):
        lse, S = oracle_kv(P.to_np(q[0, h]), P.to_np(k[0, 0]), mask, window, np.arange(N))
        check_lse(P.to_np(kv["lse"][0, h]), lse, f"N={N} h{h} lse")
        check_score(P.to_np(kv["score"][0, h]), S, f"N={N} h{h} score")
        check_keep(kv["keep"][0, h].cpu().numpy(), P.to_np(kv["score"][0, h]), S, 16,
                   f"N={N} h{h} keep")
