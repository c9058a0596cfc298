"""KV selection on the GPU vs the oracle ("How KV sparsity achieves 1.5x
acceleration for vLLM", Novita AI blog, section "2. Attention modification").

The CUDA path exports every row's normaliser lse_i from the attention kernel,
computes the window score S_j in a key-major second pass and keeps the top
keys per head.  The oracle recomputes lse and S in fp64 from the GPU's own
index sets (the same key sets J_i the GPU attended), so a near-tie in an
upstream top-k cannot move the comparison.

Tolerances (derived from the arithmetic, not fitted):
* lse: the kernel's row sum l is an f32 chain of at most (items + 32) terms,
  relative error <= ~1100 * 2^-24 < 7e-5 at 128K; the max and the logits are
  f32 as well (bf16 products, f32 sums).  |d lse| <= 1e-4.
* S: every term inherits that error plus the ex2 approximation (~2^-22) and
  terms are summed in f32 over at most 64 rows per block:
  |d S| <= 2e-4 * S + 1e-12.
* keep: exactly the top-k (ties to the lower index) of the GPU's own scores;
  against the oracle it may differ only by keys whose oracle scores lie within
  4e-4 (relative, twice the score tolerance) of the oracle's k-th score.
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
LSE_TOL = 1e-4
S_REL, S_ABS = 2e-4, 1e-12
TIE_REL = 4e-4


def qkv(B, Hq, Hkv, N, seed, vs=True, bs=False):
    q, k, v = inputs.make_qkv(B, Hq, Hkv, N, seed, vs_planting=vs, bs_planting=bs, device="cpu")
    return q.cuda(), k.cuda(), v.cuda()


def check_lse(got, ref, what):
    got, ref = np.asarray(got, np.float64), np.asarray(ref, np.float64)
    assert np.array_equal(np.isneginf(got), np.isneginf(ref)), f"{what}: empty rows differ"
    fin = np.isfinite(ref)
    err = np.abs(got[fin] - ref[fin])
    assert err.size == 0 or err.max() <= LSE_TOL, f"{what}: lse max err {err.max():.3e}"


def check_score(got, ref, what):
    got, ref = np.asarray(got, np.float64), np.asarray(ref, np.float64)
    err = np.abs(got - ref)
    bound = S_REL * np.abs(ref) + S_ABS
    bad = np.nonzero(err > bound)[0]
    assert bad.size == 0, (f"{what}: {bad.size} scores out of tolerance, worst at key {bad[0]}: "
                           f"{got[bad[0]]!r} vs {ref[bad[0]]!r}")


def check_keep(keep, gpu_score, ref_score, k, what):
    keep = np.asarray(keep, np.int64)
    assert np.all(np.diff(keep) > 0), f"{what}: keep set not strictly ascending"
    # exactly the top-k of the GPU's own scores
    assert np.array_equal(keep, O.topk_indices(np.asarray(gpu_score, np.float64), k)), \
        f"{what}: keep set is not the top-k of the returned scores"
    ref = O.topk_indices(ref_score, k)
    if np.array_equal(keep, ref):
        return
    kth = np.sort(ref_score)[::-1][min(k, ref_score.size) - 1]
    diff = np.setxor1d(keep, ref)
    bad = diff[np.abs(ref_score[diff] - kth) > TIE_REL * abs(kth)]
    assert bad.size == 0, f"{what}: {bad.size} keep differences are not near-ties"


def vs_mask_from_export(e, u, N):
    active = O.vs_active_tiles(e["slash"][u], N)
    cols = O.vs_columns(e["vertical"][u], active, N)
    return O.vs_block_mask(active, cols, N)


def oracle_kv(qn, kn, mask, window, lse_rows):
    scale = 1 / math.sqrt(D)
    N = qn.shape[0]
    lse = O.row_lse(qn, kn, lse_rows, mask, scale)
    win = np.arange(N - window, N)
    S = O.kv_score(qn, kn, O.row_lse(qn, kn, win, mask, scale), mask, window, scale)
    return lse, S


# slash 16 at N = 4160: 128 * 16 < N, the one-query-tile kernel writes the lse
@pytest.mark.parametrize("N,window,keep_k,slash", [(2048, 64, 256, 300), (1088, 100, 64, 300),
                                                   (1024, 1, 16, 300), (4160, 64, 256, 16)])
def test_vertical_slash_kv_select(N, window, keep_k, slash):
    q, k, v = qkv(1, 2, 1, N, 21)
    kv = msa.kv_select_buffers(q, window, keep_k)
    _, ex = run_vs_kv(q, k, v, 200, slash, kv)
    qn, kn = P.to_np(q[0]), P.to_np(k[0, 0])
    for h in range(2):
        mask = vs_mask_from_export(ex, h, N)
        lse, S = oracle_kv(qn[h], kn, mask, window, np.arange(N))
        check_lse(P.to_np(kv["lse"][0, h]), lse, f"vs h{h} lse")
        check_score(P.to_np(kv["score"][0, h]), S, f"vs h{h} score")
        check_keep(kv["keep"][0, h].cpu().numpy(), P.to_np(kv["score"][0, h]), S, keep_k,
                   f"vs h{h} keep")
        assert abs(float(kv["score"][0, h].double().sum()) - window) < 1e-3


def run_vs_kv(q, k, v, vertical_topk, slash, kv, heads=None):
    B, Hq, N, _ = q.shape
    U = B * (Hq if heads is None else len(heads))
    dev = q.device
    ex = {"vertical": torch.empty(U, min(vertical_topk, N), dtype=torch.int32, device=dev),
          "slash": torch.empty(U, min(slash, N), dtype=torch.int32, device=dev)}
    out = msa.msa_vertical_slash(q, k, v, vertical_topk, slash, heads=heads, export=ex,
                                 kv_select=kv)
    torch.cuda.synchronize()
    return out, {n: t.cpu().numpy() for n, t in ex.items()}


@pytest.mark.parametrize("N,topk,window", [(2048, 8, 64), (1536, 3, 200)])
def test_block_sparse_kv_select(N, topk, window):
    q, k, v = qkv(1, 2, 2, N, 22, vs=False, bs=True)
    kv = msa.kv_select_buffers(q, window, 128)
    NB = (N + 63) // 64
    ex = {"block_count": torch.empty(2, NB, dtype=torch.int32, device=q.device),
          "block_ids": torch.empty(2, NB, min(topk, NB), dtype=torch.int32, device=q.device)}
    msa.msa_block_sparse(q, k, v, topk, export=ex, kv_select=kv)
    torch.cuda.synchronize()
    cnt, ids = ex["block_count"].cpu().numpy(), ex["block_ids"].cpu().numpy()
    for h in range(2):
        sel = [ids[h, m, :cnt[h, m]] for m in range(NB)]
        mask = O.block_mask_from_blocks(sel, N)
        lse, S = oracle_kv(P.to_np(q[0, h]), P.to_np(k[0, h]), mask, window, np.arange(N))
        check_lse(P.to_np(kv["lse"][0, h]), lse, f"bs h{h} lse")
        check_score(P.to_np(kv["score"][0, h]), S, f"bs h{h} score")
        check_keep(kv["keep"][0, h].cpu().numpy(), P.to_np(kv["score"][0, h]), S, 128,
                   f"bs h{h} keep")


@pytest.mark.parametrize("N,init,local,window", [(1536, 1, 3, 64), (960, 0, 2, 130),
                                                 (512, 2, 8, 512)])
def test_streaming_kv_select(N, init, local, window):
    q, k, v = qkv(1, 2, 1, N, 23)
    kv = msa.kv_select_buffers(q, window, 40)
    msa.msa_streaming(q, k, v, init, local, kv_select=kv)
    torch.cuda.synchronize()
    NB = (N + 63) // 64
    sel = [O.streaming_blocks(m, init, local) for m in range(NB)]
    mask = O.block_mask_from_blocks(sel, N)
    for h in range(2):
        lse, S = oracle_kv(P.to_np(q[0, h]), P.to_np(k[0, 0]), mask, window, np.arange(N))
        check_lse(P.to_np(kv["lse"][0, h]), lse, f"st h{h} lse")
        check_score(P.to_np(kv["score"][0, h]), S, f"st h{h} score")
        check_keep(kv["keep"][0, h].cpu().numpy(), P.to_np(kv["score"][0, h]), S, 40,
                   f"st h{h} keep")


def test_dense_window_score_matches_gpu_vertical_estimate():
    """Dense head, window = last_q: the KV score is the column sum of the causal
    softmax of the last 64 rows, which is also the vertical-slash estimate's
    vertical score, computed by a different GPU kernel."""
    N = 4096
    q, k, v = qkv(1, 1, 1, N, 24)
    kv = msa.kv_select_buffers(q, 64, 0)
    msa.msa_streaming(q, k, v, 0, (N + 63) // 64, kv_select=kv)
    v_score = torch.empty(1, N, dtype=torch.float32, device=q.device)
    msa.msa_vertical_slash(q, k, v, 100, 100, export={"v_score": v_score})
    torch.cuda.synchronize()
    check_score(P.to_np(kv["score"][0, 0]), P.to_np(v_score[0]), "dense score vs estimate")


def test_head_subset_leaves_other_heads_untouched():
    N = 1024
    q, k, v = qkv(2, 4, 2, N, 25)
    kv = msa.kv_select_buffers(q, 64, 32)
    for name in ("lse", "score"):
        kv[name].fill_(123.0)
    kv["keep"].fill_(-5)
    msa.msa_streaming(q, k, v, 1, 4, heads=[3, 0], kv_select=kv)
    torch.cuda.synchronize()
    for b in range(2):
        for h in (1, 2):
            assert bool((kv["lse"][b, h] == 123.0).all()) and bool((kv["score"][b, h] == 123.0).all())
            assert bool((kv["keep"][b, h] == -5).all())
        for h in (0, 3):
            assert bool(torch.isfinite(kv["lse"][b, h]).all())
            assert abs(float(kv["score"][b, h].double().sum()) - 64) < 1e-3


def test_lse_only_leaves_outputs_unchanged():
    """Exporting lse alone changes nothing else: outputs match a plain call."""
    N = 1024
    q, k, v = qkv(1, 2, 1, N, 26)
    kv = {"lse": torch.zeros(1, 2, N, dtype=torch.float32, device=q.device), "window": 0,
          "keep_k": 0}
    a = msa.msa_streaming(q, k, v, 1, 3, kv_select=kv)
    b = msa.msa_streaming(q, k, v, 1, 3)
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    mask = O.block_mask_from_blocks([O.streaming_blocks(m, 1, 3) for m in range((N + 63) // 64)], N)
    lse = O.row_lse(P.to_np(q[0, 1]), P.to_np(k[0, 0]), np.arange(N), mask, 1 / math.sqrt(D))
    check_lse(P.to_np(kv["lse"][0, 1]), lse, "lse only")


@pytest.mark.parametrize("name", ["mixed_128k"])
def test_kv_select_full_size(name):
    """The benchmark workload at full size: window 64, keep 4096 per head; the
    score of every key and lse of sampled rows for one head of each type."""
    w, q, k, v, heads = inputs.make_workload(name, device="cuda")
    N, G = w.seq_len, w.n_q_heads // w.n_kv_heads
    window, keep_k = 64, 4096
    kv = msa.kv_select_buffers(q, window, keep_k)
    out = torch.zeros_like(q)
    U = len(heads["vs"])
    ex = {"vertical": torch.empty(U, min(w.vertical_topk, N), dtype=torch.int32, device=q.device),
          "slash": torch.empty(U, min(w.slash, N), dtype=torch.int32, device=q.device)}
    msa.msa_vertical_slash(q, k, v, w.vertical_topk, w.slash, out, heads=heads["vs"], export=ex,
                           kv_select=kv)
    NB = (N + 63) // 64
    Ub = len(heads["bs"])
    exb = {"block_count": torch.empty(Ub, NB, dtype=torch.int32, device=q.device),
           "block_ids": torch.empty(Ub, NB, min(w.block_topk, NB), dtype=torch.int32,
                                    device=q.device)}
    msa.msa_block_sparse(q, k, v, w.block_topk, out, heads=heads["bs"], export=exb, kv_select=kv)
    msa.msa_streaming(q, k, v, w.init_num, w.local_window_num, out, heads=heads["st"],
                      kv_select=kv)
    torch.cuda.synchronize()
    rng = np.random.default_rng(w.seed)
    rows = np.unique(np.concatenate([rng.choice(N, 12, replace=False), [0, N - 65, N - 1]]))
    scale = 1 / math.sqrt(D)
    for kind in ("vs", "bs", "st"):
        h = heads[kind][0]
        qn, kn = P.to_np(q[0, h]), P.to_np(k[0, h // G])
        if kind == "vs":
            e = {n: t.cpu().numpy() for n, t in ex.items()}
            mask = O.vs_row_block_mask(e["slash"][0], e["vertical"][0], N)
        elif kind == "bs":
            cnt, ids = exb["block_count"].cpu().numpy(), exb["block_ids"].cpu().numpy()
            mask = O.block_mask_from_blocks([ids[0, m, :cnt[0, m]] for m in range(NB)], N)
        else:
            mask = O.block_mask_from_blocks(
                [O.streaming_blocks(m, w.init_num, w.local_window_num) for m in range(NB)], N)
        lse_rows = O.row_lse(qn, kn, rows, mask, scale)
        check_lse(P.to_np(kv["lse"][0, h])[rows], lse_rows, f"{kind} h{h} lse")
        win = np.arange(N - window, N)
        S = O.kv_score(qn, kn, O.row_lse(qn, kn, win, mask, scale), mask, window, scale)
        check_score(P.to_np(kv["score"][0, h]), S, f"{kind} h{h} score")
        check_keep(kv["keep"][0, h].cpu().numpy(), P.to_np(kv["score"][0, h]), S, keep_k,
                   f"{kind} h{h} keep")
