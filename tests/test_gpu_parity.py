"""CUDA path vs the fp64 oracle on sizes the oracle finishes in seconds.

Every case spans several 128-row query tiles; the ragged cases end on a
half tile (N % 128 == 64) and use vertical counts that are not multiples of
the 128-key column chunk.  All calls go through the C ABI (ctypes binding).
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


def qkv(B, Hq, Hkv, N, seed, vs=True, bs=False):
    q, k, v = inputs.make_qkv(B, Hq, Hkv, N, seed, vs_planting=vs, bs_planting=bs, device="cpu")
    return q.cuda(), k.cuda(), v.cuda()


def np64(t):
    return P.to_np(t)


# ----------------------------------------------------------------------------- streaming / dense
@pytest.mark.parametrize("N,Hq,Hkv", [(640, 2, 1), (1024, 4, 2), (64, 1, 1)])
def test_streaming_full_window_is_dense_causal(N, Hq, Hkv):
    q, k, v = qkv(1, Hq, Hkv, N, 11)
    out = msa.msa_streaming(q, k, v, 0, (N + 63) // 64)
    torch.cuda.synchronize()
    qn, kn, vn = np64(q), np64(k), np64(v)
    for h in range(Hq):
        ref = O.dense_causal(qn[0, h], kn[0, h // (Hq // Hkv)], vn[0, h // (Hq // Hkv)], 1 / math.sqrt(D))
        P.compare_out(np64(out[0, h]), ref, f"dense h{h}")


@pytest.mark.parametrize("N,init,local", [(1088, 1, 3), (2048, 2, 4), (1536, 0, 1), (960, 3, 2)])
def test_streaming_matches_oracle(N, init, local):
    q, k, v = qkv(1, 4, 2, N, 12)
    out = msa.msa_streaming(q, k, v, init, local)
    torch.cuda.synchronize()
    ref, _ = O.streaming_forward(q.cpu(), k.cpu(), v.cpu(), init, local)
    P.compare_out(np64(out[0]), ref[0], f"streaming N={N} init={init} local={local}")


def test_streaming_head_subset_leaves_other_heads():
    q, k, v = qkv(2, 4, 2, 512, 13)
    out = torch.full_like(q, 7.0)
    msa.msa_streaming(q, k, v, 1, 2, out=out, heads=[3, 0])
    torch.cuda.synchronize()
    ref, _ = O.streaming_forward(q.cpu(), k.cpu(), v.cpu(), 1, 2, heads=[3, 0])
    for b in range(2):
        P.compare_out(np64(out[b, 3]), ref[b, 0], "h3")
        P.compare_out(np64(out[b, 0]), ref[b, 1], "h0")
        assert (out[b, 1] == 7.0).all() and (out[b, 2] == 7.0).all()


def growth_inputs(N, kind, seed):
    """Rows whose running max rises far above its first value late in the row.

    Every query shares a direction u (|u| = 8).  "jump": one key late in the
    sequence gets 2u added, about 16 (log2 units) above every other logit of
    the rows that see it, so without the row-sum check its p would overflow
    f16.  "ramp": keys drift along u over the sequence, so a row's max grows
    by about one log2 unit per 128-key tile (16 in all) and the softmax has to
    move its running max and rescale O several times along each row.
    """
    g = torch.Generator().manual_seed(seed)
    u = torch.randn(D, generator=g)
    u = 8 * u / u.norm()
    q = u + 0.5 * torch.randn(N, D, generator=g)
    k = 0.3 * torch.randn(N, D, generator=g)
    if kind == "jump":
        k[3 * N // 4 + 5] += 2 * u
    else:
        k += torch.linspace(0, 2, N)[:, None] * u[None, :]
    v = torch.randn(N, D, generator=g)
    return [t.to(torch.bfloat16).reshape(1, 1, N, D).cuda() for t in (q, k, v)]


@pytest.mark.parametrize("kind", ["jump", "ramp"])
def test_softmax_running_max_growth(kind):
    """Both attention kernels against dense causal attention when the row max
    grows far after a row's first items: dense streaming and vertical-slash
    covering every key (two query tiles per CTA), block-sparse keeping every
    block (one query tile per CTA); row normalisers within the bound the
    KV-selection tests derive (|d lse| <= 1e-4)."""
    N = 2048
    NB = N // 64
    q, k, v = growth_inputs(N, kind, 40 if kind == "jump" else 41)
    qn, kn, vn = np64(q)[0, 0], np64(k)[0, 0], np64(v)[0, 0]
    scale = 1 / math.sqrt(D)
    ref = O.dense_causal(qn, kn, vn, scale)
    lse = torch.zeros(1, 1, N, device="cuda")
    outs = {
        "streaming": msa.msa_streaming(q, k, v, 0, NB,
                                       kv_select={"lse": lse, "window": 0, "keep_k": 0}),
        "vertical-slash": msa.msa_vertical_slash(q, k, v, N, N),
        "block-sparse": msa.msa_block_sparse(q, k, v, NB),
    }
    torch.cuda.synchronize()
    for name, out in outs.items():
        P.compare_out(np64(out[0, 0]), ref, f"{kind} {name}")
    ref_lse = O.row_lse(qn, kn, np.arange(N), lambda m: np.ones(N, dtype=bool), scale)
    err = np.abs(lse[0, 0].double().cpu().numpy() - ref_lse)
    assert err.max() <= 1e-4, f"{kind}: lse max err {err.max():.3e}"


# ----------------------------------------------------------------------------- block-sparse
@pytest.mark.parametrize("N,topk", [(2048, 5), (2112, 8), (1024, 100), (4096, 3), (640, 1)])
def test_block_sparse_matches_oracle(N, topk):
    q, k, v = qkv(1, 4, 2, N, 14, vs=False, bs=True)
    out, ex = P.run_bs(q, k, v, topk)
    qn, kn, vn = np64(q), np64(k), np64(v)
    NB = (N + 63) // 64
    for h in range(4):
        g = h // 2
        sel, S = O.block_sparse_blocks(qn[0, h], kn[0, g], topk)
        gpu_sel = []
        for m in range(NB):
            cnt = int(ex["block_count"][h, m])
            assert cnt == min(topk, m + 1)
            got = ex["block_ids"][h, m, :cnt]
            assert got[-1] == m, "diagonal block must be kept"
            if m > 0:
                P.check_topk(got[:-1], S[m, :m], topk - 1, f"h{h} m{m}")
            gpu_sel.append(got.astype(np.int64))
        ref, _ = O.attend_blocks(qn[0, h], kn[0, g], vn[0, g], O.block_mask_from_blocks(gpu_sel, N),
                                 1 / math.sqrt(D))
        P.compare_out(np64(out[0, h]), ref, f"bs h{h}")


def test_block_sparse_batch_and_head_subset():
    """A batch of two with a head subset on a ragged length (an odd number of
    128-row query tiles, the last one half real): the one-tile kernel's (batch,
    head) units and their tile lists, every other head left untouched."""
    N, topk, heads = 1088, 6, [3, 0]
    q, k, v = qkv(2, 4, 2, N, 18, vs=False, bs=True)
    out = torch.full_like(q, 7.0)
    NB = (N + 63) // 64
    U = 2 * len(heads)
    ex = {"block_count": torch.empty(U, NB, dtype=torch.int32, device="cuda"),
          "block_ids": torch.empty(U, NB, min(topk, NB), dtype=torch.int32, device="cuda")}
    msa.msa_block_sparse(q, k, v, topk, out, heads=heads, export=ex)
    torch.cuda.synchronize()
    qn, kn, vn = np64(q), np64(k), np64(v)
    counts, ids = ex["block_count"].cpu().numpy(), ex["block_ids"].cpu().numpy()
    for b in range(2):
        for t, h in enumerate(heads):
            u, g = b * len(heads) + t, h // 2
            _, S = O.block_sparse_blocks(qn[b, h], kn[b, g], topk)
            sel = []
            for m in range(NB):
                cnt = int(counts[u, m])
                assert cnt == min(topk, m + 1)
                got = ids[u, m, :cnt]
                assert got[-1] == m, "diagonal block must be kept"
                if m > 0:
                    P.check_topk(got[:-1], S[m, :m], topk - 1, f"b{b} h{h} m{m}")
                sel.append(got.astype(np.int64))
            ref, _ = O.attend_blocks(qn[b, h], kn[b, g], vn[b, g], O.block_mask_from_blocks(sel, N),
                                     1 / math.sqrt(D))
            P.compare_out(np64(out[b, h]), ref, f"bs b{b} h{h}")
        for h in (1, 2):
            assert (out[b, h] == 7.0).all(), f"head {h} outside the subset was written"


@pytest.mark.parametrize("NB", [4096, 4097])
def test_block_sparse_selection_at_long_lengths(NB):
    """The block selection runs as CTAs of eight row blocks sharing staged key
    chunks up to 4096 row blocks and as one CTA per row block beyond: every row
    block's kept set against the oracle on both sides of that bound, outputs on
    sampled rows (including the first and last rows and the rows at the bound)."""
    N, topk = 64 * NB, 100
    q, k, v = qkv(1, 1, 1, N, 15, vs=False, bs=True)
    out, ex = P.run_bs(q, k, v, topk)
    qn, kn, vn = np64(q)[0, 0], np64(k)[0, 0], np64(v)[0, 0]
    _, S = O.block_sparse_blocks(qn, kn, topk)
    gpu_sel = []
    for m in range(NB):
        cnt = int(ex["block_count"][0, m])
        assert cnt == min(topk, m + 1)
        got = ex["block_ids"][0, m, :cnt]
        assert got[-1] == m, "diagonal block must be kept"
        if m > 0:
            P.check_topk(got[:-1], S[m, :m], topk - 1, f"m{m}")
        gpu_sel.append(got.astype(np.int64))
    rng = np.random.default_rng(NB)
    rows = np.unique(np.concatenate([rng.integers(0, N, 40), [0, 64 * 4095, 64 * 4096 - 1, N - 1]]))
    mask = O.block_mask_from_blocks(gpu_sel, N)
    ref, _ = O.attend_rows(qn, kn, vn, rows, lambda i: mask(i // 64), 1 / math.sqrt(D))
    P.compare_out(np64(out[0, 0, rows]), ref, f"bs NB={NB}")


# ----------------------------------------------------------------------------- vertical-slash
def check_vs_case(q, k, v, vertical_topk, slash, last_q=64, heads=None, scale=None):
    out, ex = P.run_vs(q, k, v, vertical_topk, slash, last_q=last_q, heads=heads, scale=scale)
    B, Hq, N, _ = q.shape
    G = Hq // k.shape[1]
    heads_l = list(range(Hq)) if heads is None else list(heads)
    qn, kn, vn = np64(q), np64(k), np64(v)
    scale = 1 / math.sqrt(D) if scale is None else scale
    NB = (N + 63) // 64
    for b in range(B):
        for t, h in enumerate(heads_l):
            u = b * len(heads_l) + t
            vs_, ss_, _ = O.estimate_vs(qn[b, h], kn[b, h // G], last_q, scale)
            np.testing.assert_allclose(ex["v_score"][u], vs_, rtol=1e-4, atol=1e-6 * max(1, vs_.max()))
            np.testing.assert_allclose(ex["s_score"][u], ss_, rtol=1e-4, atol=1e-6 * max(1, ss_.max()))
            P.check_topk(ex["vertical"][u], vs_, vertical_topk, f"vertical u{u}")
            P.check_topk(ex["slash"][u], ss_, slash, f"slash u{u}")
            V = ex["vertical"][u].astype(np.int64)
            S = ex["slash"][u].astype(np.int64)
            act = O.vs_active_tiles(S, N)
            np.testing.assert_array_equal(P.dist_bits_to_active(ex["tile_dist"][u], NB), act)
            cols = O.vs_columns(V, act, N)
            P.check_vs_columns(ex, u, V, S, N, list(range(NB)), f"vs b{b} h{h}")
            ref, _ = O.attend_blocks(qn[b, h], kn[b, h // G], vn[b, h // G],
                                     O.vs_block_mask(act, cols, N), scale)
            P.compare_out(np64(out[b, h]), ref, f"vs b{b} h{h}")
    return out, ex


def test_vertical_slash_tiny_workload():
    """The 4096-token single-head workload in full: scores, sets, format, outputs."""
    w, q, k, v, _ = inputs.make_workload("vs_tiny", device="cpu")
    check_vs_case(q.cuda(), k.cuda(), v.cuda(), w.vertical_topk, w.slash)


@pytest.mark.parametrize("N,kv,ks,last_q", [(2368, 300, 200, 64), (1088, 130, 40, 64),
                                            (2048, 64, 2048, 32), (960, 960, 1, 64),
                                            (64, 5, 3, 64), (1536, 100, 30, 1),
                                            (4160, 200, 16, 8)])
def test_vertical_slash_ragged(N, kv, ks, last_q):
    q, k, v = qkv(1, 4, 2, N, 15)
    check_vs_case(q, k, v, kv, ks, last_q=last_q)


@pytest.mark.parametrize("N,ks,scale", [(2368, 200, 0.03), (4160, 16, 0.2)])
def test_vertical_slash_custom_scale(N, ks, scale):
    """A softmax scale other than 1/sqrt(d) on both prefill kernels (128 * 16 <
    4160: the one-query-tile kernel), estimate included."""
    q, k, v = qkv(1, 4, 2, N, 21)
    check_vs_case(q, k, v, 150, ks, scale=scale)


def test_streaming_custom_scale():
    q, k, v = qkv(2, 4, 2, 2500, 22)
    out = msa.msa_streaming(q, k, v, 2, 5, scale=0.25)
    torch.cuda.synchronize()
    ref, _ = O.streaming_forward(np64(q), np64(k), np64(v), 2, 5, scale=0.25)
    for b in range(2):
        for h in range(4):
            P.compare_out(np64(out[b, h]), ref[b, h], f"streaming scale b{b} h{h}")


def test_eight_query_heads_per_kv_head():
    """GQA with eight query heads on one KV head (the ratio of Llama-3-70B's
    layers): vertical-slash on both prefill kernels, block-sparse and
    streaming heads, each against the oracle."""
    N = 2240
    q, k, v = qkv(1, 8, 1, N, 25, bs=True)
    check_vs_case(q, k, v, 150, 300, heads=[0, 5])   # 128 * 300 >= N: two query tiles
    check_vs_case(q, k, v, 150, 12, heads=[7, 2])    # 128 * 12 < N: one query tile
    out, ex = P.run_bs(q, k, v, 7, heads=[3, 6])
    qn, kn, vn = np64(q), np64(k), np64(v)
    NB = (N + 63) // 64
    for u, h in enumerate([3, 6]):
        sel, S = O.block_sparse_blocks(qn[0, h], kn[0, 0], 7)
        gpu_sel = []
        for m in range(NB):
            cnt = int(ex["block_count"][u, m])
            assert cnt == min(7, m + 1)
            got = ex["block_ids"][u, m, :cnt]
            if m > 0:
                P.check_topk(got[:-1], S[m, :m], 6, f"bs h{h} m{m}")
            gpu_sel.append(got.astype(np.int64))
        ref, _ = O.attend_blocks(qn[0, h], kn[0, 0], vn[0, 0], O.block_mask_from_blocks(gpu_sel, N),
                                 1 / math.sqrt(D))
        P.compare_out(np64(out[0, h]), ref, f"bs h{h}")
    out = msa.msa_streaming(q, k, v, 1, 3, heads=[1, 4])
    torch.cuda.synchronize()
    ref, _ = O.streaming_forward(qn, kn, vn, 1, 3, heads=[1, 4])
    P.compare_out(np64(out[0, 1]), ref[0, 0], "streaming h1")
    P.compare_out(np64(out[0, 4]), ref[0, 1], "streaming h4")


def test_vertical_slash_batch_and_head_subset():
    q, k, v = qkv(2, 4, 1, 1024, 16)
    check_vs_case(q, k, v, 100, 150, heads=[2, 1])


@pytest.mark.parametrize("N,kv,ks", [(4096, 200, 20), (2112, 130, 10), (8192, 300, 50),
                                     (1217, 50, 5), (4160, 1, 1)])
def test_vertical_slash_sparse_tiles_one_tile_kernel(N, kv, ks):
    """Few slash lines for the length (128 * slash < N): the call runs on the
    one-query-tile kernel with packed 64-key block items and 64-key column
    halves; scores, sets, the exact format and the outputs against the oracle,
    including a ragged length and a single line of each kind."""
    assert 128 * ks < N
    q, k, v = qkv(1, 4, 2, N, 23)
    check_vs_case(q, k, v, kv, ks)


def test_vertical_slash_one_tile_kernel_batch_subset_and_normalisers():
    """The one-tile vertical-slash path with a batch of two, a head subset and
    the row normalisers (lse) against the oracle's over the GPU's own sets."""
    N, kv, ks, heads = 2176, 90, 8, [3, 0]
    q, k, v = qkv(2, 4, 2, N, 24)
    check_vs_case(q, k, v, kv, ks, heads=heads)
    kvb = msa.kv_select_buffers(q, 64, 16)
    out, ex = P.run_vs(q, k, v, kv, ks, heads=heads)
    msa.msa_vertical_slash(q, k, v, kv, ks, heads=heads, kv_select=kvb)
    torch.cuda.synchronize()
    qn, kn = np64(q), np64(k)
    for b in range(2):
        for t, h in enumerate(heads):
            u = b * len(heads) + t
            V, S = ex["vertical"][u].astype(np.int64), ex["slash"][u].astype(np.int64)
            act = O.vs_active_tiles(S, N)
            mask = O.vs_block_mask(act, O.vs_columns(V, act, N), N)
            ref = O.row_lse(qn[b, h], kn[b, h // 2], np.arange(N), mask, 1 / math.sqrt(D))
            got = kvb["lse"][b, h].double().cpu().numpy()
            fin = np.isfinite(ref)
            assert (np.isneginf(got) == ~fin).all()
            assert np.abs(got[fin] - ref[fin]).max() <= 1e-4


def test_vertical_topk_covering_all_keys_is_dense():
    q, k, v = qkv(1, 2, 1, 1152, 17)
    out, _ = P.run_vs(q, k, v, 5000, 2)
    qn, kn, vn = np64(q), np64(k), np64(v)
    for h in range(2):
        P.compare_out(np64(out[0, h]), O.dense_causal(qn[0, h], kn[0, 0], vn[0, 0], 1 / math.sqrt(D)),
                      f"dense-by-columns h{h}")


# ----------------------------------------------------------------------------- determinism / status
def test_repeat_calls_are_bit_identical_and_status_ok():
    q, k, v = qkv(1, 4, 2, 2048, 18, bs=True)
    ws = torch.empty(msa.workspace_bytes(msa.MSA_KIND_VERTICAL_SLASH, q, k, 300, 400),
                     dtype=torch.uint8, device="cuda")
    a = msa.msa_vertical_slash(q, k, v, 300, 400, workspace=ws)
    b = msa.msa_vertical_slash(q, k, v, 300, 400, workspace=ws)
    assert torch.equal(a, b)
    assert msa.device_status(ws) == msa.MSA_OK
    c = msa.msa_block_sparse(q, k, v, 7)
    d = msa.msa_block_sparse(q, k, v, 7)
    assert torch.equal(c, d)
    e = msa.msa_streaming(q, k, v, 1, 3)
    f = msa.msa_streaming(q, k, v, 1, 3)
    assert torch.equal(e, f)


def test_host_tensors_round_trip():
    q, k, v = inputs.make_qkv(1, 2, 1, 640, 19, device="cpu")
    out = msa.msa_streaming(q.pin_memory(), k.pin_memory(), v.pin_memory(), 1, 2)
    assert out.device.type == "cpu"
    ref, _ = O.streaming_forward(q, k, v, 1, 2)
    P.compare_out(np64(out[0]), ref[0], "host path")


def _all_heads(q, k, v):
    """One call of every head type on all heads (block-sparse and hierarchical
    heads with a few kept blocks, vertical-slash with column chunks)."""
    return {
        "streaming": msa.msa_streaming(q, k, v, 1, 3),
        "vertical-slash": msa.msa_vertical_slash(q, k, v, 150, 60),
        "block-sparse": msa.msa_block_sparse(q, k, v, 5),
        "hierarchical": msa.msa_hierarchical(q, k, v, [(4, 3), (1, 5)]),
    }


def test_values_beyond_f16_range_scale_exactly():
    """The P.V product reads an f16 copy of v; a KV head whose values leave the
    f16 range is copied scaled by 2^-e and its output multiplied by 2^e.
    Powers of two scale every f16 product and f32 sum exactly, so multiplying
    one KV head's v by 2^17 (values up to ~6e5) must multiply exactly that
    head group's outputs by 2^17, bit for bit, for every head type, while the
    other group's outputs stay the same.  (Values below the f16 normal range
    are zeroed first: the unscaled copy would round them, the scaled one not.)"""
    q, k, v = qkv(1, 4, 2, 1088, 21, bs=True)
    # no value in the f16 subnormal range, where the unscaled copy would round
    v = torch.where(v.abs() < 2.0 ** -13, torch.zeros_like(v), v)
    base = _all_heads(q, k, v)
    v2 = v.clone()
    v2[0, 0] *= 2.0 ** 17
    assert v2[0, 0].abs().max().item() > 65504
    big = _all_heads(q, k, v2)
    torch.cuda.synchronize()
    for name in base:
        assert torch.equal(big[name][0, :2], base[name][0, :2] * 2.0 ** 17), name
        assert torch.equal(big[name][0, 2:], base[name][0, 2:]), name


def test_values_beyond_f16_range_match_the_oracle():
    """v ~ 3e4 N(0, 1) (up to ~1.4e5, not a power-of-two multiple of anything in
    range) against the oracle on every head type.  The kernel's error scales
    with |v|, so the bounds are the parity tolerances times 3e4 (plus half a
    bf16 ulp of the reference)."""
    F = 3.0e4
    q, k, v = qkv(1, 2, 1, 1088, 22, bs=True)
    v = (v.float() * F).to(torch.bfloat16)
    assert v.abs().max().item() > 65504
    outs = _all_heads(q, k, v)
    torch.cuda.synchronize()
    qn, kn, vn = np64(q), np64(k), np64(v)
    ref = {"streaming": O.streaming_forward(q.cpu(), k.cpu(), v.cpu(), 1, 3)[0][0],
           "block-sparse": O.block_sparse_attention(q.cpu(), k.cpu(), v.cpu(), 5)[0][0],
           "hierarchical": O.hierarchical_sparse_attention(q.cpu(), k.cpu(), v.cpu(),
                                                           [(4, 3), (1, 5)])[0][0]}
    # vertical-slash: the oracle's attention over the GPU's own sets
    _, ex = P.run_vs(q, k, v, 150, 60)
    vsr = []
    for h in range(2):
        V, S = ex["vertical"][h].astype(np.int64), ex["slash"][h].astype(np.int64)
        act = O.vs_active_tiles(S, 1088)
        vsr.append(O.attend_blocks(qn[0, h], kn[0, 0], vn[0, 0],
                                   O.vs_block_mask(act, O.vs_columns(V, act, 1088), 1088),
                                   1 / math.sqrt(D))[0])
    ref["vertical-slash"] = np.stack(vsr)
    for name, out in outs.items():
        got, want = np64(out[0]), ref[name]
        d = np.abs(got - want)
        assert np.isfinite(got).all(), name
        assert (d <= F * P.MAX_TOL + P.half_ulp_bf16(want)).all(), (name, d.max())
        assert d.mean() <= F * P.MEAN_TOL, (name, d.mean())


def test_golden_tiny_block_sparse_and_streaming():
    """The hand-worked fixture through the CUDA path: its inputs are exact in
    bf16, so the block choice must equal the fixture's and the output rows its
    closed forms (within the output tolerance)."""
    import json
    import os
    with open(os.path.join(os.path.dirname(__file__), "golden", "bs_st_tiny.json")) as f:
        g = json.load(f)
    bs = g["block_sparse"]
    N = bs["N"]
    q, k, v = (torch.zeros(1, 1, N, D, dtype=torch.bfloat16) for _ in range(3))
    for m in range(N // 64):
        q[0, 0, 64 * m:64 * (m + 1), :2] = torch.tensor(bs["a"][m], dtype=torch.bfloat16)
        k[0, 0, 64 * m:64 * (m + 1), :2] = torch.tensor(bs["b"][m], dtype=torch.bfloat16)
        v[0, 0, 64 * m:64 * (m + 1), :] = bs["c"][m]
    q, k, v = q.cuda(), k.cuda(), v.cuda()
    for case in bs["cases"]:
        out, ex = P.run_bs(q, k, v, case["topk"])
        for m, blocks in enumerate(case["blocks"]):
            cnt = int(ex["block_count"][0, m])
            assert ex["block_ids"][0, m, :cnt].tolist() == blocks, f"topk {case['topk']} m {m}"
        got = np64(out[0, 0])
        for row, val in case["rows"].items():  # a single row: the bf16 cast alone moves it
            d = np.abs(got[int(row)] - val)    # up to half an ulp, so only the max bound applies
            assert d.max() <= P.MAX_TOL + P.half_ulp_bf16(val), (case["topk"], row, got[int(row), 0])
        ref, _ = O.block_sparse_attention(q.cpu(), k.cpu(), v.cpu(), case["topk"])
        P.compare_out(got, ref[0, 0], f"topk {case['topk']}")
    st = g["streaming"]
    q, k, v = qkv(1, 1, 1, st["N"], 14)
    for case in st["cases"]:
        out = msa.msa_streaming(q, k, v, case["init_num"], case["local_window_num"])
        torch.cuda.synchronize()
        ref, info = O.streaming_forward(q.cpu(), k.cpu(), v.cpu(), case["init_num"],
                                        case["local_window_num"])
        P.compare_out(np64(out[0]), ref[0], f"streaming {case}")
