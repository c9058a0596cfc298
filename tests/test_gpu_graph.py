"""A whole step (the three entry points on their head subsets) captured once
in a CUDA graph and replayed on new inputs gives bit-identical outputs to eager
calls: every call's host work (validation, TMA descriptors) runs at capture,
and the device work is kernel launches and one async memset per call."""
import pytest
import torch

from dynamic_sparse_attention_slash_gb300 import inputs, msa

pytestmark = pytest.mark.gpu


def test_step_replays_from_a_cuda_graph():
    N, Hq, Hkv = 2048, 4, 2
    heads = {"vs": [0, 3], "bs": [1], "st": [2]}
    q, k, v = (t.cuda() for t in inputs.make_qkv(1, Hq, Hkv, N, 70, vs_planting=True,
                                                  bs_planting=True, device="cpu"))
    out = torch.zeros_like(q)
    ws = {"vs": torch.empty(msa.workspace_bytes(0, q, k, 200, 300, 2), dtype=torch.uint8, device="cuda"),
          "bs": torch.empty(msa.workspace_bytes(1, q, k, 6, 0, 1), dtype=torch.uint8, device="cuda"),
          "st": torch.empty(msa.workspace_bytes(2, q, k, 0, 0, 1), dtype=torch.uint8, device="cuda")}

    def step(qq, kk, vv, oo):
        msa.msa_vertical_slash(qq, kk, vv, 200, 300, oo, heads=heads["vs"], workspace=ws["vs"])
        msa.msa_block_sparse(qq, kk, vv, 6, oo, heads=heads["bs"], workspace=ws["bs"])
        msa.msa_streaming(qq, kk, vv, 1, 3, oo, heads=heads["st"], workspace=ws["st"])

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step(q, k, v, out)  # warm-up outside capture (one-time attribute setup)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step(q, k, v, out)
    for seed in (71, 72):
        q2, k2, v2 = inputs.make_qkv(1, Hq, Hkv, N, seed, vs_planting=True, bs_planting=True,
                                     device="cpu")
        q.copy_(q2)
        k.copy_(k2)
        v.copy_(v2)
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        ref = torch.zeros_like(out)
        step(q, k, v, ref)
        torch.cuda.synchronize()
        assert torch.equal(out, ref), f"seed {seed}"


def test_one_tile_and_hierarchical_calls_replay_from_a_cuda_graph():
    """The one-query-tile kernel's vertical-slash path (128 * slash < N) and the
    hierarchical head, captured and replayed on new inputs: bit-identical to
    eager calls."""
    N, Hq, Hkv = 4160, 4, 2
    stages = [(4, 4), (1, 8)]
    heads = {"vs": [0, 2], "hip": [1, 3]}
    q, k, v = (t.cuda() for t in inputs.make_qkv(1, Hq, Hkv, N, 80, vs_planting=True,
                                                  bs_planting=True, device="cpu"))
    out = torch.zeros_like(q)
    ws = {"vs": torch.empty(msa.workspace_bytes(0, q, k, 200, 16, 2), dtype=torch.uint8, device="cuda"),
          "hip": torch.empty(msa.workspace_bytes(3, q, k, stages[-1][1], 0, 2), dtype=torch.uint8,
                             device="cuda")}

    def step(qq, kk, vv, oo):
        msa.msa_vertical_slash(qq, kk, vv, 200, 16, oo, heads=heads["vs"], workspace=ws["vs"])
        msa.msa_hierarchical(qq, kk, vv, stages, oo, heads=heads["hip"], workspace=ws["hip"])

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step(q, k, v, out)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step(q, k, v, out)
    for seed in (81, 82):
        q2, k2, v2 = inputs.make_qkv(1, Hq, Hkv, N, seed, vs_planting=True, bs_planting=True,
                                     device="cpu")
        q.copy_(q2)
        k.copy_(k2)
        v.copy_(v2)
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        ref = torch.zeros_like(out)
        step(q, k, v, ref)
        torch.cuda.synchronize()
        assert torch.equal(out, ref), f"seed {seed}"
        assert out[0, heads["vs"] + heads["hip"]].abs().sum() > 0
