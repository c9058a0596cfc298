"""Tensors in the [B, N, H, D] storage order that projection layers produce,
passed as [B, H, N, D] views (head stride D, row stride H * D): every head type
must give bit-identical outputs to the same call on contiguous copies (the
kernels are deterministic and the strides only change addresses), and the
contiguous call is checked against the oracle by the other parity tests.
"""
import pytest
import torch

from dynamic_sparse_attention_slash_gb300 import inputs, msa

pytestmark = pytest.mark.gpu
B, HQ, HKV, N, D = 2, 4, 2, 4160, 128


def bnhd(t):
    """A [B, H, N, D] view of a copy of t stored as [B, N, H, D]."""
    s = torch.empty(t.shape[0], t.shape[2], t.shape[1], t.shape[3], dtype=t.dtype, device=t.device)
    s.copy_(t.transpose(1, 2))
    return s.transpose(1, 2)


CALLS = {
    # 128 * 16 < N: sparse tiles, the one-query-tile kernel; 128 * 100 >= N: two tiles
    "vs_one_tile": lambda q, k, v, o: msa.msa_vertical_slash(q, k, v, 200, 16, o),
    "vs_two_tile": lambda q, k, v, o: msa.msa_vertical_slash(q, k, v, 200, 100, o),
    "block_sparse": lambda q, k, v, o: msa.msa_block_sparse(q, k, v, 8, o),
    "streaming": lambda q, k, v, o: msa.msa_streaming(q, k, v, 1, 4, o),
    "hierarchical": lambda q, k, v, o: msa.msa_hierarchical(q, k, v, [(4, 4), (1, 8)], o),
}


@pytest.mark.parametrize("kind", sorted(CALLS))
def test_bnhd_views_match_contiguous_tensors(kind):
    q, k, v = inputs.make_qkv(B, HQ, HKV, N, 1007, vs_planting=True, bs_planting=True,
                              device="cuda")
    ref = torch.zeros_like(q)
    CALLS[kind](q, k, v, ref)
    qs, ks, vs = bnhd(q), bnhd(k), bnhd(v)
    out = bnhd(torch.zeros_like(q))
    assert qs.stride() == (N * HQ * D, D, HQ * D, 1) and not out.is_contiguous()
    CALLS[kind](qs, ks, vs, out)
    torch.cuda.synchronize()
    assert torch.equal(out, ref), f"{kind}: strided call differs from the contiguous one"
    assert ref.abs().sum() > 0
