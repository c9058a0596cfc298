"""parallel.sharded_attention on one GPU (no process group: one rank holds
every head) equals the plain call, for each entry point bound with
functools.partial as the wrapper expects."""
import functools

import pytest
import torch

from dynamic_sparse_attention_slash_gb300 import inputs, msa
from dynamic_sparse_attention_slash_gb300.parallel import sharded_attention

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("call", [
    functools.partial(msa.msa_vertical_slash, vertical_topk=100, slash=150),
    functools.partial(msa.msa_block_sparse, topk=4),
    functools.partial(msa.msa_streaming, init_num=1, local_window_num=3)])
def test_single_rank_equals_plain_call(call):
    q, k, v = inputs.make_qkv(1, 4, 2, 1024, 60, vs_planting=True, bs_planting=True, device="cpu")
    q, k, v = q.cuda(), k.cuda(), v.cuda()
    out = torch.zeros_like(q)
    heads = sharded_attention(call, q, k, v, out)
    ref = call(q, k, v)
    torch.cuda.synchronize()
    assert heads == [0, 1, 2, 3]
    assert torch.equal(out, ref)


@pytest.mark.parametrize("world", [2, 4])
def test_local_shards_equal_the_plain_call(world):
    """Each simulated rank's local slices (local_head_range) through
    sharded_attention_local give that rank's heads of the plain call, bit for
    bit (every head is independent; no process group is needed without the
    exchange)."""
    from dynamic_sparse_attention_slash_gb300.parallel import (local_head_range,
                                                               sharded_attention_local)
    call = functools.partial(msa.msa_vertical_slash, vertical_topk=100, slash=150)
    q, k, v = inputs.make_qkv(1, 8, 4, 1024, 61, vs_planting=True, device="cpu")
    q, k, v = q.cuda(), k.cuda(), v.cuda()
    ref = call(q, k, v)
    for rank in range(world):
        (h0, h1), (g0, g1) = local_head_range(8, 4, world, rank)
        out = sharded_attention_local(call, q[:, h0:h1].contiguous(), k[:, g0:g1].contiguous(),
                                      v[:, g0:g1].contiguous())
        torch.cuda.synchronize()
        assert torch.equal(out, ref[:, h0:h1]), f"rank {rank}"
