"""Head sharding over ranks (parallel.py) on CPU: the shards are disjoint whole
KV-head groups that cover every head, and two gloo ranks running a stand-in
for the attention call end with the full output on both ranks."""
import os
import socket
import sys

import pytest
import torch
import torch.multiprocessing as mp

from dynamic_sparse_attention_slash_gb300.parallel import shard_heads


@pytest.mark.parametrize("Hq,Hkv,world", [(32, 8, 1), (32, 8, 2), (32, 8, 3), (32, 8, 8),
                                          (4, 4, 3), (6, 2, 4)])
def test_shards_cover_whole_groups(Hq, Hkv, world):
    G = Hq // Hkv
    shards = [shard_heads(Hq, Hkv, world, r) for r in range(world)]
    flat = [h for s in shards for h in s]
    assert flat == list(range(Hq))                       # disjoint, ordered, complete
    for s in shards:
        assert len(s) % G == 0 and (not s or s[0] % G == 0)   # whole KV groups
    sizes = sorted(len(s) // G for s in shards)
    assert sizes[-1] - sizes[0] <= 1                     # balanced


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import torch.distributed as dist
    from dynamic_sparse_attention_slash_gb300.parallel import sharded_attention
    dist.init_process_group("gloo", rank=rank, world_size=world)
    B, Hq, Hkv, N, D = 2, 12, 3, 8, 4
    qq = torch.zeros(B, Hq, N, D)
    kk = torch.zeros(B, Hkv, N, D)
    out = torch.full((B, Hq, N, D), -1.0)
    seen = []

    def fake_call(q_, k_, v_, out, heads):
        seen.extend(heads)
        for h in heads:
            out[:, h] = 100.0 * h + torch.arange(B).view(B, 1, 1).float()

    mine = sharded_attention(fake_call, qq, kk, kk, out)
    ok = all(bool((out[:, h] == 100.0 * h + torch.arange(B).view(B, 1, 1).float()).all())
             for h in range(Hq))
    dist.destroy_process_group()
    q.put((rank, mine, seen, ok))


@pytest.mark.parametrize("world", [2, 3])
def test_gloo_ranks_gather_the_full_output(world):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    all_heads = []
    for rank, mine, seen, ok in res:
        assert ok, f"rank {rank} does not hold the full output"
        assert mine == seen
        all_heads += mine
    assert sorted(all_heads) == list(range(12))


def _local_worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import torch.distributed as dist
    from dynamic_sparse_attention_slash_gb300.parallel import (local_head_range,
                                                               sharded_attention_local)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    B, Hq, Hkv, N, D = 2, 12, 3, 8, 4
    (h0, h1), (g0, g1) = local_head_range(Hq, Hkv, world, rank)
    # every rank builds only its own heads: q holds the head id, k the KV head id
    q_loc = torch.arange(h0, h1).float().view(1, -1, 1, 1).expand(B, -1, N, D).contiguous()
    k_loc = torch.arange(g0, g1).float().view(1, -1, 1, 1).expand(B, -1, N, D).contiguous()

    def fake_call(q_, k_, v_, out):
        G = q_.shape[1] // k_.shape[1]
        kk = k_.repeat_interleave(G, dim=1)
        out.copy_(100.0 * q_ + kk + torch.arange(B).view(B, 1, 1, 1).float())

    full = sharded_attention_local(fake_call, q_loc, k_loc, k_loc, gather=True, n_q_heads=Hq,
                                   n_kv_heads=Hkv)
    want = (100.0 * torch.arange(Hq).view(1, Hq, 1, 1) + (torch.arange(Hq) // (Hq // Hkv)).view(
        1, Hq, 1, 1) + torch.arange(B).view(B, 1, 1, 1)).float().expand(B, Hq, N, D)
    ok = bool(torch.equal(full, want))
    dist.destroy_process_group()
    q.put((rank, h1 - h0, g1 - g0, ok))


@pytest.mark.parametrize("world", [2, 3])
def test_gloo_ranks_with_local_shards_gather_the_full_output(world):
    """Memory-sharded form: each rank holds only its heads' tensors (whole
    KV-head groups); after the exchange every rank holds the full output,
    with unequal shards (3 KV heads over 2 ranks) and equal ones (3 over 3)."""
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_local_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert sum(r[1] for r in res) == 12 and sum(r[2] for r in res) == 3
    for rank, nq, nk, ok in res:
        assert ok, f"rank {rank} does not hold the full output"
        assert nq == 4 * nk
