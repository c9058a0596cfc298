"""Head-sharded attention over several GPUs (one process per GPU).

Every query head of MInference-style sparse attention is independent: its own
estimate, index sets and attention (MInference 1.0 overview, section 2.2, per
head).  The natural split over GPUs is therefore by heads, in whole KV-head
groups so that each GPU holds only its own K/V heads, as tensor-parallel
attention splits heads (the Novita vLLM article confines sparsity to each
tensor-parallel rank for the same reason).  There is no communication inside
the operation; an optional all-gather afterwards gives every rank the full
output.
"""
from __future__ import annotations

from typing import Callable, List, Optional

import torch


def shard_heads(n_q_heads: int, n_kv_heads: int, world: int, rank: int) -> List[int]:
    """Query heads of `rank`: a contiguous run of whole KV-head groups, the
    groups dealt out as evenly as possible (earlier ranks take the extra one)."""
    if n_q_heads % n_kv_heads:
        raise ValueError("query heads must be a multiple of KV heads")
    if not 0 <= rank < world:
        raise ValueError("rank out of range")
    G = n_q_heads // n_kv_heads
    base, extra = divmod(n_kv_heads, world)
    g0 = rank * base + min(rank, extra)
    g1 = g0 + base + (1 if rank < extra else 0)
    return list(range(g0 * G, g1 * G))


def sharded_attention(call: Callable[..., object], q, k, v, out, *, gather: bool = True,
                      group=None) -> List[int]:
    """Runs call(q, k, v, out=out, heads=...) for this rank's head shard.

    call is one of the msa_* entry points with its pattern arguments bound
    (e.g. functools.partial(msa.msa_vertical_slash, vertical_topk=1000,
    slash=6096)).  q/out hold every query head and k/v every KV head (only this
    rank's heads are read or written).  With gather=True and more than one
    rank, the head shards of out are exchanged with all-gather so that every
    rank ends with the full output.  Returns this rank's heads.
    """
    import torch.distributed as dist
    world = dist.get_world_size(group) if dist.is_available() and dist.is_initialized() else 1
    rank = dist.get_rank(group) if world > 1 else 0
    Hq, Hkv = q.shape[1], k.shape[1]
    heads = shard_heads(Hq, Hkv, world, rank)
    if heads:
        call(q, k, v, out=out, heads=heads)
    if gather and world > 1:
        _gather_heads(out, Hq, Hkv, world, group)
    return heads


def _gather_heads(out, Hq: int, Hkv: int, world: int, group: Optional[object]) -> None:
    """All-gather of the head shards of out [B, Hq, N, D] (shards may differ in
    size by one KV-head group: they are padded to the largest for the exchange)."""
    import torch.distributed as dist
    shards = [shard_heads(Hq, Hkv, world, r) for r in range(world)]
    width = max(len(s) for s in shards)
    B, _, N, D = out.shape
    rank = dist.get_rank(group)
    mine = torch.zeros((B, width, N, D), dtype=out.dtype, device=out.device)
    h = shards[rank]
    if h:
        mine[:, : len(h)] = out[:, h[0]: h[-1] + 1]
    parts = [torch.empty_like(mine) for _ in range(world)]
    dist.all_gather(parts, mine, group=group)
    for r, s in enumerate(shards):
        if s:
            out[:, s[0]: s[-1] + 1] = parts[r][:, : len(s)]
