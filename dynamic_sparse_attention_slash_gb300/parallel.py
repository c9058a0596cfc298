"""Head-sharded attention over several GPUs (one process per GPU).

Every query head of MInference-style sparse attention is independent: its own
estimate, index sets and attention (MInference 1.0 overview, section 2.2, per
head).  The natural split over GPUs is therefore by heads, in whole KV-head
groups so that each GPU holds only its own K/V heads, as tensor-parallel
attention splits heads (the Novita vLLM article confines sparsity to each
tensor-parallel rank for the same reason).  There is no communication inside
the operation; an optional all-gather afterwards gives every rank the full
output.  sharded_attention works on full-size tensors of which each rank reads
and writes its heads only; sharded_attention_local works on rank-local
tensors (each rank holds only its heads' q, k, v and out: the memory is
sharded too).
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


def local_head_range(n_q_heads: int, n_kv_heads: int, world: int, rank: int):
    """(query-head range, KV-head range) of `rank` as (start, stop) pairs: the
    slices of q/out and k/v a rank needs to hold (whole KV-head groups)."""
    heads = shard_heads(n_q_heads, n_kv_heads, world, rank)
    G = n_q_heads // n_kv_heads
    if not heads:
        return (0, 0), (0, 0)
    return (heads[0], heads[-1] + 1), (heads[0] // G, heads[-1] // G + 1)


def sharded_attention_local(call: Callable[..., object], q_loc, k_loc, v_loc, out_loc=None, *,
                            gather: bool = False, n_q_heads: Optional[int] = None,
                            n_kv_heads: Optional[int] = None, group=None):
    """Runs call(q_loc, k_loc, v_loc, out=out_loc) on rank-local tensors.

    Memory-sharded form: each rank holds only its own heads, q_loc / out_loc
    [B, Hq_loc, N, D] and k_loc / v_loc [B, Hkv_loc, N, D] (the slices that
    local_head_range names, e.g. loaded from the rank's part of a checkpoint),
    and the call runs on all of the local heads.  With gather=True the shards
    are all-gathered and the full output [B, n_q_heads, N, D] is returned
    (n_q_heads and n_kv_heads are the totals over all ranks); otherwise the
    local output.
    """
    if out_loc is None:
        out_loc = torch.zeros_like(q_loc)
    if q_loc.shape[1]:
        call(q_loc, k_loc, v_loc, out=out_loc)
    if not gather:
        return out_loc
    if n_q_heads is None or n_kv_heads is None:
        raise ValueError("gather needs the total numbers of query and KV heads")
    import torch.distributed as dist
    world = dist.get_world_size(group) if dist.is_available() and dist.is_initialized() else 1
    if world == 1:
        return out_loc
    B, _, N, D = out_loc.shape
    full = torch.empty((B, n_q_heads, N, D), dtype=out_loc.dtype, device=out_loc.device)
    _exchange(out_loc, full, n_q_heads, n_kv_heads, world, dist.get_rank(group), group)
    return full


def _exchange(mine_heads, full, Hq: int, Hkv: int, world: int, rank: int,
              group: Optional[object]) -> None:
    """All-gather of head shards into full [B, Hq, N, D].  Equal shards are
    gathered as they are; unequal ones (Hkv not a multiple of world) are padded
    to the largest for the exchange."""
    import torch.distributed as dist
    shards = [shard_heads(Hq, Hkv, world, r) for r in range(world)]
    width = max(len(s) for s in shards)
    B, _, N, D = full.shape
    if all(len(s) == width for s in shards):
        mine = mine_heads.contiguous()
    else:
        mine = torch.zeros((B, width, N, D), dtype=full.dtype, device=full.device)
        mine[:, : mine_heads.shape[1]] = mine_heads
    parts = [torch.empty_like(mine) for _ in range(world)]
    dist.all_gather(parts, mine, group=group)
    for r, s in enumerate(shards):
        if s:
            full[:, s[0]: s[-1] + 1] = parts[r][:, : len(s)]


def _gather_heads(out, Hq: int, Hkv: int, world: int, group: Optional[object]) -> None:
    """All-gather of the head shards of out [B, Hq, N, D] (shards may differ in
    size by one KV-head group: they are padded to the largest for the exchange)."""
    import torch.distributed as dist
    rank = dist.get_rank(group)
    h = shard_heads(Hq, Hkv, world, rank)
    mine = out[:, h[0]: h[-1] + 1] if h else out[:, :0]
    _exchange(mine, out, Hq, Hkv, world, rank, group)
