"""Seeded synthetic attention inputs shaped like Llama-3-8B attention layers.

This module only draws tensors.  It holds none of the sparse-attention
arithmetic, so both the CUDA path and the CPU oracle can be fed from it.

Workload recipes (one per named workload, all causal, d = 128):

* ``vs_tiny``     batch 1, 1 head, N = 4096, vertical-slash planting.
* ``vs_32k``      batch 1, 32 query heads / 8 KV heads, N = 32768, vertical-slash planting.
* ``bs_64k``      batch 1, 32/8 heads, N = 65536, block-local planting.
* ``mixed_128k``  batch 1, 32/8 heads, N = 131072, both plantings, seeded split of the
                  heads into 20 vertical-slash, 8 block-sparse and 4 streaming heads.
* ``vs_1m``       batch 1, 32/8 heads, N = 1048576, vertical-slash planting.
* ``hip_64k``     batch 1, 32/8 heads, N = 65536, block-local planting, every head
                  a hierarchical pruning head (chunks of 16, 4 and 1 blocks keeping
                  16, 40 and 100: 1024 candidate blocks -> 256 -> 160 -> 100).

Generation steps, in this order (all in fp32, one bf16 cast at the end):

1. Q, K, V ~ N(0, 1) i.i.d.
2. vertical-slash planting: Q += 1.0 * u for a fixed seeded unit vector u.
3. block-local planting: each 64-token block of each KV head draws a random
   vector of norm 2 that is added to that block's K rows and to the same rows
   of every query head in the KV head's group.
4. vertical-slash planting: K[0:4] += 8 u (sinks); 32 seeded key positions per
   KV head += 4 u (heavy keys); K[j] += 0.5 * mean over the group's query
   heads of Q[j] (the diagonal).
5. cast Q, K, V to bf16.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch

HEAD_DIM = 128
BLOCK = 64


@dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    n_q_heads: int
    n_kv_heads: int
    seq_len: int
    seed: int
    vs_planting: bool
    bs_planting: bool
    # per-head-type settings
    last_q: int = 64
    vertical_topk: int = 0
    slash: int = 0
    block_topk: int = 0
    init_num: int = 0
    local_window_num: int = 0
    # number of heads of each type (vertical-slash, block-sparse, streaming)
    head_split: tuple = (0, 0, 0)
    # hierarchical pruning heads (all heads when set) and their stages
    # ((chunk_blocks, keep), ...)
    hip_heads: int = 0
    hip_stages: tuple = ()
    extra: dict = field(default_factory=dict)


WORKLOADS = {
    "vs_tiny": Workload("vs_tiny", 1, 1, 1, 4096, 1000, True, False,
                        vertical_topk=256, slash=512, head_split=(1, 0, 0)),
    "vs_32k": Workload("vs_32k", 1, 32, 8, 32768, 1001, True, False,
                       vertical_topk=1000, slash=6096, head_split=(32, 0, 0)),
    "bs_64k": Workload("bs_64k", 1, 32, 8, 65536, 1002, False, True,
                       block_topk=100, head_split=(0, 32, 0)),
    "mixed_128k": Workload("mixed_128k", 1, 32, 8, 131072, 1003, True, True,
                           vertical_topk=1000, slash=6096, block_topk=100,
                           init_num=1, local_window_num=64, head_split=(20, 8, 4)),
    "vs_1m": Workload("vs_1m", 1, 32, 8, 1048576, 1004, True, False,
                      vertical_topk=1000, slash=6096, head_split=(32, 0, 0)),
    "hip_64k": Workload("hip_64k", 1, 32, 8, 65536, 1005, False, True,
                        hip_heads=32, hip_stages=((16, 16), (4, 40), (1, 100))),
}


def head_assignment(w: Workload) -> dict:
    """Seeded split of the query heads into the three head types.

    Returns {"vs": [...], "bs": [...], "st": [...], "hip": [...]} with
    ascending head ids.
    """
    if w.hip_heads:
        assert w.hip_heads == w.n_q_heads
        return {"vs": [], "bs": [], "st": [], "hip": list(range(w.n_q_heads))}
    n_vs, n_bs, n_st = w.head_split
    assert n_vs + n_bs + n_st == w.n_q_heads
    if n_bs == 0 and n_st == 0:
        return {"vs": list(range(w.n_q_heads)), "bs": [], "st": [], "hip": []}
    if n_vs == 0 and n_st == 0:
        return {"vs": [], "bs": list(range(w.n_q_heads)), "st": [], "hip": []}
    g = torch.Generator(device="cpu")
    g.manual_seed(w.seed * 7919 + 17)
    perm = torch.randperm(w.n_q_heads, generator=g).tolist()
    return {
        "vs": sorted(perm[:n_vs]),
        "bs": sorted(perm[n_vs:n_vs + n_bs]),
        "st": sorted(perm[n_vs + n_bs:]),
        "hip": [],
    }


def make_qkv(batch: int, n_q_heads: int, n_kv_heads: int, seq_len: int, seed: int, *,
             vs_planting: bool = True, bs_planting: bool = False, device="cpu",
             head_dim: int = HEAD_DIM, dtype=torch.bfloat16):
    """Draws q [B,Hq,N,d], k and v [B,Hkv,N,d] following the module recipe.

    Draws happen per (batch, KV head) group from one seeded generator on
    `device`, so the result depends on the device type (CPU and CUDA
    generators differ) but never on anything else.
    """
    assert n_q_heads % n_kv_heads == 0
    G = n_q_heads // n_kv_heads
    N, d = seq_len, head_dim
    dev = torch.device(device)
    gen = torch.Generator(device=dev)
    gen.manual_seed(seed)
    q = torch.empty(batch, n_q_heads, N, d, dtype=dtype, device=dev)
    k = torch.empty(batch, n_kv_heads, N, d, dtype=dtype, device=dev)
    v = torch.empty(batch, n_kv_heads, N, d, dtype=dtype, device=dev)
    u = torch.randn(d, generator=gen, device=dev, dtype=torch.float32)
    u = u / u.norm()
    for b in range(batch):
        for g in range(n_kv_heads):
            qg = torch.randn(G, N, d, generator=gen, device=dev, dtype=torch.float32)
            kg = torch.randn(N, d, generator=gen, device=dev, dtype=torch.float32)
            vg = torch.randn(N, d, generator=gen, device=dev, dtype=torch.float32)
            if vs_planting:
                qg += u
            if bs_planting:
                nb = (N + BLOCK - 1) // BLOCK
                off = torch.randn(nb, d, generator=gen, device=dev, dtype=torch.float32)
                off = 2.0 * off / off.norm(dim=1, keepdim=True)
                rows = off.repeat_interleave(BLOCK, dim=0)[:N]
                kg += rows
                qg += rows.unsqueeze(0)
            if vs_planting:
                kg[:min(4, N)] += 8.0 * u
                n_heavy = min(32, N)
                heavy = torch.randperm(N, generator=gen, device=dev)[:n_heavy]
                kg[heavy] += 4.0 * u
                kg += 0.5 * qg.mean(dim=0)
            q[b, g * G:(g + 1) * G] = qg.to(dtype)
            k[b, g] = kg.to(dtype)
            v[b, g] = vg.to(dtype)
            del qg, kg, vg
    return q, k, v


def make_workload(name: str, device="cpu"):
    """Returns (workload, q, k, v, heads) for a named workload."""
    w = WORKLOADS[name]
    q, k, v = make_qkv(w.batch, w.n_q_heads, w.n_kv_heads, w.seq_len, w.seed,
                       vs_planting=w.vs_planting, bs_planting=w.bs_planting, device=device)
    return w, q, k, v, head_assignment(w)
