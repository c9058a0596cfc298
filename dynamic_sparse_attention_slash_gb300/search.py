"""Kernel-aware sparse-pattern search (MInference 1.0 overview, section 2.1
"Kernel-Aware Optimal Sparse Pattern Search").

For one reference example the search runs every candidate setting of every
pattern on every selected head through the library's own calls, counts each
candidate's work as the attention kernel computes it (admitted (query, key)
pairs of the index sets the call built, flops.py), measures the recall of the
attention output as the dense attention mass the candidate's mask keeps
(msa_mass_recall on the row normalisers exported through msa_kv_select), and
assigns each head the pattern with the best recall among candidates of similar
cost: per pattern the most expensive setting within the FLOPs budget (the
cheapest when none fits), then the best recall (ties to the earlier pattern:
vertical-slash, block-sparse, streaming).

This module only orchestrates calls and applies the two choice rules on the
host; every piece of arithmetic on the tensors runs in the library's kernels.
"""
from __future__ import annotations

import time
from typing import Dict, Optional, Sequence

import torch

from . import msa
from .flops import bs_pairs, st_pairs, vs_pairs

PATTERNS = ("vs", "bs", "st")


def choose_setting(flops: Sequence[float], budget: float) -> int:
    """The most expensive setting whose FLOPs do not exceed the budget; if every
    setting exceeds it, the cheapest.  Ties go to the earlier setting."""
    fit = [i for i, f in enumerate(flops) if f <= budget]
    if fit:
        return min(fit, key=lambda i: (-flops[i], i))
    return min(range(len(flops)), key=lambda i: (flops[i], i))


def choose_pattern(recalls: Sequence[float]) -> int:
    """Highest recall; ties go to the earlier pattern."""
    return min(range(len(recalls)), key=lambda i: (-recalls[i], i))


def search(q, k, v, candidates: Dict[str, list], budget_flops: float, *,
           heads: Optional[Sequence[int]] = None, row0: int = 0, last_q: int = 64,
           stream=None) -> dict:
    """Runs the search on q [B,Hq,N,128], k/v [B,Hkv,N,128] (CUDA bf16).

    candidates: {"vs": [(vertical_topk, slash), ...], "bs": [topk, ...],
                 "st": [(init_num, local_window_num), ...]} (any subset of patterns).
    budget_flops: attention FLOPs per head (4 * d * pairs) a candidate may use.
    Recall is averaged over rows [row0, N).

    Returns {"assignment": {(b, h): (pattern, setting)}, "records": {(b, h):
    {pattern: {"flops": [...], "recall": [...], "setting": index}}}, "ms": wall
    time of the GPU work}.
    """
    B, Hq, N, D = q.shape
    NB = (N + 63) // 64
    heads_l = list(range(Hq)) if heads is None else [int(h) for h in heads]
    units = [(b, h) for b in range(B) for h in heads_l]
    order = [p for p in PATTERNS if candidates.get(p)]
    dev = q.device
    out = torch.empty_like(q)
    ref = {"lse": torch.zeros((B, Hq, N), dtype=torch.float32, device=dev), "window": 0,
           "keep_k": 0}
    cur = {"lse": torch.zeros_like(ref["lse"]), "window": 0, "keep_k": 0}
    recall = torch.zeros((B, Hq), dtype=torch.float32, device=dev)
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    # dense reference normalisers
    msa.msa_streaming(q, k, v, 0, NB, out, heads=heads_l, kv_select=ref, stream=stream)
    records = {u: {p: {"flops": [], "recall": []} for p in order} for u in units}
    U = len(units)
    for p in order:
        for setting in candidates[p]:
            if p == "vs":
                ex = {"vertical": torch.empty(U, min(setting[0], N), dtype=torch.int32, device=dev),
                      "tile_dist": torch.empty(U, (NB + 32) // 32, dtype=torch.int32, device=dev)}
                msa.msa_vertical_slash(q, k, v, setting[0], setting[1], out, last_q=last_q,
                                       heads=heads_l, export=ex, kv_select=cur, stream=stream)
            elif p == "bs":
                ex = {"block_count": torch.empty(U, NB, dtype=torch.int32, device=dev),
                      "block_ids": torch.empty(U, NB, min(setting, NB), dtype=torch.int32,
                                               device=dev)}
                msa.msa_block_sparse(q, k, v, setting, out, heads=heads_l, export=ex,
                                     kv_select=cur, stream=stream)
            else:
                ex = None
                msa.msa_streaming(q, k, v, setting[0], setting[1], out, heads=heads_l,
                                  kv_select=cur, stream=stream)
            msa.mass_recall(cur["lse"], ref["lse"], recall, row0=row0, heads=heads_l,
                            stream=stream)
            rec = recall.cpu()
            if p == "vs":
                td, vt = ex["tile_dist"].cpu().numpy(), ex["vertical"].cpu().numpy()
                pairs = [vs_pairs(td[u], vt[u], N) for u in range(U)]
            elif p == "bs":
                bc = ex["block_count"].cpu().numpy()
                pairs = [bs_pairs(bc[u], N) for u in range(U)]
            else:
                pairs = [st_pairs(N, setting[0], min(setting[1], NB))] * U
            for u, (b, h) in enumerate(units):
                records[(b, h)][p]["flops"].append(4 * D * pairs[u])
                records[(b, h)][p]["recall"].append(float(rec[b, h]))
    ms = (time.perf_counter() - t0) * 1e3
    assignment = {}
    for u in units:
        best = []
        for p in order:
            r = records[u][p]
            r["setting"] = choose_setting(r["flops"], budget_flops)
            best.append(r["recall"][r["setting"]])
        p = order[choose_pattern(best)]
        assignment[u] = (p, candidates[p][records[u][p]["setting"]])
    return {"assignment": assignment, "records": records, "ms": ms}


def assignment_groups(assignment: dict, n_heads: int) -> list:
    """Groups a search assignment {(b, h): (pattern, setting)} into calls:
    [(pattern, setting, [heads ascending])], one per distinct (pattern,
    setting).  A head must have the same assignment in every batch entry (the
    entry points select heads for the whole batch); every head in [0, n_heads)
    must be assigned."""
    per_head = {}
    for (b, h), ps in assignment.items():
        p, setting = ps
        if p not in PATTERNS:
            raise ValueError(f"unknown pattern {p!r}")
        setting = tuple(setting) if isinstance(setting, (list, tuple)) else setting
        if per_head.setdefault(h, (p, setting)) != (p, setting):
            raise ValueError(f"head {h} has different assignments across the batch")
    if sorted(per_head) != list(range(n_heads)):
        raise ValueError("every query head must be assigned exactly once")
    groups = {}
    for h in sorted(per_head):
        groups.setdefault(per_head[h], []).append(h)
    return [(p, setting, heads) for (p, setting), heads in groups.items()]


def apply_assignment(q, k, v, assignment: dict, out=None, *, last_q: int = 64, stream=None):
    """Runs attention with each head's searched pattern (the output of search()
    or any {(b, h): (pattern, setting)} map): one library call per distinct
    (pattern, setting) on its heads, all writing into one output tensor."""
    out = torch.empty_like(q) if out is None else out
    for p, setting, heads in assignment_groups(assignment, q.shape[1]):
        if p == "vs":
            msa.msa_vertical_slash(q, k, v, setting[0], setting[1], out, last_q=last_q,
                                   heads=heads, stream=stream)
        elif p == "bs":
            msa.msa_block_sparse(q, k, v, setting, out, heads=heads, stream=stream)
        else:
            msa.msa_streaming(q, k, v, setting[0], setting[1], out, heads=heads, stream=stream)
    return out

