"""Benchmark: one step = the whole sparse-prefill hot path over one attention layer.

Default workload ``mixed_128k``: batch 1, 32 query heads / 8 KV heads, d = 128,
N = 131072 tokens, bf16, causal; a seeded split of the heads into 20
vertical-slash heads (vertical_topk 1000, slash 6096, last_q 64), 8
block-sparse heads (top-100 blocks) and 4 streaming heads (1 sink block, 64
local blocks).  One step calls msa_vertical_slash, msa_block_sparse and
msa_streaming on their head subsets of the same q/k/v/out tensors.

Metric: effective TFLOP/s = 4 * d * (admitted causal (query, key) pairs of the
method's own mask, counted exactly from the index sets) / step time, inputs
resident in HBM; `e2e` repeats it with the inputs in pinned host memory and
the host<->device copies inside the timed region.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
For N > 1 launch under torchrun: every rank runs its own copy of the workload
(weak scaling, no data-path collective).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from dynamic_sparse_attention_slash_gb300 import inputs  # noqa: E402
from dynamic_sparse_attention_slash_gb300.flops import (  # noqa: E402,F401
    bs_pairs, st_pairs, vs_exact_line_pairs, vs_pairs)

D = 128
METRIC = "sparse prefill attention effective TFLOP/s at 128K tokens"
UNIT = "TFLOP/s"


# ----------------------------------------------------------------------------- exact pair counts
# dram__bytes_read.sum + dram__bytes_write.sum of the vertical-slash prefill
# launch of the mixed 128K step, from one ncu capture of that one launch (one
# pass, full size).  The figure belongs to the kernel source it was taken on:
# once any of its files changes, the bench reports null until it is measured
# again.
MEASURED_TRAFFIC = {
    "workload": "mixed_128k",
    "kind": "vs",
    "bytes": 2.500e9 + 0.654e9,
    "sources": ("dynamic_sparse_attention_slash_gb300/csrc/prefill.cu",
                "dynamic_sparse_attention_slash_gb300/csrc/prefill_common.cuh",
                "dynamic_sparse_attention_slash_gb300/csrc/sm103_ptx.cuh",
                "dynamic_sparse_attention_slash_gb300/csrc/msa_internal.h"),
    "sha256": "dfaef1d9e422347163dddd5b709e13ce86816d072b1a65a4aa4aca3365612a4c",
}


# KV selection after the prefill: the observation window (query rows) follows
# the KV-sparsity page's worked example (256 instruction tokens); the page gives
# no kept count per head, 4096 is used here.
KV_WINDOW = 256
KV_KEEP = 4096

# Hierarchical pruning head measured beside the block-sparse heads of the step:
# chunks of 16, 4 and 1 blocks keeping 16, 40 and the block-sparse top-k.
HIER_STAGES = ((16, 16), (4, 40), (1, 100))

# Kernel-aware pattern search on the benchmark's own example: four settings per
# pattern around the workload's settings, at a budget of 10 % of the dense
# causal attention FLOPs per head.
SEARCH_BUDGET_FRAC = 0.10
SEARCH_CANDIDATES = {"vs": [(1000, 128), (1000, 256), (1000, 512), (1000, 1024)],
                     "bs": [25, 50, 100, 200],
                     "st": [(1, 64), (1, 128), (1, 256), (1, 512)]}


def measured_traffic(workload: str, kind: str):
    """DRAM bytes per launch of the dominant prefill launch, or None when no
    capture matches this workload and the current kernel source."""
    import hashlib
    t = MEASURED_TRAFFIC
    if workload != t["workload"] or kind != t["kind"]:
        return None
    h = hashlib.sha256()
    try:
        for f in t["sources"]:
            with open(os.path.join(ROOT, f), "rb") as fh:
                h.update(fh.read())
    except OSError:
        return None
    return t["bytes"] if h.hexdigest() == t["sha256"] else None


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 8:
                rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[0]) for r in rows if r[0].replace(".", "").isdigit()]
        mx = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, val in zip(names, r[4:8]) if val == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


# ----------------------------------------------------------------------------- distributed
def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend=backend)
    return rank, local, world


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    """Largest value of x over the ranks (timing: the slowest rank sets the time)."""
    if world <= 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x: float, world: int) -> float:
    if world <= 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# ----------------------------------------------------------------------------- CPU oracle leg
def oracle_sample(w, q, k, v, heads, rows_per_head: int, seed: int = 0):
    """Times the oracle on a bounded sample of the workload: for one head of each
    type, the full index construction plus attention for `rows_per_head` seeded
    query rows.  Returns (effective FLOPs of the sampled rows, seconds, label)."""
    from oracle import msa_oracle as O
    N = w.seq_len
    G = w.n_q_heads // w.n_kv_heads
    rng = np.random.default_rng(seed)
    scale = 1 / np.sqrt(D)
    flops = 0
    t0 = time.perf_counter()
    for kind in ("vs", "bs", "st", "hip"):
        if not heads[kind]:
            continue
        h = heads[kind][0]
        qn = q[0, h].to(torch.float64).numpy()
        kn = k[0, h // G].to(torch.float64).numpy()
        vn = v[0, h // G].to(torch.float64).numpy()
        rows = np.sort(rng.choice(N, size=rows_per_head, replace=False))
        if kind == "vs":
            idx = O.vertical_slash_indices(qn, kn, w.vertical_topk, w.slash, w.last_q, scale)
            mask = O.vs_block_mask(idx["active"], idx["columns"], N)
        elif kind == "bs":
            sel, _ = O.block_sparse_blocks(qn, kn, w.block_topk, scale)
            mask = O.block_mask_from_blocks(sel, N)
        elif kind == "hip":
            sel, _ = O.hierarchical_blocks(qn, kn, w.hip_stages, scale)
            mask = O.block_mask_from_blocks(sel, N)
        else:
            sel = [O.streaming_blocks(m, w.init_num, w.local_window_num) for m in range((N + 63) // 64)]
            mask = O.block_mask_from_blocks(sel, N)
        _, counts = O.attend_rows(qn, kn, vn, rows, lambda i: mask(i // 64), scale)
        flops += 4 * D * int(counts.sum())
    secs = time.perf_counter() - t0
    label = (f"one head of each type of {w.name}: full index construction + attention for "
             f"{rows_per_head} seeded query rows per head")
    return flops, secs, label


def sdpa_selected_backend(q, k, v) -> str:
    """The backend torch's scaled_dot_product_attention picks for these causal
    inputs by default (its own dispatch rule, asked without running it)."""
    try:
        from torch.nn.attention import SDPBackend
        idx = torch._fused_sdp_choice(q, k, v, None, 0.0, True)
        return SDPBackend(idx).name
    except Exception as exc:  # noqa: BLE001 - private helper; report why it failed
        return f"unknown ({type(exc).__name__})"


def time_sdpa(q, k, v, stream, d0, d1) -> float:
    """ms of one causal SDPA call after one warm-up call."""
    torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=True)
    d0.record(stream)
    torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=True)
    d1.record(stream)
    torch.cuda.synchronize()
    return d0.elapsed_time(d1)


def time_sdpa_backends(q, k, v, stream, d0, d1) -> dict:
    """ms of causal SDPA forced onto each fused backend in turn (a string where
    torch refuses the backend for these inputs)."""
    from torch.nn.attention import SDPBackend, sdpa_kernel
    res = {}
    for b in (SDPBackend.CUDNN_ATTENTION, SDPBackend.FLASH_ATTENTION,
              SDPBackend.EFFICIENT_ATTENTION):
        try:
            with sdpa_kernel([b]):
                res[b.name] = time_sdpa(q, k, v, stream, d0, d1)
        except RuntimeError as exc:
            res[b.name] = f"unavailable: {exc}"[:80]
    return res


def l2_note(q, k) -> str:
    """How the timed steps avoid an L2-warm advantage: the inputs' sizes
    against the 129 MB L2 (a step reads all of q, k and v)."""
    def size(t):
        n = t.numel() * t.element_size()
        return f"{n / 2**30:g} GiB" if n >= 2**30 else f"{n / 2**20:g} MiB"
    total = (q.numel() * q.element_size() + 2 * k.numel() * k.element_size()) / 1e6
    rel = "larger than" if total > 129 else "within"
    return f"inputs {rel} L2 (q {size(q)}, k and v {size(k)} each)"


def cpu_description() -> dict:
    """The host CPU the oracle ran on: architecture, model (as /proc/cpuinfo
    names it, when it does) and the logical CPU count."""
    import platform
    model = None
    try:
        with open("/proc/cpuinfo") as fh:
            for line in fh:
                key = line.split(":", 1)[0].strip().lower()
                if key in ("model name", "cpu part", "hardware"):
                    model = line.split(":", 1)[1].strip()
                    if key == "model name":
                        break
    except OSError:
        pass
    return {"machine": platform.machine(), "model": model, "os_cpu_count": os.cpu_count()}


def cpu_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def run_reference(args, rank, world):
    """Reference arm: the CPU oracle as it stands, timed on the host cores."""
    if rank != 0:
        return
    w = inputs.WORKLOADS[args.workload]
    q, k, v = inputs.make_qkv(w.batch, w.n_q_heads, w.n_kv_heads, w.seq_len, w.seed,
                              vs_planting=w.vs_planting, bs_planting=w.bs_planting, device="cpu")
    heads = inputs.head_assignment(w)
    for _ in range(args.warmup and 1):
        oracle_sample(w, q, k, v, heads, 8, seed=99)
    tot_f, tot_s = 0, 0.0
    label = ""
    for s in range(args.steps):
        f, secs, label = oracle_sample(w, q, k, v, heads, args.ref_rows, seed=s)
        tot_f += f
        tot_s += secs
    value = tot_f / tot_s / 1e12
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tot_s / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "impl": "reference",
            "config": {"workload": w.name, "seq_len": w.seq_len, "batch": w.batch,
                       "q_heads": w.n_q_heads, "kv_heads": w.n_kv_heads},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cpu_threads(),
                             "kind": "oracle", "sample": label},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- GPU arm
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="mixed_128k", choices=sorted(inputs.WORKLOADS))
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--cpu-rows", type=int, default=1536, help="oracle rows per head (cpu_baseline)")
    ap.add_argument("--ref-rows", type=int, default=24, help="oracle rows per head (reference arm)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-dense", action="store_true")
    ap.add_argument("--no-search", action="store_true",
                    help="skip the kernel-aware pattern search measurement")
    ap.add_argument("--no-kv-select", action="store_true",
                    help="skip the KV-selection measurement (window score + keep set)")
    ap.add_argument("--no-hier", action="store_true",
                    help="skip the hierarchical-head measurement on the block-sparse heads")
    args = ap.parse_args()
    rank, local, world = dist_setup()
    if args.impl == "reference":
        run_reference(args, rank, world)
        return

    from dynamic_sparse_attention_slash_gb300 import msa
    import json as _json

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w = inputs.WORKLOADS[args.workload]
    q, k, v = inputs.make_qkv(w.batch, w.n_q_heads, w.n_kv_heads, w.seq_len, w.seed,
                              vs_planting=w.vs_planting, bs_planting=w.bs_planting, device=dev)
    heads = inputs.head_assignment(w)
    N, B = w.seq_len, w.batch
    out = torch.zeros_like(q)
    stream = torch.cuda.current_stream(dev)

    ws = {}
    if heads["vs"]:
        ws["vs"] = torch.empty(msa.workspace_bytes(msa.MSA_KIND_VERTICAL_SLASH, q, k,
                                                   w.vertical_topk, w.slash, len(heads["vs"])),
                               dtype=torch.uint8, device=dev)
    if heads["bs"]:
        ws["bs"] = torch.empty(msa.workspace_bytes(msa.MSA_KIND_BLOCK_SPARSE, q, k, w.block_topk,
                                                   0, len(heads["bs"])), dtype=torch.uint8, device=dev)
    if heads["st"]:
        ws["st"] = torch.empty(msa.workspace_bytes(msa.MSA_KIND_STREAMING, q, k, 0, 0,
                                                   len(heads["st"])), dtype=torch.uint8, device=dev)
    if heads["hip"]:
        ws["hip"] = torch.empty(msa.workspace_bytes(msa.MSA_KIND_HIERARCHICAL, q, k,
                                                    w.hip_stages[-1][1], 0, len(heads["hip"])),
                                dtype=torch.uint8, device=dev)

    def new_events():
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(2 * msa.MSA_STAGE_COUNT)]
        for e in evs:
            e.record(stream)
        return evs

    def step(events=None, export=None, qq=q, kk=k, vv=v, oo=out, kv=None):
        ev = events or {}
        if heads["vs"]:
            msa.msa_vertical_slash(qq, kk, vv, w.vertical_topk, w.slash, oo, last_q=w.last_q,
                                   heads=heads["vs"], workspace=ws["vs"], stage_events=ev.get("vs"),
                                   export=(export or {}).get("vs"), kv_select=kv)
        if heads["bs"]:
            msa.msa_block_sparse(qq, kk, vv, w.block_topk, oo, heads=heads["bs"], workspace=ws["bs"],
                                 stage_events=ev.get("bs"), export=(export or {}).get("bs"),
                                 kv_select=kv)
        if heads["st"]:
            msa.msa_streaming(qq, kk, vv, w.init_num, w.local_window_num, oo, heads=heads["st"],
                              workspace=ws["st"], stage_events=ev.get("st"), kv_select=kv)
        if heads["hip"]:
            msa.msa_hierarchical(qq, kk, vv, w.hip_stages, oo, heads=heads["hip"],
                                 workspace=ws["hip"], stage_events=ev.get("hip"),
                                 export=(export or {}).get("hip"), kv_select=kv)

    # exact work of one step, from the GPU's own index sets
    U_vs, U_bs, U_hip = B * len(heads["vs"]), B * len(heads["bs"]), B * len(heads["hip"])
    export = {}
    if U_vs:
        export["vs"] = {"vertical": torch.empty(U_vs, min(w.vertical_topk, N), dtype=torch.int32, device=dev),
                        "slash": torch.empty(U_vs, min(w.slash, N), dtype=torch.int32, device=dev),
                        "tile_dist": torch.empty(U_vs, ((N + 63) // 64 + 32) // 32, dtype=torch.int32, device=dev)}
    if U_bs:
        export["bs"] = {"block_count": torch.empty(U_bs, (N + 63) // 64, dtype=torch.int32, device=dev)}
    if U_hip:
        export["hip"] = {"block_count": torch.empty(U_hip, (N + 63) // 64, dtype=torch.int32,
                                                    device=dev)}
    step(export=export)
    torch.cuda.synchronize()
    pairs = {"vs": 0, "bs": 0, "st": 0, "hip": 0}
    exact_line = 0  # vertical-slash pairs on the chosen lines alone (diagnostic)
    if U_vs:
        td, vt = export["vs"]["tile_dist"].cpu().numpy(), export["vs"]["vertical"].cpu().numpy()
        sl = export["vs"]["slash"].cpu().numpy()
        pairs["vs"] = sum(vs_pairs(td[u], vt[u], N) for u in range(U_vs))
        exact_line = sum(vs_exact_line_pairs(vt[u], sl[u], N) for u in range(U_vs))
    if U_bs:
        pairs["bs"] = bs_pairs(export["bs"]["block_count"].cpu().numpy(), N)
    if heads["st"]:
        pairs["st"] = B * len(heads["st"]) * st_pairs(N, w.init_num, w.local_window_num)
    if U_hip:  # whole kept blocks, the query block's own always among them
        pairs["hip"] = bs_pairs(export["hip"]["block_count"].cpu().numpy(), N)
    flops = {kk_: 4 * D * vv_ for kk_, vv_ in pairs.items()}
    step_flops = sum(flops.values())
    dense_pairs = B * w.n_q_heads * N * (N + 1) // 2

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    status = {kind: msa.device_status(buf) for kind, buf in ws.items()}

    # ---- timed region (device-resident inputs)
    kinds = [kind for kind in ("vs", "bs", "st", "hip") if heads[kind]]
    ev_sets = [{kind: new_events() for kind in kinds} for _ in range(args.steps)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    l0 = msa.kernel_launches()
    barrier(world)
    torch.cuda.synchronize()
    clocks.start()
    t_start.record(stream)
    for s in range(args.steps):
        step(events=ev_sets[s])
    t_end.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clock_info = clocks.stop()
    launches = msa.kernel_launches() - l0
    ms_total = t_start.elapsed_time(t_end)
    ms_total = max_over_ranks(ms_total, world)
    ms_step = ms_total / args.steps
    total_flops = sum_over_ranks(step_flops * args.steps, world)
    value = total_flops / (ms_total * 1e-3) / 1e12

    stage_ms = {}
    names = ["estimate", "topk", "index", "prefill"]
    for kind in kinds:
        for si, nm in enumerate(names):
            if kind != "vs" and nm in ("estimate", "topk"):
                continue
            if kind == "st" and nm == "index":
                continue
            vals = [ev[kind][2 * si].elapsed_time(ev[kind][2 * si + 1]) for ev in ev_sets]
            stage_ms[f"{kind}_{nm}"] = sum(vals) / len(vals)

    # ---- roofline of the dominant kernel: the first head kind present of
    # vertical-slash, block-sparse, hierarchical, streaming (block-sparse and
    # hierarchical heads run the one-tile kernel, the others the two-tile kernel)
    peaks = {}
    try:
        peaks = _json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
        peak, peak_src = float(peaks["bf16_tflops_sustained"]), "measured (sustained)"
    except (OSError, KeyError, ValueError):
        peak, peak_src = 1700.0, "fallback (sustained)"
    dom = next(kind for kind in ("vs", "bs", "hip", "st") if heads[kind])
    dom_ms = stage_ms[f"{dom}_prefill"]
    achieved = flops[dom] / (dom_ms * 1e-3) / 1e12
    roofline = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak, "traffic": measured_traffic(args.workload, dom),
                "kernel": ("sparse_prefill_tile_kernel" if dom in ("bs", "hip")
                           else "sparse_prefill_kernel"),
                "peak_source": peak_src,
                "frac_of_burst": achieved / float(peaks.get("bf16_tflops", 1900.0))}

    # ---- end to end: pinned host inputs and outputs, every copy inside the timed
    # region, through the package's host pipeline (pipeline.run_pipelined: inputs
    # and outputs double-buffered, copies on two side streams while steps compute)
    e2e = None
    if args.e2e_steps > 0:
        from dynamic_sparse_attention_slash_gb300 import pipeline as pl
        S = args.e2e_steps
        # pinned buffers in the memory of the GPU's own NUMA node (the CPU
        # affinity is restored after the measurement)
        affinity = os.sched_getaffinity(0)
        numa = pl.bind_to_gpu_node(dev)
        qh, kh, vh = (t.cpu().pin_memory() for t in (q, k, v))
        oh = [torch.empty(out.shape, dtype=out.dtype, pin_memory=True) for _ in range(2)]
        numa["q_pages_per_node"] = pl.buffer_numa_pages(qh)
        numa["out_pages_per_node"] = pl.buffer_numa_pages(oh[0])
        barrier(world)
        torch.cuda.synchronize()
        evs = pl.run_pipelined(lambda qq, kk, vv, oo: step(qq=qq, kk=kk, vv=vv, oo=oo),
                            [(qh, kh, vh)] * S, [oh[i % 2] for i in range(S)], stream=stream,
                            device=dev)
        torch.cuda.synchronize()
        barrier(world)
        e_ms = max_over_ranks(evs["start"].elapsed_time(evs["end"]), world)
        compute_ms = sum(a_.elapsed_time(b_) for a_, b_ in evs["compute"]) / S
        h2d_ms = sum(a_.elapsed_time(b_) for a_, b_ in evs["h2d"]) / S
        d2h_ms = sum(a_.elapsed_time(b_) for a_, b_ in evs["d2h"]) / S
        # where the time between the steps' compute went: before the first
        # step (its inputs' upload), between steps, after the last (the last
        # output's download)
        comp = evs["compute"]
        gaps = [comp[i - 1][1].elapsed_time(comp[i][0]) for i in range(1, S)]
        head_ms = evs["start"].elapsed_time(comp[0][0])
        tail_ms = comp[-1][1].elapsed_time(evs["end"])
        e_val = sum_over_ranks(step_flops * S, world) / (e_ms * 1e-3) / 1e12
        h2d = sum(t.numel() * t.element_size() for t in (qh, kh, vh))
        d2h = oh[0].numel() * oh[0].element_size()
        e2e = {"value": e_val, "unit": UNIT, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h,
               "ms_per_step": e_ms / S, "compute_ms_per_step": compute_ms, "steps": S,
               "h2d_ms_per_step": h2d_ms, "d2h_ms_per_step": d2h_ms,
               "h2d_gbps": h2d / (h2d_ms * 1e6), "d2h_gbps": d2h / (d2h_ms * 1e6),
               "before_first_ms": head_ms, "after_last_ms": tail_ms,
               "gap_ms_mean": sum(gaps) / max(len(gaps), 1), "gap_ms_max": max(gaps, default=0.0),
               "numa": numa,
               "pipelined": "pipeline.run_pipelined: double-buffered inputs/outputs, "
                            "copies on two side streams"}
        del qh, kh, vh, oh, evs
        os.sched_setaffinity(0, affinity)

    # ---- dense causal attention on the same GPU (context)
    dense = None
    if not args.no_dense and rank == 0:
        dout = torch.empty_like(q)
        d0, d1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        msa.msa_streaming(q, k, v, 0, (N + 63) // 64, dout)
        d0.record(stream)
        msa.msa_streaming(q, k, v, 0, (N + 63) // 64, dout)
        d1.record(stream)
        torch.cuda.synchronize()
        ours_ms = d0.elapsed_time(d1)
        sdpa_ms, backend, per_backend = None, None, {}
        try:
            G = w.n_q_heads // w.n_kv_heads
            kr, vr = k.repeat_interleave(G, dim=1), v.repeat_interleave(G, dim=1)
            backend = sdpa_selected_backend(q, kr, vr)
            sdpa_ms = time_sdpa(q, kr, vr, stream, d0, d1)
            per_backend = time_sdpa_backends(q, kr, vr, stream, d0, d1)
            del kr, vr
        except RuntimeError as exc:  # pragma: no cover
            backend = f"unavailable: {exc}"[:120]
        dense = {"flops": 4 * D * dense_pairs, "ours_ms": ours_ms,
                 "ours_tflops": 4 * D * dense_pairs / (ours_ms * 1e-3) / 1e12,
                 "sdpa_ms": sdpa_ms, "sdpa_backend": backend, "sdpa_ms_per_backend": per_backend,
                 "sdpa_tflops": (4 * D * dense_pairs / (sdpa_ms * 1e-3) / 1e12) if sdpa_ms else None}
        del dout

    # ---- KV selection after the prefill (a separate measurement, not part of the
    # step): row normalisers exported by the attention kernel, the score of every
    # key over the last KV_WINDOW query rows, and the KV_KEEP best keys per head
    kvsel = None
    if not args.no_kv_select and rank == 0:
        kvb = msa.kv_select_buffers(q, KV_WINDOW, KV_KEEP)
        step(kv=kvb)  # warm-up
        ev = {kind: new_events() for kind in kinds}
        torch.cuda.synchronize()
        step(events=ev, kv=kvb)
        torch.cuda.synchronize()
        kv_ms = {kind: e[2 * msa.MSA_STAGE_KV_SELECT].elapsed_time(e[2 * msa.MSA_STAGE_KV_SELECT + 1])
                 for kind, e in ev.items()}
        pf_ms = {kind: e[2 * msa.MSA_STAGE_PREFILL].elapsed_time(e[2 * msa.MSA_STAGE_PREFILL + 1])
                 for kind, e in ev.items()}
        n_heads = sum(B * len(heads[kind]) for kind in ev)
        # logits of the window rows against their causal keys, as dense work
        win_pairs = KV_WINDOW * N - KV_WINDOW * (KV_WINDOW - 1) // 2
        kvsel = {"window": KV_WINDOW, "keep_k": KV_KEEP, "ms": kv_ms, "ms_total": sum(kv_ms.values()),
                 "prefill_ms_with_lse_export": pf_ms,
                 "share_of_prefill": sum(kv_ms.values()) / max(sum(pf_ms.values()), 1e-9),
                 "score_tflops_dense_window": 2 * D * win_pairs * n_heads
                 / (sum(kv_ms.values()) * 1e-3) / 1e12}
        del kvb

    # ---- hierarchical pruning head (NEXT-3) on the step's block-sparse heads: the
    # same inputs and attention work budget (the last stage keeps the block-sparse
    # head's top-k), timed beside the block-sparse call (not part of the step)
    hier = None
    if not args.no_hier and rank == 0 and heads["bs"] and not heads["hip"]:
        hstages = HIER_STAGES[:-1] + ((1, w.block_topk),)
        hws = torch.empty(msa.workspace_bytes(msa.MSA_KIND_HIERARCHICAL, q, k, w.block_topk, 0,
                                              len(heads["bs"])), dtype=torch.uint8, device=dev)
        hcount = torch.empty(U_bs, (N + 63) // 64, dtype=torch.int32, device=dev)
        hout = torch.zeros_like(q)
        kw = dict(heads=heads["bs"], workspace=hws)
        msa.msa_hierarchical(q, k, v, hstages, hout, export={"block_count": hcount}, **kw)
        evh = new_events()
        evb = new_events()
        torch.cuda.synchronize()
        msa.msa_hierarchical(q, k, v, hstages, hout, stage_events=evh, **kw)
        msa.msa_block_sparse(q, k, v, w.block_topk, hout, heads=heads["bs"], workspace=ws["bs"],
                             stage_events=evb)
        torch.cuda.synchronize()
        si, sp = msa.MSA_STAGE_INDEX, msa.MSA_STAGE_PREFILL
        h_idx = evh[2 * si].elapsed_time(evh[2 * si + 1])
        h_pf = evh[2 * sp].elapsed_time(evh[2 * sp + 1])
        b_ms = evb[2 * si].elapsed_time(evb[2 * sp + 1])
        h_flops = 4 * D * bs_pairs(hcount.cpu().numpy(), N)
        hier = {"heads": len(heads["bs"]), "stages": [list(x) for x in hstages],
                "index_ms": h_idx, "prefill_ms": h_pf, "ms": h_idx + h_pf,
                "effective_tflops": h_flops / ((h_idx + h_pf) * 1e-3) / 1e12,
                "prefill_tflops": h_flops / (h_pf * 1e-3) / 1e12,
                "block_sparse_ms_same_heads": b_ms,
                "device_status": msa.device_status(hws)}
        del hws, hout

    # ---- kernel-aware pattern search (a separate measurement, not part of the step)
    psearch = None
    if not args.no_search and rank == 0:
        from dynamic_sparse_attention_slash_gb300 import search as msearch
        budget = SEARCH_BUDGET_FRAC * 4 * D * N * (N + 1) / 2
        res = msearch.search(q, k, v, SEARCH_CANDIDATES, budget, last_q=w.last_q)
        chosen = {p: 0 for p in msearch.PATTERNS}
        recalls = []
        for (b_, h_), (p_, _) in res["assignment"].items():
            chosen[p_] += 1
            r = res["records"][(b_, h_)][p_]
            recalls.append(r["recall"][r["setting"]])
        n_calls = 1 + sum(len(c) for c in SEARCH_CANDIDATES.values())
        psearch = {"ms": res["ms"], "calls": n_calls, "heads": len(res["assignment"]),
                   "budget_frac_of_dense": SEARCH_BUDGET_FRAC, "candidates": SEARCH_CANDIDATES,
                   "chosen": chosen, "mean_recall_of_choice": float(np.mean(recalls)),
                   "min_recall_of_choice": float(np.min(recalls))}

    # ---- CPU oracle on the host cores (rank 0, N = 1 only)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        qc, kc, vc = q.cpu(), k.cpu(), v.cpu()
        f, secs, label = oracle_sample(w, qc, kc, vc, heads, args.cpu_rows)
        cpu = {"value": f / secs / 1e12, "unit": UNIT, "cores": cpu_threads(), "kind": "oracle",
               "sample": label, "seconds": secs, "cpu": cpu_description()}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": w.name, "seq_len": N, "batch": B, "q_heads": w.n_q_heads,
                       "kv_heads": w.n_kv_heads, "head_dim": D,
                       "heads": {kk_: len(vv_) for kk_, vv_ in heads.items()},
                       "vertical_topk": w.vertical_topk, "slash": w.slash, "last_q": w.last_q,
                       "block_topk": w.block_topk, "init_num": w.init_num,
                       "local_window_num": w.local_window_num,
                       "hip_stages": [list(x) for x in w.hip_stages],
                       "l2": l2_note(q, k)},
            "roofline": roofline,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": launches,
            "clocks": clock_info,
            "stage_ms": stage_ms,
            "effective_tflop": {kk_: vv_ / 1e12 for kk_, vv_ in flops.items()},
            "density_vs_dense_causal": sum(pairs.values()) / dense_pairs,
            "vs_exact_line_pairs_fraction": (exact_line / pairs["vs"]) if pairs["vs"] else None,
            "dense_causal": dense,
            "device_status": status,
            "kv_select": kvsel,
            "hierarchical": hier,
            "pattern_search": psearch,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
