"""Host-to-device pipelining for batches that live in host memory.

A prefill service receives q/k/v on the host and returns the attention output
to the host.  run_pipelined() overlaps those copies with the attention itself:
inputs and outputs are double-buffered on the device, the host->device copy of
batch i+1 runs on one side stream and the device->host copy of batch i-1 on
another while batch i computes on the caller's stream.  Stream events order
every reuse of a buffer, so the result of each batch is exactly what one
synchronous call would give.
"""
from __future__ import annotations

import os
from typing import Callable, Sequence, Tuple

import torch


def run_pipelined(step: Callable[[torch.Tensor, torch.Tensor, torch.Tensor, torch.Tensor], None],
                  batches: Sequence[Tuple[torch.Tensor, torch.Tensor, torch.Tensor]],
                  outs: Sequence[torch.Tensor], stream: torch.cuda.Stream | None = None,
                  device=None) -> dict:
    """Runs step(q, k, v, out) on the device for every host batch.

    batches: (q, k, v) host tensors, pinned, all batches of one shape each;
    outs:    host tensors (pinned) receiving each batch's output; an entry may
             repeat (it is rewritten only after its previous copy finished).
    step:    enqueues the attention of device q, k, v into device out on the
             current stream (e.g. one or more msa_* calls).
    Returns the CUDA events of the run once everything is enqueued: "start" and
    "end" on the compute stream, and per batch the (start, end) pairs of its
    "compute", its host->device copies ("h2d", on the upload stream) and its
    device->host copy ("d2h", on the download stream); the caller
    synchronises (events["end"].synchronize()).
    """
    if len(batches) != len(outs) or not batches:
        raise ValueError("one host output per batch, at least one batch")
    device = torch.device(device) if device is not None else torch.device("cuda",
                                                                          torch.cuda.current_device())
    stream = stream or torch.cuda.current_stream(device)
    q0, k0, v0 = batches[0]
    for t in (q0, k0, v0, outs[0]):
        if t.is_cuda or not t.is_pinned():
            raise ValueError("batches and outs must be pinned host tensors")
    up, down = torch.cuda.Stream(device), torch.cuda.Stream(device)
    with torch.cuda.stream(stream):
        dev_in = [tuple(torch.empty(t.shape, dtype=t.dtype, device=device) for t in (q0, k0, v0))
                  for _ in range(2)]
        dev_out = [torch.zeros(outs[0].shape, dtype=outs[0].dtype, device=device)
                   for _ in range(2)]
    # the side streams use these buffers too: the allocator must not hand their
    # memory out again before that work is done
    for bufs in dev_in:
        for t in bufs:
            t.record_stream(up)
    for t in dev_out:
        t.record_stream(down)
    n = len(batches)
    ev = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    h2d_start, h2d_done = [ev() for _ in range(n)], [ev() for _ in range(n)]
    comp = [(ev(), ev()) for _ in range(n)]
    d2h_start, d2h_done = [ev() for _ in range(n)], [ev() for _ in range(n)]
    start, end = ev(), ev()
    last_out_copy = {}
    start.record(stream)
    for i, (qh, kh, vh) in enumerate(batches):
        b = i % 2
        qd, kd, vd = dev_in[b]
        with torch.cuda.stream(up):
            up.wait_event(start)
            if i >= 2:                      # device inputs b were read by batch i-2
                up.wait_event(comp[i - 2][1])
            h2d_start[i].record(up)
            qd.copy_(qh, non_blocking=True)
            kd.copy_(kh, non_blocking=True)
            vd.copy_(vh, non_blocking=True)
            h2d_done[i].record(up)
        stream.wait_event(h2d_done[i])
        if i >= 2:                          # device output b was read by copy-out i-2
            stream.wait_event(d2h_done[i - 2])
        comp[i][0].record(stream)
        with torch.cuda.stream(stream):
            step(qd, kd, vd, dev_out[b])
        comp[i][1].record(stream)
        with torch.cuda.stream(down):
            down.wait_event(comp[i][1])
            prev = last_out_copy.get(id(outs[i]))
            if prev is not None:            # same host buffer: keep the copies in order
                down.wait_event(prev)
            d2h_start[i].record(down)
            outs[i].copy_(dev_out[b], non_blocking=True)
            d2h_done[i].record(down)
            last_out_copy[id(outs[i])] = d2h_done[i]
    stream.wait_event(d2h_done[n - 1])
    end.record(stream)
    return {"start": start, "end": end, "compute": comp,
            "h2d": list(zip(h2d_start, h2d_done)), "d2h": list(zip(d2h_start, d2h_done))}


# ----------------------------------------------------------------------------- NUMA placement
def gpu_numa_node(device) -> int | None:
    """NUMA node of the host CPUs attached to a GPU (its PCI device's node in
    sysfs), or None where the system does not say."""
    try:
        p = torch.cuda.get_device_properties(torch.device(device))
        bdf = f"{p.pci_domain_id:04x}:{p.pci_bus_id:02x}:{p.pci_device_id:02x}.0"
        with open(f"/sys/bus/pci/devices/{bdf}/numa_node") as f:
            node = int(f.read().strip())
        return node if node >= 0 else None
    except (AttributeError, OSError, ValueError):
        return None


def node_cpus(node: int) -> set:
    """The CPUs of a NUMA node (sysfs cpulist, e.g. "0-71,144-215")."""
    cpus = set()
    with open(f"/sys/devices/system/node/node{node}/cpulist") as f:
        for part in f.read().strip().split(","):
            if part:
                lo, _, hi = part.partition("-")
                cpus.update(range(int(lo), int(hi or lo) + 1))
    return cpus


def bind_to_gpu_node(device) -> dict:
    """Restricts this process to the CPUs of the GPU's NUMA node (those the
    process may use), so that pinned host buffers allocated afterwards are
    placed in that node's memory (first touch).  Returns what was done."""
    node = gpu_numa_node(device)
    if node is None:
        return {"gpu_numa_node": None, "bound": False}
    try:
        cpus = node_cpus(node) & os.sched_getaffinity(0)
        if cpus:
            os.sched_setaffinity(0, cpus)
        return {"gpu_numa_node": node, "bound": bool(cpus), "cpus": len(cpus)}
    except OSError:
        return {"gpu_numa_node": node, "bound": False}


def buffer_numa_pages(t: torch.Tensor) -> dict:
    """Pages of the host mapping holding tensor t, per NUMA node, from
    /proc/self/numa_maps ({node: pages}; empty where the kernel does not say)."""
    addr = t.data_ptr()
    best = None
    try:
        with open("/proc/self/numa_maps") as f:
            for line in f:
                start = int(line.split(" ", 1)[0], 16)
                if start <= addr and (best is None or start > best[0]):
                    best = (start, line)
    except OSError:
        return {}
    pages = {}
    if best is not None:
        for field in best[1].split():
            if field[:1] == "N" and "=" in field:
                node, cnt = field[1:].split("=")
                if node.isdigit():
                    pages[int(node)] = pages.get(int(node), 0) + int(cnt)
    return pages
