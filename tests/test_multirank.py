"""The benchmark's multi-rank host logic on CPU with two gloo ranks: timing is
the maximum over ranks, work is the sum over ranks, and only rank 0 prints."""
import io
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    import bench
    r, local, w = bench.dist_setup()
    bench.barrier(w)
    mx = bench.max_over_ranks(10.0 + rank, w)
    sm = bench.sum_over_ranks(1.5 * (rank + 1), w)

    class Args:
        steps, warmup, gpus, workload, ref_rows = 1, 0, w, "vs_tiny", 2
    buf = io.StringIO()
    if rank == 1:  # the reference arm does no work and prints nothing off rank 0
        with redirect_stdout(buf):
            bench.run_reference(Args, r, w)
    import torch.distributed as dist
    dist.destroy_process_group()
    q.put((rank, r, w, mx, sm, buf.getvalue()))


def test_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, r, w, mx, sm, printed in res:
        assert r == rank and w == 2
        assert mx == 11.0 and sm == 1.5 + 3.0
        assert printed == ""
