"""The benchmark's exact pair counts (its FLOP numerator) agree with the
oracle's mask popcounts on small cases."""
import numpy as np
import pytest

import bench
from oracle import msa_oracle as O


def dist_words(S, N):
    NB = (N + 63) // 64
    words = np.zeros((NB + 32) // 32, dtype=np.int64)
    for o in S:
        for t in ([o // 64] + ([o // 64 + 1] if o % 64 else [])):
            words[t >> 5] |= 1 << (t & 31)
    return words


@pytest.mark.parametrize("seed", range(12))
def test_vs_pairs_match_mask_popcount(seed):
    rng = np.random.default_rng(seed)
    # half the cases end on a partial block
    N = 64 * int(rng.integers(1, 24)) - (int(rng.integers(1, 64)) if seed % 2 else 0)
    S = np.sort(rng.choice(N, size=int(rng.integers(1, 10)), replace=False))
    V = np.sort(rng.choice(N, size=int(rng.integers(1, 30)), replace=False))
    act = O.vs_active_tiles(S, N)
    cols = O.vs_columns(V, act, N)
    q = k = v = np.zeros((N, 128))
    _, counts = O.attend_blocks(q, k, v, O.vs_block_mask(act, cols, N), 1.0)
    assert bench.vs_pairs(dist_words(S, N), V, N) == int(counts.sum())


def test_bs_and_st_pairs():
    N = 1024
    rng = np.random.default_rng(0)
    q, k = rng.standard_normal((N, 128)), rng.standard_normal((N, 128))
    sel, _ = O.block_sparse_blocks(q, k, 3)
    assert bench.bs_pairs([len(s) for s in sel]) == O.nnz_from_blocks(sel, N)
    st = [O.streaming_blocks(m, 2, 3) for m in range(N // 64)]
    assert bench.st_pairs(N, 2, 3) == O.nnz_from_blocks(st, N)


@pytest.mark.parametrize("N", [1, 70, 1000, 1217])
def test_bs_and_st_pairs_at_ragged_length(N):
    rng = np.random.default_rng(N)
    q, k = rng.standard_normal((N, 128)), rng.standard_normal((N, 128))
    sel, _ = O.block_sparse_blocks(q, k, 3)
    assert bench.bs_pairs([len(s) for s in sel], N) == O.nnz_from_blocks(sel, N)
    NB = (N + 63) // 64
    st = [O.streaming_blocks(m, 1, 2) for m in range(NB)]
    assert bench.st_pairs(N, 1, 2) == O.nnz_from_blocks(st, N)


def test_measured_traffic_is_tied_to_kernel_source(monkeypatch):
    """The bench reports the captured DRAM traffic only for the workload and the
    kernel source it was measured on; anything else gives null."""
    import bench
    assert bench.measured_traffic("vs_32k", "vs") is None
    assert bench.measured_traffic("mixed_128k", "bs") is None
    stale = dict(bench.MEASURED_TRAFFIC, sha256="0" * 64)
    monkeypatch.setattr(bench, "MEASURED_TRAFFIC", stale)
    assert bench.measured_traffic("mixed_128k", "vs") is None


@pytest.mark.parametrize("N,nv,ns,seed", [(300, 20, 30, 1), (130, 130, 5, 2), (64, 1, 64, 3), (1000, 0, 7, 4)])
def test_exact_line_pairs_brute_force(N, nv, ns, seed):
    """The exact-line count (chosen columns and offsets without tile expansion)
    against the N x N causal mask built element by element."""
    import bench
    rng = np.random.default_rng(seed)
    V = np.sort(rng.choice(N, size=nv, replace=False)) if nv else np.zeros(0, np.int64)
    S = np.sort(rng.choice(N, size=ns, replace=False))
    i = np.arange(N)[:, None]
    j = np.arange(N)[None, :]
    mask = (j <= i) & (np.isin(j, V) | np.isin(i - j, S))
    assert bench.vs_exact_line_pairs(V, S, N) == int(mask.sum())


def test_reference_arm_prints_its_line_on_cpu():
    """bench.py --impl reference times the oracle on the host cores and prints
    one JSON line with the contract's keys (no GPU needed)."""
    import json
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference",
                        "--workload", "vs_tiny", "--steps", "1", "--warmup", "0",
                        "--ref-rows", "8"], capture_output=True, text=True, timeout=300, cwd=root)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0 and line["steps"] == 1
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"] == {"value": line["value"], "unit": line["unit"], "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}
    assert line["config"]["workload"] == "vs_tiny" and line["higher_is_better"] is True


def test_reference_arm_under_torchrun_prints_once():
    """Two ranks (gloo on CPU): rank 0 alone runs the oracle and prints; the
    other rank exits 0 without work."""
    import json
    import os
    import random
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    port = str(random.randint(20000, 40000))
    r = subprocess.run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
                        "--nproc-per-node", "2", "--master-addr", "127.0.0.1", "--master-port", port,
                        os.path.join(root, "bench.py"), "--impl", "reference", "--gpus", "2",
                        "--workload", "vs_tiny", "--steps", "1", "--warmup", "0", "--ref-rows", "8"],
                       capture_output=True, text=True, timeout=300, cwd=root)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [json.loads(l) for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    assert lines[0]["impl"] == "reference" and lines[0]["n_gpus"] == 2 and lines[0]["value"] > 0
