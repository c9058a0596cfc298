"""msa_vertical_slash_static: vertical-slash attention for callers that cannot
allocate device memory where they run attention (a frozen allocator in a
fixed-pool serving runtime, a plugin host that passes an operator only its
inputs and outputs, or code that must avoid the synchronisation an allocation
can cause).  The entry point takes its scratch space from one fixed device
array inside the library instead of a caller workspace.

The GPU test calls it through the C ABI twice in a row, the second time with a
shorter sequence and other line counts, so the second call's buffers sit on the
first call's leftovers in the shared array.  Each output must equal the
workspace-taking msa_vertical_slash on the same inputs bit for bit (both run
the same deterministic kernels), and match the fp64 oracle given the index sets
the workspace call exports (which are themselves checked against the oracle's
scores).  The array's status word must read back OK.  This file is named to be
collected last; it passes both alone in a fresh process and after the other
tests.
"""
import ctypes
import math

import numpy as np
import pytest
import torch

from oracle import msa_oracle as O
from dynamic_sparse_attention_slash_gb300 import inputs, msa
from tests import parity as P

MSA_STATIC_SCRATCH_BYTES = 64 << 20


def static_entry():
    lib = msa.load_library()
    fn = lib.msa_vertical_slash_static
    T = ctypes.POINTER(msa.MsaTensor)
    fn.argtypes = [T, T, T, ctypes.c_int64, ctypes.c_int64, T, ctypes.c_void_p]
    fn.restype = ctypes.c_int
    status = lib.msa_vertical_slash_static_status
    status.argtypes = [ctypes.c_void_p]
    status.restype = ctypes.c_int
    return lib, fn, status


def fake(B, H, N, ptr):
    """A descriptor with a fake, never-dereferenced pointer (host-side checks only)."""
    return msa.MsaTensor(ptr, B, H, N, 128, H * N * 128, N * 128, 128)


def test_static_entry_rejects_on_host():
    """Sizes beyond the array, and invalid arguments, are refused before any work."""
    from dynamic_sparse_attention_slash_gb300 import build
    build.build()
    lib, fn, _ = static_entry()
    q, k, out = fake(1, 32, 32768, 1 << 32), fake(1, 8, 32768, 2 << 32), fake(1, 32, 32768, 3 << 32)
    need = lib.msa_workspace_bytes(msa.MSA_KIND_VERTICAL_SLASH, ctypes.byref(q), ctypes.byref(k),
                                   1000, 6096, 32)
    assert need > MSA_STATIC_SCRATCH_BYTES
    assert fn(ctypes.byref(q), ctypes.byref(k), ctypes.byref(k), 1000, 6096, ctypes.byref(out),
              None) == msa.MSA_ERR_WORKSPACE
    q4, k2, out4 = fake(1, 4, 32768, 1 << 32), fake(1, 2, 32768, 2 << 32), fake(1, 4, 32768, 3 << 32)
    assert lib.msa_workspace_bytes(msa.MSA_KIND_VERTICAL_SLASH, ctypes.byref(q4), ctypes.byref(k2),
                                   1000, 6096, 4) <= MSA_STATIC_SCRATCH_BYTES
    assert fn(ctypes.byref(q4), ctypes.byref(k2), ctypes.byref(k2), 0, 6096, ctypes.byref(out4),
              None) == msa.MSA_ERR_INVALID
    bad = fake(1, 4, 100, 4 << 32)
    assert fn(ctypes.byref(bad), ctypes.byref(k2), ctypes.byref(k2), 10, 10, ctypes.byref(out4),
              None) == msa.MSA_ERR_INVALID
    assert fn(ctypes.byref(q4), ctypes.byref(k2), ctypes.byref(k2), 10, 10, ctypes.byref(q4),
              None) == msa.MSA_ERR_INVALID  # out overlaps q


# (seed, N, vertical_topk, slash): the second call is shorter, so its buffers
# lie on the first call's leftovers in the array; the third runs the
# one-query-tile kernel (128 * 16 < N) over both
CALLS = [(41, 4096, 300, 500), (42, 2112, 130, 260), (43, 4160, 200, 16)]


@pytest.mark.gpu
def test_static_entry_matches_workspace_entry_twice():
    _, fn, status_fn = static_entry()
    stream = torch.cuda.current_stream()
    scale = 1 / math.sqrt(128)
    for call, (seed, N, kv, ks) in enumerate(CALLS):
        q, k, v = inputs.make_qkv(1, 4, 2, N, seed, vs_planting=True, device="cpu")
        q, k, v = q.cuda(), k.cuda(), v.cuda()
        ref, ex = P.run_vs(q, k, v, kv, ks)
        out = torch.zeros_like(q)
        qt, kt, vt, ot = (msa.describe(t) for t in (q, k, v, out))
        status = fn(ctypes.byref(qt), ctypes.byref(kt), ctypes.byref(vt), kv, ks,
                    ctypes.byref(ot), ctypes.c_void_p(stream.cuda_stream))
        assert status == msa.MSA_OK, f"call {call}: status {status}"
        assert status_fn(ctypes.c_void_p(stream.cuda_stream)) == msa.MSA_OK
        torch.cuda.synchronize()
        assert torch.equal(out, ref), f"call {call}: differs from the workspace call"
        qn, kn, vn = P.to_np(q), P.to_np(k), P.to_np(v)
        for h in range(4):
            g = h // 2
            vs_, ss_, _ = O.estimate_vs(qn[0, h], kn[0, g], 64, scale)
            P.check_topk(ex["vertical"][h], vs_, kv, f"call {call} h{h} vertical")
            P.check_topk(ex["slash"][h], ss_, ks, f"call {call} h{h} slash")
            V, S = ex["vertical"][h].astype(np.int64), ex["slash"][h].astype(np.int64)
            act = O.vs_active_tiles(S, N)
            want, _ = O.attend_blocks(qn[0, h], kn[0, g], vn[0, g],
                                      O.vs_block_mask(act, O.vs_columns(V, act, N), N), scale)
            P.compare_out(P.to_np(out[0, h]), want, f"static-scratch call {call} h{h}")
