"""C-ABI checks that need no GPU: the library loads, exports every function
include/msa.h declares, sizes workspaces, and rejects bad arguments on the
host before anything is enqueued (fake, never-dereferenced pointers)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_checked_build_exports_the_same_functions():
    """The bounds-checking build declares and rejects exactly like the ordinary one."""
    from dynamic_sparse_attention_slash_gb300 import build
    chk = ctypes.CDLL(build.build(checked=True))
    for name in declared_functions():
        assert hasattr(chk, name), name
    chk.msa_status_string.restype = ctypes.c_char_p
    assert b"bounds" in chk.msa_status_string(6)


@pytest.fixture(scope="module")
def lib():
    from dynamic_sparse_attention_slash_gb300 import build, msa
    build.build()
    return msa.load_library()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "msa.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(msa_[a-z_]+)\s*\(", src)))


def test_exports_every_declared_function(lib):
    from dynamic_sparse_attention_slash_gb300 import msa
    names = declared_functions()
    assert set(msa.EXPORTED_SYMBOLS) <= set(names)
    for name in names:
        assert hasattr(lib, name), name


_next_ptr = [0]


def T(B=1, H=4, N=1024, D=128, ptr=None, sb=None, sh=None, sn=None):
    """A tensor descriptor; without ptr, a fresh fake address 4 GiB from the last."""
    from dynamic_sparse_attention_slash_gb300.msa import MsaTensor
    if ptr is None:
        _next_ptr[0] += 1
        ptr = _next_ptr[0] << 32
    sn = D if sn is None else sn
    sh = N * sn if sh is None else sh
    sb = H * sh if sb is None else sb
    return MsaTensor(ptr, B, H, N, D, sb, sh, sn)


def opts(**kw):
    from dynamic_sparse_attention_slash_gb300.msa import MsaOpts
    o = MsaOpts()
    for k_, v_ in kw.items():
        setattr(o, k_, v_)
    return o


def call_vs(lib, q, k, v, out, kv=100, ks=100, o=None):
    return lib.msa_vertical_slash(ctypes.byref(q), ctypes.byref(k), ctypes.byref(v), kv, ks,
                                  ctypes.byref(out), ctypes.byref(o) if o is not None else None)


def test_workspace_bytes(lib):
    q, k = T(H=32), T(H=8)
    vs = lib.msa_workspace_bytes(0, ctypes.byref(q), ctypes.byref(k), 1000, 6096, 0)
    bs = lib.msa_workspace_bytes(1, ctypes.byref(q), ctypes.byref(k), 100, 0, 0)
    st = lib.msa_workspace_bytes(2, ctypes.byref(q), ctypes.byref(k), 0, 0, 0)
    assert vs > 32 * 1024 * 4 * 2 and bs > 0 and st > 256
    assert st >= 8 * 1024 * 128 * 2  # staged f16 copy of v
    assert vs % 256 == 0 and bs % 256 == 0 and st % 256 == 0
    assert lib.msa_workspace_bytes(0, ctypes.byref(q), ctypes.byref(k), 0, 6096, 0) == 0
    assert lib.msa_workspace_bytes(7, ctypes.byref(q), ctypes.byref(k), 1, 1, 0) == 0
    # fewer heads need less
    assert lib.msa_workspace_bytes(0, ctypes.byref(q), ctypes.byref(k), 1000, 6096, 4) < vs


@pytest.mark.parametrize("case,expect", [
    ("null_q", 1), ("d64", 2), ("n_huge", 2), ("misaligned", 1), ("gqa", 1), ("kv0", 1),
    ("flags", 1), ("lastq", 1), ("head_range", 1), ("head_dup", 1), ("no_ws", 3),
    ("small_ws", 3), ("ws_align", 3), ("odd_stride", 1), ("n_mismatch", 1),
    ("out_is_q", 1), ("out_overlaps_v", 1), ("ws_overlaps_k", 3),
    ("rows_overlap", 1), ("heads_alias", 1), ("bnhd_layout", 3), ("bnhd_rows_overlap", 1),
])
def test_vertical_slash_rejects(lib, case, expect):
    q, k, v, out = T(), T(H=2), T(H=2), T()
    o = opts(workspace=0x100000, workspace_bytes=1 << 40)
    kv = 100
    if case == "null_q":
        q = T(ptr=0)
    elif case == "d64":
        q, out = T(D=64), T(D=64)
    elif case == "n_huge":
        n = (1 << 21) + 64
        q, k, v, out = T(N=n), T(H=2, N=n), T(H=2, N=n), T(N=n)
    elif case == "misaligned":
        k = T(H=2, ptr=(1 << 40) + 8)
    elif case == "gqa":
        k, v = T(H=3), T(H=3)
    elif case == "kv0":
        kv = 0
    elif case == "flags":
        o.flags = 1
    elif case == "lastq":
        o.last_q = 65
    elif case in ("head_range", "head_dup"):
        arr = (ctypes.c_int32 * 2)(*([0, 4] if case == "head_range" else [1, 1]))
        o.heads = ctypes.cast(arr, ctypes.POINTER(ctypes.c_int32))
        o.n_heads = 2
    elif case == "no_ws":
        o = None
    elif case == "small_ws":
        o.workspace_bytes = 1024
    elif case == "ws_align":
        o.workspace = 0x100010
    elif case == "odd_stride":
        q = T(sn=130)
    elif case == "n_mismatch":
        v = T(H=2, N=2048)
    elif case == "out_is_q":
        out = T(ptr=q.data)
    elif case == "out_overlaps_v":  # out starts inside v's last head
        out = T(ptr=v.data + (2 * 1024 * 128 - 64) * 2)
    elif case == "ws_overlaps_k":
        o.workspace = k.data + 0x1000
    elif case == "rows_overlap":  # row i + 1 starts inside row i
        q = T(sn=64)
    elif case == "heads_alias":  # every head on the same memory
        q = T(sh=0)
    elif case == "bnhd_layout":  # [B, N, H, D] storage seen as [B, H, N, D]: valid,
        q = T(sn=4 * 128, sh=128, sb=1024 * 4 * 128)  # stops at the missing workspace
        o = None
    elif case == "bnhd_rows_overlap":  # heads interleaved with too small a row stride
        q = T(sn=2 * 128, sh=128, sb=1024 * 4 * 128)
    assert call_vs(lib, q, k, v, out, kv=kv, o=o) == expect


def test_block_sparse_and_streaming_reject(lib):
    q, k, v, out = T(), T(H=2), T(H=2), T()
    o = opts(workspace=0x100000, workspace_bytes=1 << 40)
    args = [ctypes.byref(x) for x in (q, k, v)]
    assert lib.msa_block_sparse(*args, 0, ctypes.byref(out), ctypes.byref(o)) == 1
    assert lib.msa_block_sparse(*args, 5, ctypes.byref(out), None) == 3
    assert lib.msa_streaming(*args, -1, 4, ctypes.byref(out), ctypes.byref(o)) == 1
    assert lib.msa_streaming(*args, 1, 0, ctypes.byref(out), ctypes.byref(o)) == 1
    small = opts(workspace=0x100000, workspace_bytes=64)
    assert lib.msa_streaming(*args, 1, 4, ctypes.byref(out), ctypes.byref(small)) == 3


@pytest.mark.parametrize("stages,expect", [
    ([(4, 3), (1, 4)], 3),            # valid: stops at the missing workspace
    ([(1, 5)], 3),
    ([], 1),                          # no stage
    ([(4, 3), (2, 4)], 1),            # the last stage must select single blocks
    ([(4, 3), (4, 2), (1, 4)], 1),    # chunk sizes must decrease
    ([(6, 3), (4, 2), (1, 4)], 1),    # ... each dividing the one before
    ([(4, 0), (1, 4)], 1),            # keep >= 1
    ([(0, 3), (1, 4)], 1),
    ([(2 ** c, 2) for c in range(8, -1, -1)], 1),  # more than MSA_HIP_MAX_STAGES stages
])
def test_hierarchical_rejects(lib, stages, expect):
    from dynamic_sparse_attention_slash_gb300 import msa
    q, k, v, out = T(), T(H=2), T(H=2), T()
    arr = msa.hip_stages(stages) if stages else (msa.MsaHipStage * 1)()
    st = lib.msa_hierarchical(ctypes.byref(q), ctypes.byref(k), ctypes.byref(v), arr,
                              len(stages), ctypes.byref(out), None)
    assert st == expect


def test_hierarchical_workspace_bytes(lib):
    from dynamic_sparse_attention_slash_gb300 import msa
    q, k = T(H=32, N=131072), T(H=8, N=131072)
    w = lib.msa_workspace_bytes(msa.MSA_KIND_HIERARCHICAL, ctypes.byref(q), ctypes.byref(k),
                                100, 0, 8)
    NB = 131072 // 64
    # pooled queries, one slab of block maxima (all 2048 query blocks fit), kept ids
    assert w >= 8 * NB * (128 * 4 + NB * 4 + 100 * 4) and w % 256 == 0
    assert lib.msa_workspace_bytes(msa.MSA_KIND_HIERARCHICAL, ctypes.byref(q), ctypes.byref(k),
                                   0, 0, 8) == 0
    # long sequences keep the block maxima to one slab of query blocks
    q2, k2 = T(H=32, N=1 << 20), T(H=8, N=1 << 20)
    w2 = lib.msa_workspace_bytes(msa.MSA_KIND_HIERARCHICAL, ctypes.byref(q2), ctypes.byref(k2),
                                 100, 0, 32)
    NB2 = (1 << 20) // 64
    assert w2 < 32 * NB2 * NB2 * 4 / 8 and w2 > (512 << 20)


def test_status_strings_and_counter(lib):
    for code in range(7):
        assert lib.msa_status_string(code)
    assert lib.msa_status_string(99) == b"unknown status"
    assert lib.msa_kernel_launches() >= 0


def test_struct_layout_matches_header(tmp_path):
    """The ctypes mirror of msa_opts / msa_kv_select has the C layout (gcc)."""
    from dynamic_sparse_attention_slash_gb300.msa import MsaKvSelect, MsaOpts
    src = tmp_path / "layout.c"
    src.write_text(
        '#include <stddef.h>\n#include <stdio.h>\n#include "msa.h"\n'
        'int main(void) { printf("%zu %zu %zu %zu %zu %zu\\n", sizeof(msa_opts), '
        'offsetof(msa_opts, flags), offsetof(msa_opts, kv_select), sizeof(msa_kv_select), '
        'offsetof(msa_kv_select, window), offsetof(msa_kv_select, keep_k)); return 0; }\n')
    exe = tmp_path / "layout"
    import subprocess
    subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)],
                   check=True)
    got = [int(x) for x in subprocess.run([str(exe)], capture_output=True, text=True,
                                          check=True).stdout.split()]
    assert got == [ctypes.sizeof(MsaOpts), MsaOpts.flags.offset, MsaOpts.kv_select.offset,
                   ctypes.sizeof(MsaKvSelect), MsaKvSelect.window.offset,
                   MsaKvSelect.keep_k.offset]


def test_kv_select_rejected_on_host(lib):
    from dynamic_sparse_attention_slash_gb300 import msa
    q, k, v, out = T(), T(), T(), T()

    def status(**kw):
        kv = msa.MsaKvSelect(**kw)
        o = opts(kv_select=ctypes.pointer(kv))
        return call_vs(lib, q, k, v, out, o=o)

    ok_buf = 0x20000
    assert status(lse=None, score=ok_buf, window=64) == msa.MSA_ERR_INVALID
    assert status(lse=ok_buf, score=ok_buf, window=0) == msa.MSA_ERR_INVALID
    assert status(lse=ok_buf, score=ok_buf, window=1025) == msa.MSA_ERR_INVALID
    assert status(lse=ok_buf, keep=ok_buf, keep_k=8) == msa.MSA_ERR_INVALID   # keep needs score
    assert status(lse=ok_buf, score=ok_buf, window=64, keep=ok_buf, keep_k=0) == msa.MSA_ERR_INVALID
    assert status(lse=ok_buf + 2, window=64) == msa.MSA_ERR_INVALID           # misaligned
    # a valid selection block passes validation and then fails on the missing workspace
    assert status(lse=ok_buf, score=ok_buf, window=64, keep=ok_buf, keep_k=8) == \
        msa.MSA_ERR_WORKSPACE


def test_binding_refuses_buffers_the_library_would_overrun():
    """The Python binding checks every export / KV buffer before the call."""
    import torch
    from dynamic_sparse_attention_slash_gb300 import msa

    class Q:  # only the shape is read
        shape = (1, 4, 1000, 128)

    with pytest.raises(ValueError):  # not written by a block-sparse call
        msa._check_buffers(Q, msa.MSA_KIND_BLOCK_SPARSE, 8, 0, None,
                           {"slash": torch.zeros(4, dtype=torch.int32)}, None)
    with pytest.raises(ValueError):  # host memory
        msa._check_buffers(Q, msa.MSA_KIND_VERTICAL_SLASH, 10, 10, None,
                           {"vertical": torch.zeros(40, dtype=torch.int32)}, None)
    with pytest.raises(ValueError):
        msa._check_buffers(Q, msa.MSA_KIND_STREAMING, 0, 0, None, None,
                           {"lse": torch.zeros(4000), "window": 1, "keep_k": 0})


def test_selftest_wait_timeout_rejects_on_host(lib):
    """Bad arguments are refused before anything is launched."""
    import ctypes
    from dynamic_sparse_attention_slash_gb300 import msa
    ok_ptr = ctypes.c_void_p(0x100000)  # never dereferenced: every case below is refused
    assert lib.msa_selftest_wait_timeout(None, 1000, None) == msa.MSA_ERR_INVALID
    assert lib.msa_selftest_wait_timeout(ctypes.c_void_p(0x100010), 1000, None) == msa.MSA_ERR_INVALID
    assert lib.msa_selftest_wait_timeout(ok_ptr, 0, None) == msa.MSA_ERR_INVALID
    assert lib.msa_selftest_wait_timeout(ok_ptr, 1000001, None) == msa.MSA_ERR_INVALID


def _build_c_example(out_path):
    """Compiles include/msa_example.cu against the in-tree libmsa.so."""
    import subprocess
    from dynamic_sparse_attention_slash_gb300 import build
    build.build()
    pkg = os.path.dirname(build.LIB_PATH)
    cmd = [build.nvcc(), "-std=c++17", *build.ARCH, "-I", os.path.join(ROOT, "include"),
           os.path.join(ROOT, "include", "msa_example.cu"), "-L", pkg, "-l:libmsa.so",
           "-Xlinker", f"-rpath={pkg}", "-o", str(out_path)]
    return subprocess.run(cmd, capture_output=True, text=True)


def test_c_example_compiles_and_links(tmp_path):
    """The C ABI is usable from C++ alone: the example builds and links."""
    r = _build_c_example(tmp_path / "msa_example")
    assert r.returncode == 0, r.stderr[-2000:]
