"""Python binding of libmsa (argument marshalling only).

Every function here forwards torch tensors to the C ABI declared in
include/msa.h as raw device pointers plus the current CUDA stream; all
computation happens in the library's CUDA kernels.  The library must have
been built (``python -m dynamic_sparse_attention_slash_gb300.build`` or
``__graft_entry__.build()``): there is no fallback.

Host (CPU) tensors are accepted for the end-to-end path: they are copied to the
device on the call's stream, the kernels run, and the output is copied back.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import torch

_PKG_DIR = os.path.dirname(os.path.abspath(__file__))
# MSA_LIBRARY names another build of the same library to load instead (for
# instance the bounds-checking build, libmsa_checked.so).
LIB_PATH = os.environ.get("MSA_LIBRARY") or os.path.join(_PKG_DIR, "libmsa.so")
# MSA_STRICT_STATUS=1: every call waits for its work and raises MsaError when
# its device status word is not MSA_OK (a debugging mode; it synchronises).
STRICT_STATUS = bool(os.environ.get("MSA_STRICT_STATUS"))

MSA_OK = 0
MSA_ERR_INVALID = 1
MSA_ERR_UNSUPPORTED = 2
MSA_ERR_WORKSPACE = 3
MSA_ERR_CUDA = 4
MSA_ERR_TIMEOUT = 5
MSA_ERR_BOUNDS = 6

MSA_KIND_VERTICAL_SLASH = 0
MSA_KIND_BLOCK_SPARSE = 1
MSA_KIND_STREAMING = 2
MSA_KIND_HIERARCHICAL = 3
MSA_HIP_MAX_STAGES = 8

MSA_STAGE_ESTIMATE = 0
MSA_STAGE_TOPK = 1
MSA_STAGE_INDEX = 2
MSA_STAGE_PREFILL = 3
MSA_STAGE_KV_SELECT = 4
MSA_STAGE_COUNT = 5

EXPORTED_SYMBOLS = (
    "msa_vertical_slash", "msa_block_sparse", "msa_streaming", "msa_workspace_bytes",
    "msa_device_status", "msa_status_string", "msa_kernel_launches", "msa_mass_recall",
    "msa_selftest_wait_timeout", "msa_hierarchical", "msa_vertical_slash_static",
    "msa_vertical_slash_static_status",
)


class MsaError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} (status {status})")


class MsaTensor(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("B", ctypes.c_int64), ("H", ctypes.c_int64),
                ("N", ctypes.c_int64), ("D", ctypes.c_int64), ("sb", ctypes.c_int64),
                ("sh", ctypes.c_int64), ("sn", ctypes.c_int64)]


class MsaIndexExport(ctypes.Structure):
    _fields_ = [("v_score", ctypes.c_void_p), ("s_score", ctypes.c_void_p),
                ("vertical", ctypes.c_void_p), ("slash", ctypes.c_void_p),
                ("tile_dist", ctypes.c_void_p), ("block_count", ctypes.c_void_p),
                ("block_ids", ctypes.c_void_p), ("col_count", ctypes.c_void_p),
                ("col_chunks", ctypes.c_void_p)]


class MsaHipStage(ctypes.Structure):
    _fields_ = [("chunk_blocks", ctypes.c_int64), ("keep", ctypes.c_int64)]


class MsaKvSelect(ctypes.Structure):
    _fields_ = [("lse", ctypes.c_void_p), ("score", ctypes.c_void_p), ("keep", ctypes.c_void_p),
                ("window", ctypes.c_int64), ("keep_k", ctypes.c_int64)]


class MsaOpts(ctypes.Structure):
    _fields_ = [("stream", ctypes.c_void_p), ("last_q", ctypes.c_int64), ("scale", ctypes.c_float),
                ("heads", ctypes.POINTER(ctypes.c_int32)), ("n_heads", ctypes.c_int32),
                ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t),
                ("export_idx", ctypes.POINTER(MsaIndexExport)),
                ("stage_events", ctypes.POINTER(ctypes.c_void_p)), ("flags", ctypes.c_int32),
                ("kv_select", ctypes.POINTER(MsaKvSelect))]


_lib = None


def load_library():
    """Loads libmsa.so; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build the CUDA library first "
                          "(python -m dynamic_sparse_attention_slash_gb300.build)")
    lib = ctypes.CDLL(LIB_PATH)
    T = ctypes.POINTER(MsaTensor)
    O = ctypes.POINTER(MsaOpts)
    lib.msa_vertical_slash.argtypes = [T, T, T, ctypes.c_int64, ctypes.c_int64, T, O]
    lib.msa_vertical_slash.restype = ctypes.c_int
    lib.msa_block_sparse.argtypes = [T, T, T, ctypes.c_int64, T, O]
    lib.msa_block_sparse.restype = ctypes.c_int
    lib.msa_streaming.argtypes = [T, T, T, ctypes.c_int64, ctypes.c_int64, T, O]
    lib.msa_streaming.restype = ctypes.c_int
    lib.msa_hierarchical.argtypes = [T, T, T, ctypes.POINTER(MsaHipStage), ctypes.c_int32, T, O]
    lib.msa_hierarchical.restype = ctypes.c_int
    lib.msa_workspace_bytes.argtypes = [ctypes.c_int, T, T, ctypes.c_int64, ctypes.c_int64,
                                        ctypes.c_int32]
    lib.msa_workspace_bytes.restype = ctypes.c_size_t
    lib.msa_device_status.argtypes = [ctypes.c_void_p, ctypes.c_void_p]
    lib.msa_device_status.restype = ctypes.c_int
    lib.msa_status_string.argtypes = [ctypes.c_int]
    lib.msa_status_string.restype = ctypes.c_char_p
    lib.msa_kernel_launches.argtypes = []
    lib.msa_kernel_launches.restype = ctypes.c_uint64
    F = ctypes.c_void_p
    lib.msa_mass_recall.argtypes = [F, F, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                    ctypes.c_int64, ctypes.POINTER(ctypes.c_int32), ctypes.c_int32,
                                    F, ctypes.c_void_p]
    lib.msa_mass_recall.restype = ctypes.c_int
    lib.msa_selftest_wait_timeout.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p]
    lib.msa_selftest_wait_timeout.restype = ctypes.c_int
    _lib = lib
    return lib


def status_string(status: int) -> str:
    return load_library().msa_status_string(status).decode()


def kernel_launches() -> int:
    """Kernel launches libmsa has enqueued in this process."""
    return int(load_library().msa_kernel_launches())


def describe(t: torch.Tensor) -> MsaTensor:
    """msa_tensor view of a [B, H, N, D] bf16 tensor (pointer, shape, element strides)."""
    if t.dim() != 4:
        raise ValueError("expected a [B, H, N, D] tensor")
    if t.dtype != torch.bfloat16:
        raise TypeError("expected bf16")
    if t.stride(3) != 1:
        raise ValueError("the head dimension must be contiguous")
    B, H, N, D = t.shape
    return MsaTensor(t.data_ptr(), B, H, N, D, t.stride(0), t.stride(1), t.stride(2))


def _stream_ptr(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream)


def workspace_bytes(kind: int, q: torch.Tensor, k: torch.Tensor, p0: int = 0, p1: int = 0,
                    n_heads: int = 0) -> int:
    lib = load_library()
    qt, kt = describe(q), describe(k)
    return int(lib.msa_workspace_bytes(kind, ctypes.byref(qt), ctypes.byref(kt), p0, p1, n_heads))


def selftest_wait_timeout(limit_us: int = 2000, stream=None, device=None) -> dict:
    """Runs the library's bounded-wait self-test (msa_selftest_wait_timeout) and
    reads its outcome: {"status": msa_device_status's code (MSA_ERR_TIMEOUT
    expected), "control_ok": the control wait succeeded, "waited_us": how long
    the abandoned wait lasted}."""
    lib = load_library()
    dev = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
    ws = torch.zeros(64, dtype=torch.int32, device=dev)  # 256 bytes; allocations are 256-byte aligned
    rc = int(lib.msa_selftest_wait_timeout(ctypes.c_void_p(ws.data_ptr()), int(limit_us),
                                           ctypes.c_void_p(_stream_ptr(stream))))
    if rc != MSA_OK:
        raise MsaError(rc, "msa_selftest_wait_timeout")
    status = device_status(ws, stream)  # synchronises the stream, then clears word 0 only
    words = ws[1:3].cpu()
    return {"status": status, "control_ok": bool(int(words[0]) == 1), "waited_us": int(words[1])}


def device_status(workspace: torch.Tensor, stream=None) -> int:
    return int(load_library().msa_device_status(ctypes.c_void_p(workspace.data_ptr()),
                                                ctypes.c_void_p(_stream_ptr(stream))))


class _Prepared:
    """Keeps every buffer a call touches alive until the call returns.

    Host inputs are copied to the current device on the call's stream; the
    device output is copied back into `out` (or a new pinned tensor).
    """

    def __init__(self, q, k, v, out, stream):
        self.host = q.device.type == "cpu"
        self.stream = stream
        self.host_out = None
        if self.host:
            dev = torch.device("cuda", torch.cuda.current_device())
            s = stream if stream is not None else torch.cuda.current_stream(dev)
            self.host_out = out
            with torch.cuda.stream(s):
                q, k, v = (t.to(dev, non_blocking=True) for t in (q, k, v))
                out = torch.zeros_like(q) if out is None else out.to(dev, non_blocking=True)
        elif out is None:
            out = torch.zeros_like(q)
        self.q, self.k, self.v, self.out = q, k, v, out

    def result(self):
        if not self.host:
            return self.out
        s = self.stream if self.stream is not None else torch.cuda.current_stream()
        if self.host_out is None:
            self.host_out = torch.empty(self.out.shape, dtype=self.out.dtype, pin_memory=True)
        with torch.cuda.stream(s):
            self.host_out.copy_(self.out, non_blocking=True)
        s.synchronize()
        return self.host_out


def _check_buffers(q, kind, p0, p1, heads, export, kv_select):
    """Every device buffer the library will write must hold what it writes
    (sizes from include/msa.h); a short buffer is refused here, before the call."""
    B, Hq, N, _ = q.shape
    NB = (N + 63) // 64
    U = B * (len(heads) if heads is not None else Hq)
    need = {}
    if kind == MSA_KIND_VERTICAL_SLASH:
        NQ = (N + 127) // 128
        chunk_words = ((min(p0, N) + 127) // 128 + 31) // 32
        need = {"v_score": U * N, "s_score": U * N, "vertical": U * min(p0, N),
                "slash": U * min(p1, N), "tile_dist": U * ((NB + 32) // 32),
                "col_count": U * NB, "col_chunks": U * NQ * chunk_words}
    elif kind in (MSA_KIND_BLOCK_SPARSE, MSA_KIND_HIERARCHICAL):
        need = {"block_count": U * NB, "block_ids": U * NB * min(p0, NB)}
    for name, t in (export or {}).items():
        if t is None:
            continue
        if name not in need:
            raise ValueError(f"export['{name}'] is not written by this call")
        if not t.is_cuda or t.numel() * t.element_size() < 4 * need[name]:
            raise ValueError(f"export['{name}'] must be a CUDA buffer of >= {need[name]} 4-byte entries")
    if kv_select is not None:
        kk = min(int(kv_select.get("keep_k", 0) or 0), N)
        for name, n in (("lse", B * Hq * N), ("score", B * Hq * N), ("keep", B * Hq * kk)):
            t = kv_select.get(name)
            if t is not None and (not t.is_cuda or not t.is_contiguous()
                                  or t.numel() * t.element_size() < 4 * n):
                raise ValueError(f"kv_select['{name}'] must be a contiguous CUDA buffer of >= {n} "
                                 "4-byte entries")


def _opts(q, k, kind, p0, p1, last_q, scale, heads, workspace, export, stage_events, stream,
          keep, kv_select=None):
    _check_buffers(q, kind, p0, p1, heads, export, kv_select)
    opts = MsaOpts()
    opts.stream = _stream_ptr(stream)
    opts.last_q = int(last_q)
    opts.scale = float(scale or 0.0)
    if heads is not None:
        arr = (ctypes.c_int32 * len(heads))(*[int(h) for h in heads])
        keep.append(arr)
        opts.heads = ctypes.cast(arr, ctypes.POINTER(ctypes.c_int32))
        opts.n_heads = len(heads)
    n_heads = len(heads) if heads is not None else 0
    if workspace is None and kind is not None:
        nbytes = workspace_bytes(kind, q, k, p0, p1, n_heads)
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
    if workspace is not None:
        keep.append(workspace)
        opts.workspace = workspace.data_ptr()
        opts.workspace_bytes = workspace.numel() * workspace.element_size()
    if export is not None:
        ex = MsaIndexExport(**{name: (t.data_ptr() if t is not None else None)
                               for name, t in export.items()})
        keep.append(ex)
        opts.export_idx = ctypes.pointer(ex)
    if stage_events is not None:
        arr = (ctypes.c_void_p * (2 * MSA_STAGE_COUNT))(*[ev.cuda_event for ev in stage_events])
        keep.append(arr)
        opts.stage_events = arr
    if kv_select is not None:
        def ptr(name):
            t = kv_select.get(name)
            if t is None:
                return None
            if not t.is_cuda:
                raise ValueError(f"kv_select['{name}'] must be a CUDA tensor (the kernels write it)")
            return t.data_ptr()
        kv = MsaKvSelect(ptr("lse"), ptr("score"), ptr("keep"), int(kv_select.get("window", 0)),
                         int(kv_select.get("keep_k", 0)))
        keep.append(kv)
        opts.kv_select = ctypes.pointer(kv)
    return opts, workspace


def _run(fn_name, kind, q, k, v, args, out, p0, p1, last_q, scale, heads, workspace, export,
         stage_events, stream, kv_select=None):
    lib = load_library()
    prep = _Prepared(q, k, v, out, stream)
    keep = []
    opts, ws = _opts(prep.q, prep.k, kind, p0, p1, last_q, scale, heads, workspace, export,
                     stage_events, stream, keep, kv_select)
    qt, kt, vt, ot = describe(prep.q), describe(prep.k), describe(prep.v), describe(prep.out)
    status = getattr(lib, fn_name)(ctypes.byref(qt), ctypes.byref(kt), ctypes.byref(vt), *args,
                                   ctypes.byref(ot), ctypes.byref(opts))
    if status != MSA_OK:
        raise MsaError(status, fn_name)
    if STRICT_STATUS:  # wait for the call and read (and clear) its device status word
        status = device_status(ws, stream)
        if status != MSA_OK:
            raise MsaError(status, f"{fn_name} (device status)")
    return prep.result()


def kv_select_buffers(q, window: int, keep_k: int = 0, score: bool = True):
    """Device buffers for the KV selection of a call on q [B,Hq,N,d]: lse and
    score f32 [B,Hq,N], keep int32 [B,Hq,min(keep_k,N)] (keep_k = 0: no keep set).
    Pass the returned dict as kv_select=."""
    B, Hq, N, _ = q.shape
    f = dict(dtype=torch.float32, device=q.device)
    out = {"lse": torch.zeros((B, Hq, N), **f), "score": None, "keep": None,
           "window": int(window), "keep_k": int(keep_k)}
    if score:
        out["score"] = torch.zeros((B, Hq, N), **f)
        if keep_k > 0:
            out["keep"] = torch.zeros((B, Hq, min(keep_k, N)), dtype=torch.int32, device=q.device)
    return out


def msa_vertical_slash(q, k, v, vertical_topk: int, slash: int, out=None, *, last_q: int = 64,
                       scale: Optional[float] = None, heads: Optional[Sequence[int]] = None,
                       workspace=None, export=None, stage_events=None, stream=None,
                       kv_select=None):
    """Vertical-slash sparse attention (MInference 1.0 overview, section 2.2).

    q [B,Hq,N,128], k/v [B,Hkv,N,128] bf16.  Writes the selected heads of `out`
    (allocated with zeros when None) and returns it.  kv_select (see
    kv_select_buffers) adds the row normalisers and the KV-selection score.
    """
    return _run("msa_vertical_slash", MSA_KIND_VERTICAL_SLASH, q, k, v,
                (ctypes.c_int64(vertical_topk), ctypes.c_int64(slash)), out, vertical_topk, slash,
                last_q, scale, heads, workspace, export, stage_events, stream, kv_select)


def msa_block_sparse(q, k, v, topk: int, out=None, *, scale: Optional[float] = None,
                     heads: Optional[Sequence[int]] = None, workspace=None, export=None,
                     stage_events=None, stream=None, kv_select=None):
    """Block-sparse attention (MInference 1.0 overview, section 2.2)."""
    return _run("msa_block_sparse", MSA_KIND_BLOCK_SPARSE, q, k, v, (ctypes.c_int64(topk),), out,
                topk, 0, 0, scale, heads, workspace, export, stage_events, stream, kv_select)


def hip_stages(stages):
    """ctypes array of msa_hip_stage from [(chunk_blocks, keep), ...]."""
    arr = (MsaHipStage * len(stages))()
    for i, (c, kp) in enumerate(stages):
        arr[i].chunk_blocks = int(c)
        arr[i].keep = int(kp)
    return arr


def msa_hierarchical(q, k, v, stages, out=None, *, scale: Optional[float] = None,
                     heads: Optional[Sequence[int]] = None, workspace=None, export=None,
                     stage_events=None, stream=None, kv_select=None):
    """Hierarchical multi-stage pruning head (InfiniteHiP summary page, modular
    hierarchical token pruning).  stages: [(chunk_blocks, keep), ...], chunk
    sizes in 64-token blocks, decreasing, each dividing the previous, the last 1."""
    arr = hip_stages(stages)
    keep_last = int(stages[-1][1]) if len(stages) else 0
    return _run("msa_hierarchical", MSA_KIND_HIERARCHICAL, q, k, v,
                (arr, ctypes.c_int32(len(stages))), out, keep_last, 0, 0, scale, heads, workspace,
                export, stage_events, stream, kv_select)


def msa_streaming(q, k, v, init_num: int, local_window_num: int, out=None, *,
                  scale: Optional[float] = None, heads: Optional[Sequence[int]] = None,
                  workspace=None, stage_events=None, stream=None, kv_select=None):
    """Streaming / A-shape attention (MInference 1.0 overview, kernel listing)."""
    return _run("msa_streaming", MSA_KIND_STREAMING, q, k, v,
                (ctypes.c_int64(init_num), ctypes.c_int64(local_window_num)), out, 0, 0, 0, scale,
                heads, workspace, None, stage_events, stream, kv_select)


def mass_recall(lse, ref_lse, recall=None, *, row0: int = 0, heads: Optional[Sequence[int]] = None,
                stream=None):
    """Mean kept dense-attention mass per head over rows [row0, N) (MInference 1.0
    overview, section 2.1): lse / ref_lse are f32 [B,Hq,N] normalisers of a sparse
    and a dense call; writes the selected heads of recall f32 [B,Hq]."""
    lib = load_library()
    B, Hq, N = lse.shape
    for name, t in (("lse", lse), ("ref_lse", ref_lse)):
        if not (t.is_cuda and t.dtype == torch.float32 and t.is_contiguous() and t.shape == lse.shape):
            raise ValueError(f"{name} must be a contiguous CUDA float32 tensor of shape {tuple(lse.shape)}")
    if recall is None:
        recall = torch.zeros((B, Hq), dtype=torch.float32, device=lse.device)
    if not (recall.is_cuda and recall.dtype == torch.float32 and recall.is_contiguous()
            and tuple(recall.shape) == (B, Hq)):
        raise ValueError("recall must be a contiguous CUDA float32 tensor [B, Hq]")
    arr, n = None, 0
    if heads is not None:
        arr = (ctypes.c_int32 * len(heads))(*[int(h) for h in heads])
        n = len(heads)
    status = lib.msa_mass_recall(lse.data_ptr(), ref_lse.data_ptr(), B, Hq, N, int(row0),
                                 ctypes.cast(arr, ctypes.POINTER(ctypes.c_int32)) if arr else None,
                                 n, recall.data_ptr(), _stream_ptr(stream))
    if status != MSA_OK:
        raise MsaError(status, "msa_mass_recall")
    return recall
