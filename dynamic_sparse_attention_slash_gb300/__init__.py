"""MInference-style dynamic sparse prefill attention for one GB300 GPU.

Public API (all computation runs in the CUDA kernels of libmsa.so):

    msa_vertical_slash(q, k, v, vertical_topk, slash, out=None, ...)
    msa_block_sparse(q, k, v, topk, out=None, ...)
    msa_streaming(q, k, v, init_num, local_window_num, out=None, ...)
"""
from .msa import (  # noqa: F401
    MsaError,
    device_status,
    kernel_launches,
    load_library,
    msa_block_sparse,
    msa_streaming,
    msa_vertical_slash,
    workspace_bytes,
)
