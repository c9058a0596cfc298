"""The host pipeline (pipeline.run_pipelined) gives, for every batch, exactly
the output of one synchronous call: double buffering and the side-stream
copies reorder nothing that matters.  The kernels are deterministic, so the
comparison is bit-exact."""
import pytest
import torch

from dynamic_sparse_attention_slash_gb300 import inputs, msa
from dynamic_sparse_attention_slash_gb300.pipeline import run_pipelined

pytestmark = pytest.mark.gpu


def test_pipelined_outputs_equal_one_call_per_batch():
    N, n_batches = 1088, 5
    batches = []
    for i in range(n_batches):
        q, k, v = inputs.make_qkv(1, 4, 2, N, 50 + i, vs_planting=True, device="cpu")
        batches.append(tuple(t.pin_memory() for t in (q, k, v)))
    outs = [torch.empty_like(batches[0][0]).pin_memory() for _ in range(2)]
    out_seq = [outs[i % 2] for i in range(n_batches)]

    def step(q, k, v, out):
        msa.msa_vertical_slash(q, k, v, 100, 120, out, heads=[0, 2])
        msa.msa_streaming(q, k, v, 1, 3, out, heads=[1, 3])

    ref = []
    for qh, kh, vh in batches:
        out = torch.zeros(qh.shape, dtype=qh.dtype, device="cuda")
        step(qh.cuda(), kh.cuda(), vh.cuda(), out)
        ref.append(out.cpu())
    # outputs alternate between two host buffers: check each batch right after
    # its own copy, before the buffer is reused two batches later
    for i in range(n_batches):
        evs = run_pipelined(step, batches[: i + 1], out_seq[: i + 1])
        evs["end"].synchronize()
        assert torch.equal(out_seq[i], ref[i]), f"batch {i}"
