"""Failure detection on the GPU without a GPU fault.

Every kernel of the library waits on mbarriers with a bounded wait: past its
limit the wait gives up, the CTA drains and exits, and the call's status word
gets the timeout bit, which msa_device_status reports as MSA_ERR_TIMEOUT.  The
self-test entry point runs that wait on a barrier nothing arrives at (the flag
that nothing sets) beside a control barrier that completes; the host must read
MSA_ERR_TIMEOUT, and the context must stay usable for ordinary calls.
"""
import math

import pytest
import torch

from oracle import msa_oracle as O
from dynamic_sparse_attention_slash_gb300 import inputs, msa
from tests import parity as P

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("limit_us", [1000, 20000])
def test_abandoned_wait_reports_timeout_and_context_stays_usable(limit_us):
    r = msa.selftest_wait_timeout(limit_us)
    assert r["status"] == msa.MSA_ERR_TIMEOUT, msa.status_string(r["status"])
    assert r["control_ok"], "a barrier whose arrivals all came must not time out"
    # the wait lasted at least its limit and gave up soon after it (the limit
    # is checked every 64 polls of the barrier)
    assert limit_us <= r["waited_us"] < limit_us + 50000, r
    # the status word was cleared by reading it, and ordinary work still runs
    N = 640
    q, k, v = inputs.make_qkv(1, 2, 1, N, 77, device="cpu")
    ws = torch.empty(msa.workspace_bytes(2, q, k, 1, 3), dtype=torch.uint8, device="cuda")
    out = msa.msa_streaming(q.cuda(), k.cuda(), v.cuda(), 1, 3, workspace=ws)
    assert msa.device_status(ws) == msa.MSA_OK
    ref, _ = O.streaming_forward(q, k, v, 1, 3)
    P.compare_out(P.to_np(out[0]), ref[0], "after the self-test")
