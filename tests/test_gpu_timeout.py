"""Failure detection on the GPU without a fault: the tensor-core kernels'
bounded waits (global-timer deadline) end in SKV_ERR_TIMEOUT, read by the
host, and leave the context usable.  The test mode of skv_set_wait_limit
(negative limit) makes every block wait on a barrier that nothing completes."""
import pytest
import torch

import lse_merge_gb300 as skv
from gpu_helpers import TOL_BF16, TOL_BF16_LSE, dev_inputs
from test_gpu_attn import check_backward, check_forward
from workloads import random_small

pytestmark = pytest.mark.gpu


def test_bounded_wait_timeout_reports_status():
    w = random_small(31, 1, 1024, 8, 16, 1, 128, 256, 4, "bf16", order="contiguous")
    inp, d, prob = dev_inputs(w)
    _, roc, _, _ = skv.plan(prob, "contiguous")
    o = torch.zeros(w.Q, w.H, w.d, dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros(w.Q, w.H, device="cuda")
    try:
        skv.set_wait_limit(-50_000_000)              # 50 ms deadline, stuck barrier first
        skv.attn_fwd(prob, d["q"], d["k"], d["v"], roc)
        assert skv.stream_status() == 4          # SKV_ERR_TIMEOUT, read and cleared
        skv.attn_bwd(prob, d["q"], d["k"], d["v"], o, lse, d["dO"], roc)
        assert skv.stream_status() == 4
    finally:
        skv.set_wait_limit(0)
    # the context is still usable and the normal path is unaffected
    inp, d, prob, roc, o, lse = check_forward(w, TOL_BF16, TOL_BF16_LSE)
    check_backward(w, inp, d, prob, roc, o, lse, TOL_BF16)
