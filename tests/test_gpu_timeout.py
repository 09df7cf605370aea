"""Failure detection on the GPU without a fault: the tensor-core kernels'
bounded waits (global-timer deadline) end in SKV_ERR_TIMEOUT, read by the
host, and leave the context usable."""
import pytest

import lse_merge_gb300 as skv
from gpu_helpers import TOL_BF16, TOL_BF16_LSE, dev_inputs
from test_gpu_attn import check_forward
from workloads import random_small

pytestmark = pytest.mark.gpu


def test_bounded_wait_timeout_reports_status():
    # A 1 ns limit makes the tensor-core kernel's waits run out: it must
    # record SKV_ERR_TIMEOUT and finish (no hang, no fault), and the context
    # stays usable for a normal run afterwards.
    w = random_small(31, 1, 1024, 8, 16, 1, 128, 256, 4, "bf16", order="contiguous")
    inp, d, prob = dev_inputs(w)
    _, roc, _, _ = skv.plan(prob, "contiguous")
    try:
        skv.set_wait_limit(1)
        skv.attn_fwd(prob, d["q"], d["k"], d["v"], roc)
        assert skv.stream_status() == 4          # SKV_ERR_TIMEOUT
    finally:
        skv.set_wait_limit(0)
    check_forward(w, TOL_BF16, TOL_BF16_LSE)
