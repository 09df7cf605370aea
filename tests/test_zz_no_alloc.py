"""skv_attn_fwd_static: the forward partials for callers that may not allocate
device memory (a plug-in inside a framework that owns the device memory pool,
a loop that cannot pay for cudaMalloc's device synchronisation).  Its scratch
is a fixed array inside the library; this test calls it through the C ABI
twice in a row, on two different problems, and compares each result with the
regular workspace entry point (skv_attn_fwd) at the bf16 parity tolerances.
Collected last on purpose; it needs no state from other tests."""
import ctypes

import numpy as np
import pytest
import torch

import lse_merge_gb300 as skv
from lse_merge_gb300 import _lib
from gpu_helpers import TOL_BF16, TOL_BF16_LSE, dev_inputs, maxabs
from workloads import random_small

pytestmark = pytest.mark.gpu


def _static_call(prob, d, roc, P, Q, H, D):
    o_part = torch.full((P, Q, H, D), float("nan"), device="cuda")
    lse_part = torch.full((P, Q, H), float("nan"), device="cuda")
    st = _lib.load().skv_attn_fwd_static(ctypes.byref(prob.c), d["q"].data_ptr(), d["k"].data_ptr(),
                                         d["v"].data_ptr(), roc.data_ptr(), o_part.data_ptr(), lse_part.data_ptr(),
                                         ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, st
    return o_part, lse_part


def _compare(ref, got):
    r_op, r_lp = (x.cpu().numpy() for x in ref)
    g_op, g_lp = (x.cpu().numpy() for x in got)
    assert np.array_equal(np.isneginf(r_lp), np.isneginf(g_lp))
    fin = np.isfinite(r_lp)
    assert maxabs(g_lp, r_lp, fin) <= TOL_BF16_LSE
    assert maxabs(g_op, r_op, np.broadcast_to(fin[..., None], r_op.shape)) <= TOL_BF16


def test_static_scratch_forward_matches_workspace_forward_twice():
    cases = [random_small(41, 2, 1024, 8, 16, 2, 128, 256, 8, "bf16", order="lpt"),
             random_small(42, 3, 768, 6, 16, 1, 64, 128, 6, "bf16", order="contiguous")]
    for w in cases:
        inp, d, prob = dev_inputs(w, with_grad=False)
        _, roc, _, _ = skv.plan(prob, w.order)
        ref = skv.attn_fwd(prob, d["q"], d["k"], d["v"], roc)
        got = _static_call(prob, d, roc, w.P, w.Q, w.H, w.d)
        assert skv.stream_status() == 0
        _compare(ref, got)


def test_static_scratch_rejects_oversized_plans():
    # 32768 chunks need more chunk-list scratch than the fixed array holds
    s = torch.zeros(1, dtype=torch.int32, device="cuda")
    a = torch.full((1,), 128, dtype=torch.int32, device="cuda")
    prob = skv.Problem(s, a, 16, 1, 64, 32768 * 128, 128, 1024, torch.bfloat16)
    st = _lib.load().skv_attn_fwd_static(ctypes.byref(prob.c), 0x100, 0x100, 0x100, 0x100, 0x100, 0x100, None)
    assert st == _lib.SKV_ERR_WORKSPACE
