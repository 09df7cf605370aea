"""Degenerate shapes of the attention path on the GPU, against the CPU fp64
oracle: no query block at all, a single rank (P = 1: one partial, the merge an
identity), one chunk per rank (J = 1), and a single anchor block of one row."""
import numpy as np
import pytest
import torch

import lse_merge_gb300 as skv
from gpu_helpers import TOL_BF16, TOL_BF16_LSE, TOL_FP32
from test_gpu_attn import check_backward, check_forward
from workloads import random_small

pytestmark = pytest.mark.gpu


def test_no_query_blocks():
    # N = 0: the calls succeed without a launch; dk, dv are all zero
    S, H, d, m, P = 1024, 2, 64, 256, 2
    s = torch.empty(0, dtype=torch.int32, device="cuda")
    a = torch.empty(0, dtype=torch.int32, device="cuda")
    prob = skv.Problem(s, a, 16, H, d, S, m, P, torch.bfloat16)
    q = torch.empty(0, H, d, dtype=torch.bfloat16, device="cuda")
    k = torch.randn(S, H, d, device="cuda").to(torch.bfloat16)
    v = torch.randn(S, H, d, device="cuda").to(torch.bfloat16)
    costs, roc, _, _ = skv.plan(prob, "lpt")
    assert int(costs.abs().sum()) == 0
    o_part, lse_part = skv.attn_fwd(prob, q, k, v, roc)
    o, lse = skv.lse_merge(o_part, lse_part, out_dtype=torch.bfloat16)
    dk = torch.full((S, H, d), 7.0, device="cuda")
    dv = torch.full((S, H, d), 7.0, device="cuda")
    dq, dk, dv = skv.attn_bwd(prob, q, k, v, o, lse, q, roc, dk=dk, dv=dv)
    assert skv.stream_status() == 0
    assert dq.numel() == 0 and o.numel() == 0
    assert float(dk.abs().max()) == 0.0 and float(dv.abs().max()) == 0.0


@pytest.mark.parametrize("cfg", [
    # (seed, samples, L, anchors/sample, B, H, d, m, P, dtype, order)
    (51, 2, 1024, 6, 16, 2, 128, 256, 1, "bf16", "lpt"),         # one rank: the merge is an identity
    (52, 1, 768, 5, 16, 2, 64, 128, 1, "fp32", "contiguous"),    # the same on the CUDA-core path
    (53, 2, 1024, 6, 16, 2, 128, 128, 16, "bf16", "lpt"),        # J = 1: every rank holds one chunk
    (54, 1, 512, 1, 1, 1, 128, 128, 4, "bf16", "contiguous"),    # one block of one row
])
def test_degenerate_shapes(cfg):
    seed, b, L, A, B, H, dd, m, P, dt, order = cfg
    w = random_small(seed, b, L, A, B, H, dd, m, P, dt, order=order)
    assert w.S // w.m == w.P * w.J
    tol = TOL_FP32 if dt == "fp32" else TOL_BF16
    tol_l = TOL_FP32 if dt == "fp32" else TOL_BF16_LSE
    inp, d, prob, roc, o, lse = check_forward(w, tol, tol_l, order=order)
    check_backward(w, inp, d, prob, roc, o, lse, tol)
