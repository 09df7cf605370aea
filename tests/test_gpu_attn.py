"""GPU parity of the attention path (per-rank partials, LSE merge, backward)
against the CPU fp64 oracle on the same seeded inputs.

Element-by-element at sizes the oracle finishes in seconds (several tiles and
ragged tails); the tiny fp32 workload at 1e-4, bf16 workloads at 2e-2 (o, dq,
dk, dv) and 1e-3 (lse)."""
import math

import numpy as np
import pytest
import torch

import lse_merge_gb300 as skv
import oracle as orc
from gpu_helpers import TOL_BF16, TOL_BF16_LSE, TOL_FP32, assert_lse_equal, dev_inputs, maxabs
from workloads import BF16_FWD, TINY_FP32, random_small

pytestmark = pytest.mark.gpu


def run_forward(w, d, prob, order):
    costs, roc, _, _ = skv.plan(prob, order)
    o_part, lse_part = skv.attn_fwd(prob, d["q"], d["k"], d["v"], roc)
    o, lse = skv.lse_merge(o_part, lse_part, out_dtype=d["q"].dtype)
    return roc, o_part, lse_part, o, lse


def check_forward(w, tol, tol_lse, order="contiguous", check_parts=True):
    inp, d, prob = dev_inputs(w)
    roc, o_part, lse_part, o, lse = run_forward(w, d, prob, order)
    assert skv.stream_status() == 0
    roc_c = roc.cpu().numpy()
    if check_parts:
        r_op, r_lp = orc.partition_forward(inp.q, inp.k, inp.v, inp.s, inp.a, w.B, roc_c, w.m, w.P)
        g_lp = lse_part.cpu().numpy()
        assert_lse_equal(g_lp, r_lp, tol_lse)
        fin = np.isfinite(r_lp)
        err = maxabs(o_part.cpu().numpy(), r_op, np.broadcast_to(fin[..., None], r_op.shape))
        assert err <= tol, f"o_part err {err}"
    r_o, r_l = orc.attention_forward(inp.q, inp.k, inp.v, inp.s, inp.a, w.B)
    assert_lse_equal(lse.cpu().numpy(), r_l, tol_lse)
    err = maxabs(o.float().cpu().numpy(), r_o)
    assert err <= tol, f"o err {err}"
    return inp, d, prob, roc, o, lse


def check_backward(w, inp, d, prob, roc, o, lse, tol):
    dq, dk, dv = skv.attn_bwd(prob, d["q"], d["k"], d["v"], o, lse, d["dO"], roc)
    assert skv.stream_status() == 0
    r_dq, r_dk, r_dv = orc.attention_backward(inp.q, inp.k, inp.v, inp.s, inp.a, w.B, inp.dO)
    for name, g, r in (("dq", dq, r_dq), ("dk", dk, r_dk), ("dv", dv, r_dv)):
        err = maxabs(g.cpu().numpy(), r)
        assert err <= tol, f"{name} err {err}"


def test_tiny_fp32_forward_merge_backward():
    inp, d, prob, roc, o, lse = check_forward(TINY_FP32, TOL_FP32, TOL_FP32)
    check_backward(TINY_FP32, inp, d, prob, roc, o, lse, TOL_FP32)


@pytest.mark.parametrize("cfg", [
    # (seed, samples, L, anchors/sample, B, H, d, m, P, dtype, order)
    (11, 2, 1024, 5, 16, 2, 64, 256, 4, "fp32", "lpt"),
    (12, 3, 768, 7, 5, 1, 128, 128, 6, "fp32", "contiguous"),   # ragged B, 3 samples
    (13, 1, 1408, 9, 16, 2, 128, 128, 11, "bf16", "lpt"),       # odd P
    (14, 4, 512, 3, 24, 3, 64, 256, 2, "bf16", "contiguous"),   # B > 16 rows
    (15, 2, 640, 6, 16, 2, 128, 640, 2, "bf16", "lpt"),          # m not a power of two
])
def test_small_workloads(cfg):
    seed, b, L, A, B, H, dd, m, P, dt, order = cfg
    w = random_small(seed, b, L, A, B, H, dd, m, P, dt, order=order)
    tol = TOL_FP32 if dt == "fp32" else TOL_BF16
    tol_l = TOL_FP32 if dt == "fp32" else TOL_BF16_LSE
    inp, d, prob, roc, o, lse = check_forward(w, tol, tol_l, order=order)
    check_backward(w, inp, d, prob, roc, o, lse, tol)


def test_empty_windows_and_partitions():
    # anchors at the sample start (empty windows) and a rank that sees nothing
    w = random_small(21, 2, 1024, 4, 16, 2, 64, 128, 8, "fp32", anchor_lo=0, anchor_hi=300)
    inp, d, prob = dev_inputs(w)
    s = torch.tensor([0, 0, 0, 0, 1024, 1024, 1024, 1024], dtype=torch.int32)
    a = torch.tensor([0, 1, 130, 300, 1024, 1030, 1100, 1300], dtype=torch.int32)
    inp.s, inp.a = s, a
    d["s"].copy_(s)
    d["a"].copy_(a)
    roc, o_part, lse_part, o, lse = run_forward(w, d, prob, "contiguous")
    r_o, r_l = orc.attention_forward(inp.q, inp.k, inp.v, s, a, w.B)
    assert_lse_equal(lse.cpu().numpy(), r_l, TOL_FP32)
    assert np.all(o[:16].cpu().numpy() == 0)     # block 0 sees no key: o = 0, lse = -inf
    assert maxabs(o.cpu().numpy(), r_o) <= TOL_FP32
    r_op, r_lp = orc.partition_forward(inp.q, inp.k, inp.v, s, a, w.B, roc.cpu().numpy(), w.m, w.P)
    assert_lse_equal(lse_part.cpu().numpy(), r_lp, TOL_FP32)
    check_backward(w, inp, d, prob, roc, o, lse, TOL_FP32)


def test_bf16_fwd_workload_full():
    check_forward(BF16_FWD, TOL_BF16, TOL_BF16_LSE, order="contiguous", check_parts=False)


def test_merge_random_partials():
    g = torch.Generator().manual_seed(3)
    for P, rows, dd in ((1, 7, 64), (5, 1000, 128), (33, 333, 64), (64, 100, 128), (3, 50, 32)):
        o_part = torch.randn(P, rows, dd, generator=g)
        lse_part = torch.randn(P, rows, generator=g) * 5
        drop = torch.rand(P, rows, generator=g) < 0.4
        lse_part[drop] = -math.inf
        lse_part[:, :3] = -math.inf                      # all-empty rows
        o_part[drop] = float("nan")                      # unspecified rows must not be read
        r_o, r_l = orc.lse_merge(np.where(drop[..., None].numpy(), 0.0, o_part.double().numpy()),
                                 lse_part.double().numpy())
        for dt, tol in ((torch.float32, 1e-5), (torch.bfloat16, 2e-2)):
            o, lse = skv.lse_merge(o_part.cuda(), lse_part.cuda(), out_dtype=dt)
            assert_lse_equal(lse.cpu().numpy(), r_l, 1e-5)
            got = o.float().cpu().numpy()
            assert np.all(np.isfinite(got))
            assert np.all(got[:3] == 0)
            assert maxabs(got, r_o) <= tol * max(1.0, float(np.abs(r_o).max()))

