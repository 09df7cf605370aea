"""skv_attn_fwd_static: the forward partials for callers that may not allocate
device memory (a plug-in inside a framework that owns the device memory pool,
a loop that cannot pay for cudaMalloc's device synchronisation).  Its scratch
is a fixed array inside the library.

The test calls it through the C ABI several times in a row on different
problems and checks each result against the CPU oracle (bf16 tolerances) and
bit for bit against the regular workspace entry point, which runs the same
kernels on the same inputs: stale scratch left by the previous call would show
as a difference.  One problem gives a rank more chunks than the forward keeps
in shared memory, so the kernel reads its chunk list from the static array
itself.  Device memory must not change across a (warm) call.  Collected last
on purpose; it needs no state from other tests."""
import ctypes

import numpy as np
import pytest
import torch

import lse_merge_gb300 as skv
import oracle as orc
from lse_merge_gb300 import _lib
from gpu_helpers import TOL_BF16, TOL_BF16_LSE, assert_lse_equal, dev_inputs, maxabs
from workloads import random_small

pytestmark = pytest.mark.gpu

CASES = [
    random_small(41, 2, 1024, 8, 16, 2, 128, 256, 8, "bf16", order="lpt"),
    random_small(42, 3, 768, 6, 16, 1, 64, 128, 6, "bf16", order="contiguous"),
    # one rank holding 130 chunks of 128 keys: more than the 64 chunk indices the
    # forward stages in shared memory
    random_small(43, 1, 130 * 128, 8, 16, 1, 128, 128, 1, "bf16", order="contiguous"),
]


def _static_call(prob, d, roc, o_part, lse_part):
    st = _lib.load().skv_attn_fwd_static(ctypes.byref(prob.c), d["q"].data_ptr(), d["k"].data_ptr(),
                                         d["v"].data_ptr(), roc.data_ptr(), o_part.data_ptr(), lse_part.data_ptr(),
                                         ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, st


def _bit_equal(ref, got):
    r_op, r_lp = (x.cpu().numpy() for x in ref)
    g_op, g_lp = (x.cpu().numpy() for x in got)
    assert np.array_equal(r_lp, g_lp)                    # -inf where a partial is empty, on both sides
    fin = np.isfinite(r_lp)
    assert np.array_equal(r_op[fin], g_op[fin])


def _vs_oracle(w, inp, roc, got):
    r_op, r_lp = orc.partition_forward(inp.q, inp.k, inp.v, inp.s, inp.a, w.B, roc.cpu().numpy(), w.m, w.P)
    g_op, g_lp = (x.cpu().numpy() for x in got)
    assert_lse_equal(g_lp, r_lp, TOL_BF16_LSE)
    fin = np.isfinite(r_lp)
    err = maxabs(g_op, r_op, np.broadcast_to(fin[..., None], r_op.shape))
    assert err <= TOL_BF16, f"o_part err {err}"


def test_static_scratch_forward_matches_oracle_and_workspace_forward():
    runs = []
    for w in CASES:
        inp, d, prob = dev_inputs(w, with_grad=False)
        _, roc, _, _ = skv.plan(prob, w.order)
        ref = skv.attn_fwd(prob, d["q"], d["k"], d["v"], roc)
        o_part = torch.full((w.P, w.Q, w.H, w.d), float("nan"), device="cuda")
        lse_part = torch.full((w.P, w.Q, w.H), float("nan"), device="cuda")
        runs.append((w, inp, d, prob, roc, ref, o_part, lse_part))
    torch.cuda.synchronize()
    # the calls follow each other on one stream with nothing between them
    for w, inp, d, prob, roc, ref, o_part, lse_part in runs:
        _static_call(prob, d, roc, o_part, lse_part)
    assert skv.stream_status() == 0
    for w, inp, d, prob, roc, ref, o_part, lse_part in runs:
        _bit_equal(ref, (o_part, lse_part))
        _vs_oracle(w, inp, roc, (o_part, lse_part))


def test_static_scratch_call_allocates_nothing():
    w = CASES[0]
    inp, d, prob = dev_inputs(w, with_grad=False)
    _, roc, _, _ = skv.plan(prob, w.order)
    o_part = torch.empty(w.P, w.Q, w.H, w.d, device="cuda")
    lse_part = torch.empty(w.P, w.Q, w.H, device="cuda")
    skv.attn_fwd_static(prob, d["q"], d["k"], d["v"], roc, o_part, lse_part)   # through the binding; loads the module
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    reserved0 = torch.cuda.memory_reserved()
    _static_call(prob, d, roc, o_part, lse_part)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0
    assert torch.cuda.memory_reserved() == reserved0
    assert skv.stream_status() == 0
    _vs_oracle(w, inp, roc, (o_part, lse_part))


def test_static_scratch_rejects_oversized_plans():
    # 32768 chunks need more chunk-list scratch than the fixed array holds.  Every
    # buffer is real and sized for the problem, so even a call that got past the
    # size check would stay inside its buffers.
    P, J, m, H, D = 1024, 32, 128, 1, 64
    S = P * J * m
    s = torch.zeros(1, dtype=torch.int32, device="cuda")
    a = torch.full((1,), 128, dtype=torch.int32, device="cuda")
    prob = skv.Problem(s, a, 16, H, D, S, m, P, torch.bfloat16)
    assert skv.workspace_bytes(prob, 0) > 131072
    q = torch.zeros(16, H, D, dtype=torch.bfloat16, device="cuda")
    k = torch.zeros(S, H, D, dtype=torch.bfloat16, device="cuda")
    v = torch.zeros(S, H, D, dtype=torch.bfloat16, device="cuda")
    roc = (torch.arange(P * J, dtype=torch.int32, device="cuda") // J).contiguous()
    o_part = torch.empty(P, 16, H, D, device="cuda")
    lse_part = torch.empty(P, 16, H, device="cuda")
    st = _lib.load().skv_attn_fwd_static(ctypes.byref(prob.c), q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                         roc.data_ptr(), o_part.data_ptr(), lse_part.data_ptr(),
                                         ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == _lib.SKV_ERR_WORKSPACE
    assert skv.stream_status() == 0
