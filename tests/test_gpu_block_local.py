"""GPU parity of the block-local term of the anchor mask (each block's rows over
the block's own B keys) and of the whole mask it completes, against the CPU
fp64 oracle on the same seeded inputs [Split-KV §3.1 Fig. 1; Eq. 4].

Small workloads element by element (fp32 1e-4; bf16 2e-2 on o, dq, dk, dv and
1e-3 on lse); the full packed workload on sampled heads and blocks."""
import numpy as np
import pytest
import torch

import lse_merge_gb300 as skv
import oracle as orc
from gpu_helpers import TOL_BF16, TOL_BF16_LSE, TOL_FP32, assert_lse_equal, dev_inputs, maxabs
from workloads import PACKED, TINY_FP32, block_kv, make_inputs, random_small

pytestmark = pytest.mark.gpu


def whole_mask_forward(w, d, prob, kb, vb, order="contiguous"):
    """P rank partials + the block-local partial in slot P, merged (P + 1)."""
    _, roc, _, _ = skv.plan(prob, order)
    o_part = torch.empty(w.P + 1, w.Q, w.H, w.d, device="cuda")
    lse_part = torch.empty(w.P + 1, w.Q, w.H, device="cuda")
    skv.attn_fwd(prob, d["q"], d["k"], d["v"], roc, o_part[:w.P], lse_part[:w.P])
    skv.block_local_fwd(prob, d["q"], kb, vb, o_part[w.P], lse_part[w.P])
    o, lse = skv.lse_merge(o_part, lse_part, out_dtype=d["q"].dtype)
    return roc, o_part, lse_part, o, lse


@pytest.mark.parametrize("w,tol,tol_l", [
    (TINY_FP32, TOL_FP32, TOL_FP32),
    (random_small(31, 2, 1024, 24, 16, 4, 128, 256, 4, dtype="bf16"), TOL_BF16, TOL_BF16_LSE),
    (random_small(32, 1, 768, 10, 7, 2, 64, 256, 3, dtype="fp32"), TOL_FP32, TOL_FP32),
])
def test_block_local_forward(w, tol, tol_l):
    inp, d, prob = dev_inputs(w, with_grad=False)
    kb, vb = block_kv(w)
    o, lse = skv.block_local_fwd(prob, d["q"], kb.cuda(), vb.cuda())
    assert skv.stream_status() == 0
    r_o, r_l = orc.block_local_forward(inp.q, kb, vb, w.B)
    assert_lse_equal(lse.cpu().numpy(), r_l, tol_l)
    assert maxabs(o.cpu().numpy(), r_o) <= tol


def test_block_local_single_token_is_v():
    w = random_small(33, 1, 512, 40, 1, 2, 64, 128, 4, dtype="bf16")
    inp, d, prob = dev_inputs(w, with_grad=False)
    kb, vb = block_kv(w)
    o, _ = skv.block_local_fwd(prob, d["q"], kb.cuda(), vb.cuda())
    assert skv.stream_status() == 0
    assert maxabs(o.cpu().numpy(), vb.float().numpy()) <= 1e-6


@pytest.mark.parametrize("w,tol,tol_l", [
    (TINY_FP32, TOL_FP32, TOL_FP32),
    (random_small(34, 2, 1536, 20, 16, 3, 128, 256, 6, dtype="bf16"), TOL_BF16, TOL_BF16_LSE),
    # B past 16 (eight rows a warp, one lane a key): the largest block, and a ragged one
    (random_small(35, 1, 1024, 12, 32, 3, 128, 256, 4, dtype="bf16"), TOL_BF16, TOL_BF16_LSE),
    (random_small(36, 1, 1024, 9, 32, 2, 128, 256, 4, dtype="fp32"), TOL_FP32, TOL_FP32),
    (random_small(37, 1, 1024, 10, 17, 2, 64, 256, 4, dtype="bf16"), TOL_BF16, TOL_BF16_LSE),
])
def test_whole_mask_forward_and_backward(w, tol, tol_l):
    inp, d, prob = dev_inputs(w, with_grad=True)
    kb, vb = block_kv(w)
    kbd, vbd = kb.cuda(), vb.cuda()
    roc, _, _, o, lse = whole_mask_forward(w, d, prob, kbd, vbd)
    r_o, r_l = orc.full_mask_forward(inp.q, inp.k, inp.v, kb, vb, inp.s, inp.a, w.B)
    assert_lse_equal(lse.cpu().numpy(), r_l, tol_l)
    assert maxabs(o.float().cpu().numpy(), r_o) <= tol
    dq, dk, dv = skv.attn_bwd(prob, d["q"], d["k"], d["v"], o, lse, d["dO"], roc)
    dq, dkb, dvb = skv.block_local_bwd(prob, d["q"], kbd, vbd, o, lse, d["dO"], dq)
    assert skv.stream_status() == 0
    r_dq, r_dk, r_dv = orc.context_backward_given(inp.q, inp.k, inp.v, inp.s, inp.a, w.B, inp.dO, r_o, r_l)
    r_dqb, r_dkb, r_dvb = orc.block_local_backward(inp.q, kb, vb, inp.dO, r_o, r_l, w.B)
    for name, g, r in (("dq", dq, r_dq + r_dqb), ("dk", dk, r_dk), ("dv", dv, r_dv),
                       ("dk_blk", dkb, r_dkb), ("dv_blk", dvb, r_dvb)):
        err = maxabs(g.cpu().numpy(), r)
        assert err <= tol, f"{name} err {err}"


def test_block_local_packed_sampled():
    """Full packed workload (b=4 x 128k, Q=32768, H=32, d=128, bf16): the block-local
    partial on two heads at every row; the whole-mask gradients of the block-local
    term on sampled blocks, against the oracle's full-mask o and lse of those rows."""
    w = PACKED
    inp = make_inputs(w, with_grad=True, device="cuda")
    prob = skv.Problem(inp.s.cuda(), inp.a.cuda(), w.B, w.H, w.d, w.S, w.m, w.P, torch.bfloat16)
    d = {"q": inp.q, "k": inp.k, "v": inp.v, "dO": inp.dO}
    kb, vb = block_kv(w, device="cuda")
    o_l, lse_l = skv.block_local_fwd(prob, d["q"], kb, vb)
    heads = [0, w.H - 1]
    r_o, r_l = orc.block_local_forward(d["q"][:, heads].cpu(), kb[:, heads].cpu(), vb[:, heads].cpu(), w.B)
    assert_lse_equal(lse_l[:, heads].cpu().numpy(), r_l, TOL_BF16_LSE)
    assert maxabs(o_l[:, heads].cpu().numpy(), r_o) <= TOL_BF16
    # whole mask on the GPU, then only the block-local backward (dq starts at zero)
    _, _, _, o, lse = whole_mask_forward(w, d, prob, kb, vb, order=w.order)
    dq0 = torch.zeros(w.Q, w.H, w.d, device="cuda")
    dqb, dkb, dvb = skv.block_local_bwd(prob, d["q"], kb, vb, o, lse, d["dO"], dq0)
    assert skv.stream_status() == 0
    blocks = [0, 777, 1500, w.N - 1]
    h = 5
    one = lambda t: t[:, h:h + 1].cpu()          # the sampled head, on the host
    f_o, f_l = orc.full_mask_forward(one(d["q"]), one(d["k"]), one(d["v"]), one(kb), one(vb),
                                     inp.s, inp.a, w.B, blocks=blocks)
    rows = np.concatenate([np.arange(i * w.B, (i + 1) * w.B) for i in blocks])
    assert maxabs(o[:, h:h + 1].float().cpu().numpy()[rows], f_o[rows]) <= TOL_BF16
    r_dq, r_dk, r_dv = orc.block_local_backward(one(d["q"])[rows], one(kb)[rows], one(vb)[rows],
                                                one(d["dO"])[rows], f_o[rows], f_l[rows], w.B)
    for name, g, r in (("dq_local", dqb, r_dq), ("dk_blk", dkb, r_dk), ("dv_blk", dvb, r_dv)):
        err = maxabs(one(g).numpy()[rows], r)
        assert err <= TOL_BF16, f"{name} err {err}"


def test_block_local_rejects_large_blocks():
    w = random_small(35, 1, 512, 4, 64, 1, 64, 128, 4)
    inp, d, prob = dev_inputs(w, with_grad=False)
    kb, vb = block_kv(w)
    with pytest.raises(skv.SkvError):
        skv.block_local_fwd(prob, d["q"], kb.cuda(), vb.cuda())
