"""GPU parity of the grouped-query layouts [Split-KV Table 2: 32 query heads
over 4 or 8 key/value heads] against the CPU fp64 oracle on the same seeded
inputs: query head h reads key/value head h // (H / Hkv), and dk, dv (and the
block-local dk_blk, dv_blk) sum over each key/value head's query heads.  The
tensor-core forward and dQ kernels stack a group's g query heads in one
128-row tile (128/g rows each); the cases cover g = 2, 4, 8 and 16.
Element by element at sizes the oracle finishes in seconds (tensor-core bf16
and CUDA-core fp32 paths, multi-query Hkv = 1, ragged B); the full packed
shape with Hkv = 8 runs in tests/test_gpu_full.py.  Tolerances as for the
other parity tests: fp32 1e-4, bf16 2e-2 (o, dq, dk, dv) and 1e-3 (lse)."""
import pytest

import lse_merge_gb300 as skv
import oracle as orc
from gpu_helpers import TOL_BF16, TOL_BF16_LSE, TOL_FP32, assert_lse_equal, dev_inputs, maxabs
from test_gpu_attn import check_backward, check_forward
from test_gpu_block_local import whole_mask_forward
from workloads import block_kv, random_small

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("cfg", [
    # (seed, samples, L, anchors/sample, B, H, Hkv, d, m, P, dtype, order)
    (41, 2, 1024, 6, 16, 4, 2, 128, 256, 4, "bf16", "lpt"),
    (42, 1, 1408, 9, 16, 8, 1, 128, 128, 11, "bf16", "contiguous"),  # one key/value head
    (43, 2, 768, 5, 5, 4, 2, 64, 128, 3, "fp32", "lpt"),             # CUDA-core path, ragged B
    (44, 1, 640, 4, 24, 6, 3, 64, 128, 5, "bf16", "lpt"),            # B > 16, groups of 2
    (48, 1, 1024, 9, 16, 16, 1, 128, 256, 4, "bf16", "lpt"),         # 16 heads a tile, 8 rows each
])
def test_gqa_forward_backward(cfg):
    seed, b, L, A, B, H, Hkv, dd, m, P, dt, order = cfg
    w = random_small(seed, b, L, A, B, H, dd, m, P, dt, order=order).with_(Hkv=Hkv)
    tol = TOL_FP32 if dt == "fp32" else TOL_BF16
    tol_l = TOL_FP32 if dt == "fp32" else TOL_BF16_LSE
    inp, d, prob, roc, o, lse = check_forward(w, tol, tol_l, order=order)
    assert tuple(d["k"].shape) == (w.S, Hkv, dd)
    check_backward(w, inp, d, prob, roc, o, lse, tol)


@pytest.mark.parametrize("w,tol,tol_l", [
    (random_small(45, 2, 1536, 20, 16, 4, 128, 256, 6, dtype="bf16").with_(Hkv=2), TOL_BF16, TOL_BF16_LSE),
    (random_small(46, 1, 512, 12, 7, 6, 64, 128, 4, dtype="fp32").with_(Hkv=2), TOL_FP32, TOL_FP32),
    # the largest block with d = 128, four query heads on one key/value head
    (random_small(47, 1, 1024, 10, 32, 4, 128, 256, 4, dtype="bf16").with_(Hkv=1), TOL_BF16, TOL_BF16_LSE),
])
def test_gqa_whole_mask(w, tol, tol_l):
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
        assert tuple(g.shape) == r.shape, name
        err = maxabs(g.cpu().numpy(), r)
        assert err <= tol, f"{name} err {err}"
