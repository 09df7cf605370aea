"""Pins of the oracle's grouped-query layouts (CPU only).

[Split-KV Table 2: the drafters' attention, 32 query heads over 4 or 8
key/value heads.]  Query head h reads key/value head h // (H / Hkv); the
gradients of a key/value head sum over its query heads.  Pinned against torch's
scaled_dot_product_attention with enable_gqa (fp64, explicit masks, autograd for
the backward), for the context path, the per-rank partition + merge, the
key-row sampler and the block-local term.
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle as orc
from workloads import make_inputs, random_small
from test_oracle_pins import rand_problem


def gqa_problem(seed, H=4, Hkv=2, **kw):
    s, a, q, k, v, dO = rand_problem(seed, H=H, **kw)
    g = torch.Generator().manual_seed(seed + 99)
    k = torch.randn(k.shape[0], Hkv, k.shape[2], generator=g, dtype=torch.float64)
    v = torch.randn(v.shape[0], Hkv, v.shape[2], generator=g, dtype=torch.float64)
    return s, a, q, k, v, dO


def sdpa_gqa(q, k, v, mask, scale, dO=None):
    """torch SDPA with enable_gqa; q [R, H, d], k/v [S, Hkv, d], mask [R, S]."""
    qq = q.permute(1, 0, 2).clone().requires_grad_(dO is not None)
    kk = k.permute(1, 0, 2).clone().requires_grad_(dO is not None)
    vv = v.permute(1, 0, 2).clone().requires_grad_(dO is not None)
    o = F.scaled_dot_product_attention(qq[None], kk[None], vv[None], attn_mask=mask[None, None], scale=scale,
                                       enable_gqa=True)[0].permute(1, 0, 2)
    if dO is None:
        return o.detach().numpy()
    (o * dO).sum().backward()
    return (o.detach().numpy(), qq.grad.permute(1, 0, 2).numpy(), kk.grad.permute(1, 0, 2).numpy(),
            vv.grad.permute(1, 0, 2).numpy())


def window_mask(s, a, B, Qn, S):
    m = torch.zeros(Qn, S, dtype=torch.bool)
    for r in range(Qn):
        m[r, s[r // B]:a[r // B]] = True
    return m


def test_kv_head_map():
    assert [orc.kv_head(h, 32, 8) for h in range(32)] == [h // 4 for h in range(32)]
    assert [orc.kv_head(h, 32, 4) for h in range(32)] == [h // 8 for h in range(32)]
    assert [orc.kv_head(h, 6, 6) for h in range(6)] == list(range(6))


@pytest.mark.parametrize("H,Hkv", [(4, 2), (4, 1), (6, 3)])
def test_gqa_forward_backward_vs_sdpa(H, Hkv):
    s, a, q, k, v, dO = gqa_problem(3 + H + Hkv, H=H, Hkv=Hkv, n_samples=2, L=40, A=4, B=3, d=8)
    sc = 1 / math.sqrt(8)
    mask = window_mask(s, a, 3, q.shape[0], k.shape[0])
    o, _ = orc.attention_forward(q, k, v, s, a, 3, sc)
    dq, dk, dv = orc.attention_backward(q, k, v, s, a, 3, dO, sc)
    ro, rq, rk, rv = sdpa_gqa(q, k, v, mask, sc, dO)
    np.testing.assert_allclose(o, ro, atol=1e-12)
    np.testing.assert_allclose(dq, rq, atol=1e-12)
    assert dk.shape == (k.shape[0], Hkv, 8)
    np.testing.assert_allclose(dk, rk, atol=1e-12)
    np.testing.assert_allclose(dv, rv, atol=1e-12)


def test_gqa_partitions_merge_and_key_rows():
    s, a, q, k, v, dO = gqa_problem(8, H=4, Hkv=2, n_samples=2, L=32, A=3, B=2, d=4)
    S, m = 64, 8
    o, lse = orc.attention_forward(q, k, v, s, a, 2)
    costs = orc.chunk_costs(s, a, 2, S, m)
    roc = orc.lpt_assign(costs, 4, 2)[0]
    op, lp = orc.partition_forward(q, k, v, s, a, 2, roc, m, 4)
    om, lm = orc.lse_merge(op, lp)
    np.testing.assert_allclose(om, o, atol=1e-12)
    np.testing.assert_allclose(lm, lse, atol=1e-12)
    dq, dk, dv = orc.attention_backward(q, k, v, s, a, 2, dO)
    pq, pk, pv, _ = orc.partitioned_backward(q, k, v, s, a, 2, dO, roc, m, 4)
    np.testing.assert_allclose(pq, dq, atol=1e-12)
    np.testing.assert_allclose(pk, dk, atol=1e-12)
    np.testing.assert_allclose(pv, dv, atol=1e-12)
    keys = [0, 5, 17, 33, 40, 63]
    rk, rv = orc.backward_key_rows(q, k, v, s, a, 2, dO, keys, [1, 0])
    np.testing.assert_allclose(rk, dk[keys][:, [1, 0]], atol=1e-12)
    np.testing.assert_allclose(rv, dv[keys][:, [1, 0]], atol=1e-12)


def test_gqa_block_local_term_vs_sdpa():
    # the whole mask (context window + own block, one softmax) per block, with
    # grouped k_blk, v_blk [Q, Hkv, d]; forward and gradients
    s, a, q, k, v, dO = gqa_problem(12, H=4, Hkv=2, n_samples=2, L=24, A=3, B=2, d=4)
    B, sc = 2, 0.6
    Qn, S = q.shape[0], k.shape[0]
    g = torch.Generator().manual_seed(5)
    kb = torch.randn(Qn, 2, 4, generator=g, dtype=torch.float64)
    vb = torch.randn(Qn, 2, 4, generator=g, dtype=torch.float64)
    o, lse = orc.full_mask_forward(q, k, v, kb, vb, s, a, B, sc)
    cq, ck, cv = orc.context_backward_given(q, k, v, s, a, B, dO, o, lse, sc)
    lq, lk, lv = orc.block_local_backward(q, kb, vb, dO, o, lse, B, sc)
    for i in range(len(s)):
        rows = slice(i * B, (i + 1) * B)
        keys = torch.cat([k, kb[rows]])
        vals = torch.cat([v, vb[rows]])
        mask = torch.zeros(B, S + B, dtype=torch.bool)
        mask[:, s[i]:a[i]] = True
        mask[:, S:] = True
        ro, rq, rk, rv = sdpa_gqa(q[rows], keys, vals, mask, sc, dO[rows])
        np.testing.assert_allclose(o[rows], ro, atol=1e-12)
        np.testing.assert_allclose(cq[rows] + lq[rows], rq, atol=1e-12)
        np.testing.assert_allclose(lk[rows], rk[S:], atol=1e-12)
        np.testing.assert_allclose(lv[rows], rv[S:], atol=1e-12)
    # context key gradients: every block's contribution summed
    tk = np.zeros_like(ck)
    tv = np.zeros_like(cv)
    for i in range(len(s)):
        rows = slice(i * B, (i + 1) * B)
        mask = torch.zeros(B, S + B, dtype=torch.bool)
        mask[:, s[i]:a[i]] = True
        mask[:, S:] = True
        _, _, rk, rv = sdpa_gqa(q[rows], torch.cat([k, kb[rows]]), torch.cat([v, vb[rows]]), mask, sc, dO[rows])
        tk += rk[:S]
        tv += rv[:S]
    np.testing.assert_allclose(ck, tk, atol=1e-12)
    np.testing.assert_allclose(cv, tv, atol=1e-12)


def test_backward_kv_heads_only_selects_the_same_sums():
    # the compact dk/dv of kv_heads_only are the full arrays' columns of the
    # key/value heads in use, in order of first use (here heads 5 then 0 of an
    # 8-over-2 layout: key/value heads 1, then 0)
    w = random_small(71, 1, 384, 5, 4, 8, 16, 128, 3, "fp32").with_(Hkv=2)
    inp = make_inputs(w)
    full = orc.attention_backward(inp.q, inp.k, inp.v, inp.s, inp.a, w.B, inp.dO, heads=[5, 0])
    part = orc.attention_backward(inp.q, inp.k, inp.v, inp.s, inp.a, w.B, inp.dO, heads=[5, 0], kv_heads_only=True)
    assert np.array_equal(full[0], part[0])
    for f, p_ in zip(full[1:], part[1:]):
        assert p_.shape == (w.S, 2, w.d)
        assert np.array_equal(f[:, 1], p_[:, 0]) and np.array_equal(f[:, 0], p_[:, 1])
