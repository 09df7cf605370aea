"""Pins of the oracle's block-local term and full-mask definitions (CPU only).

Source: "Split-KV: Efficient Context Parallelism for Training Diffusion
Drafters", §3.1 Fig. 1 (each block's B tokens attend to the context window and,
bidirectionally, to each other) and Eq. 4 (disjoint key sets merge exactly).
Pins: closed forms (B = 1, q = 0), torch scaled_dot_product_attention in fp64
with an explicit mask over the concatenated keys (forward and autograd), the
merge identity for every partition, and central finite differences.
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle as orc
from test_oracle_pins import rand_problem


def block_inputs(seed, Qn, H, d):
    g = torch.Generator().manual_seed(1000 + seed)
    return (torch.randn(Qn, H, d, generator=g, dtype=torch.float64),
            torch.randn(Qn, H, d, generator=g, dtype=torch.float64))


def sdpa_full(q, k, v, kb, vb, s, a, B, scale, dO=None):
    """fp64 SDPA over [context keys; block keys] with the anchor mask written out."""
    Qn, S = q.shape[0], k.shape[0]
    mask = torch.zeros(Qn, S + Qn, dtype=torch.bool)
    for r in range(Qn):
        i = r // B
        mask[r, s[i]:a[i]] = True
        mask[r, S + i * B:S + (i + 1) * B] = True
    keys = torch.cat([k, kb]).permute(1, 0, 2).clone().requires_grad_(dO is not None)
    vals = torch.cat([v, vb]).permute(1, 0, 2).clone().requires_grad_(dO is not None)
    qq = q.permute(1, 0, 2).clone().requires_grad_(dO is not None)
    o = F.scaled_dot_product_attention(qq[None], keys[None], vals[None], attn_mask=mask[None, None],
                                       scale=scale)[0].permute(1, 0, 2)
    if dO is None:
        return o.detach().numpy()
    (o * dO).sum().backward()
    gk = keys.grad.permute(1, 0, 2).numpy()
    gv = vals.grad.permute(1, 0, 2).numpy()
    return (o.detach().numpy(), qq.grad.permute(1, 0, 2).numpy(), gk[:S], gv[:S], gk[S:], gv[S:])


def test_block_local_single_token_closed_form():
    # B = 1: one key per row, softmax weight 1: o = v_blk, l = scale q . k_blk.
    g = torch.Generator().manual_seed(3)
    q, kb, vb = (torch.randn(7, 2, 5, generator=g, dtype=torch.float64) for _ in range(3))
    o, lse = orc.block_local_forward(q, kb, vb, 1, 0.8)
    np.testing.assert_allclose(o, vb.numpy(), atol=1e-14)
    np.testing.assert_allclose(lse, 0.8 * (q * kb).sum(-1).numpy(), atol=1e-13)


def test_block_local_q_zero_closed_form():
    # q = 0: all B scores are 0: l = log B, o = mean of the block's v_blk rows.
    B = 4
    g = torch.Generator().manual_seed(4)
    kb, vb = (torch.randn(12, 3, 6, generator=g, dtype=torch.float64) for _ in range(2))
    o, lse = orc.block_local_forward(torch.zeros(12, 3, 6, dtype=torch.float64), kb, vb, B)
    np.testing.assert_allclose(lse, math.log(B), atol=1e-14)
    for r in range(12):
        i = r // B
        np.testing.assert_allclose(o[r], vb[i * B:(i + 1) * B].mean(0).numpy(), atol=1e-14)


@pytest.mark.parametrize("seed", range(3))
def test_full_mask_forward_vs_torch_sdpa(seed):
    s, a, q, k, v, _ = rand_problem(seed, n_samples=2, L=30, A=3, B=3, H=2, d=8)
    kb, vb = block_inputs(seed, q.shape[0], 2, 8)
    sc = 1 / math.sqrt(8)
    o, _ = orc.full_mask_forward(q, k, v, kb, vb, s, a, 3, sc)
    np.testing.assert_allclose(o, sdpa_full(q, k, v, kb, vb, s, a, 3, sc), atol=1e-12)


@pytest.mark.parametrize("seed", range(3))
def test_block_partial_merges_with_every_partition(seed):
    # the block-local (o, l) is one more disjoint partial: merging it with the
    # rank partials of any chunk assignment gives the full-mask result (Eq. 4)
    s, a, q, k, v, _ = rand_problem(seed, n_samples=2, L=32, A=3, B=2, H=2, d=4)
    kb, vb = block_inputs(seed, q.shape[0], 2, 4)
    S, m = 64, 8
    ref_o, ref_l = orc.full_mask_forward(q, k, v, kb, vb, s, a, 2)
    ob, lb = orc.block_local_forward(q, kb, vb, 2)
    rng = np.random.default_rng(seed)
    for P in (1, 2, 4, 8):
        roc = rng.permutation(np.repeat(np.arange(P), (S // m) // P))
        op, lp = orc.partition_forward(q, k, v, s, a, 2, roc, m, P)
        o, lse = orc.lse_merge(np.concatenate([op, ob[None]]), np.concatenate([lp, lb[None]]))
        np.testing.assert_allclose(o, ref_o, atol=1e-12)
        np.testing.assert_allclose(lse, ref_l, atol=1e-12)


@pytest.mark.parametrize("seed", range(3))
def test_full_mask_backward_vs_torch_autograd(seed):
    # context part (merged form) + block-local part = autograd of the full mask
    s, a, q, k, v, dO = rand_problem(seed, n_samples=2, L=30, A=3, B=3, H=2, d=8)
    kb, vb = block_inputs(seed, q.shape[0], 2, 8)
    sc = 1 / math.sqrt(8)
    o, lse = orc.full_mask_forward(q, k, v, kb, vb, s, a, 3, sc)
    dq_c, dk, dv = orc.context_backward_given(q, k, v, s, a, 3, dO, o, lse, sc)
    dq_b, dkb, dvb = orc.block_local_backward(q, kb, vb, dO, o, lse, 3, sc)
    _, rq, rk, rv, rkb, rvb = sdpa_full(q, k, v, kb, vb, s, a, 3, sc, dO)
    np.testing.assert_allclose(dq_c + dq_b, rq, atol=1e-12)
    np.testing.assert_allclose(dk, rk, atol=1e-12)
    np.testing.assert_allclose(dv, rv, atol=1e-12)
    np.testing.assert_allclose(dkb, rkb, atol=1e-12)
    np.testing.assert_allclose(dvb, rvb, atol=1e-12)


def test_given_route_without_block_is_attention_backward():
    s, a, q, k, v, dO = rand_problem(6, n_samples=2, L=24, A=3, B=2, H=2, d=4)
    o, lse = orc.attention_forward(q, k, v, s, a, 2)
    got = orc.context_backward_given(q, k, v, s, a, 2, dO, o, lse)
    ref = orc.attention_backward(q, k, v, s, a, 2, dO)
    for x, y in zip(got, ref):
        np.testing.assert_allclose(x, y, atol=1e-12)


def test_block_local_finite_differences():
    s, a, q, k, v, dO = rand_problem(12, n_samples=2, L=10, A=2, B=2, H=1, d=3)
    kb, vb = block_inputs(12, q.shape[0], 1, 3)
    sc = 0.9
    o, lse = orc.full_mask_forward(q, k, v, kb, vb, s, a, 2, sc)
    dq_c, _, _ = orc.context_backward_given(q, k, v, s, a, 2, dO, o, lse, sc)
    dq_b, dkb, dvb = orc.block_local_backward(q, kb, vb, dO, o, lse, 2, sc)
    g = dO.numpy()

    def loss(qq, kk, vv):
        oo, _ = orc.full_mask_forward(qq, k, v, kk, vv, s, a, 2, sc)
        return float((oo * g).sum())

    h = 1e-6
    rng = np.random.default_rng(1)
    base = {"q": q.numpy(), "kb": kb.numpy(), "vb": vb.numpy()}
    for name, grad in (("q", dq_c + dq_b), ("kb", dkb), ("vb", dvb)):
        flat = base[name].reshape(-1)
        for idx in rng.choice(flat.size, size=6, replace=False):
            args = {n: t.copy() for n, t in base.items()}
            args[name].reshape(-1)[idx] += h
            up = loss(args["q"], args["kb"], args["vb"])
            args[name].reshape(-1)[idx] -= 2 * h
            dn = loss(args["q"], args["kb"], args["vb"])
            fd = (up - dn) / (2 * h)
            an = grad.reshape(-1)[idx]
            assert abs(fd - an) <= 1e-6 * max(1.0, abs(an)), (name, idx, fd, an)
