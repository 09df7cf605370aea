"""Pins of the oracle's per-partial merge backward (CPU only).

[Split-KV §4.1, Eq. 4; the MERGE_BWD step of Alg. 1's backward]: the gradients
of o = sum_p exp(l_p - l) o_p and l = log sum_p exp(l_p) with respect to every
partial, checked against central finite differences of the oracle's forward
merge, the invariant sum_p dl_p = dlse, the single-partial special case, and
the route through the attention backward.
"""
import numpy as np
import pytest

import oracle as orc


def rand_partials(seed, P=4, rows=6, d=5, n_inf=3):
    rng = np.random.default_rng(seed)
    op = rng.standard_normal((P, rows, d))
    lp = rng.standard_normal((P, rows)) * 2.0
    # some partials empty (-inf), and one row with every partial empty
    for _ in range(n_inf):
        lp[rng.integers(0, P), rng.integers(0, rows - 1)] = -np.inf
    lp[:, rows - 1] = -np.inf
    return op, lp, rng


def loss(op, lp, g, gl):
    o, l = orc.lse_merge(op, lp)
    fin = np.isfinite(l)
    return (g * o).sum() + (gl * np.where(fin, l, 0.0)).sum()


@pytest.mark.parametrize("seed", range(4))
def test_merge_backward_finite_differences(seed):
    op, lp, rng = rand_partials(seed)
    g = rng.standard_normal(op.shape[1:])
    gl = rng.standard_normal(lp.shape[1:])
    do_p, dl_p = orc.lse_merge_backward(op, lp, g, gl)
    eps = 1e-6
    fin = np.isfinite(lp)
    for idx in np.ndindex(*op.shape):
        if not fin[idx[:2]]:
            continue
        a, b = op.copy(), op.copy()
        a[idx] += eps
        b[idx] -= eps
        num = (loss(a, lp, g, gl) - loss(b, lp, g, gl)) / (2 * eps)
        assert abs(num - do_p[idx]) < 1e-6
    for idx in np.ndindex(*lp.shape):
        if not fin[idx]:
            continue
        a, b = lp.copy(), lp.copy()
        a[idx] += eps
        b[idx] -= eps
        num = (loss(op, a, g, gl) - loss(op, b, g, gl)) / (2 * eps)
        assert abs(num - dl_p[idx]) < 1e-6


def test_merge_backward_empty_partials_and_rows():
    op, lp, rng = rand_partials(7)
    g = rng.standard_normal(op.shape[1:])
    do_p, dl_p = orc.lse_merge_backward(op, lp, g)
    fin = np.isfinite(lp)
    assert np.all(do_p[~fin] == 0) and np.all(dl_p[~fin] == 0)
    assert np.all(do_p[:, -1] == 0) and np.all(dl_p[:, -1] == 0)


@pytest.mark.parametrize("seed", range(3))
def test_merge_backward_invariants(seed):
    # sum_p w_p = 1 gives sum_p dl_p = dlse and sum_p do_p = dO on every row
    # with a finite partial; one partial alone passes the gradients through.
    op, lp, rng = rand_partials(seed, P=5, rows=7, d=3, n_inf=4)
    g = rng.standard_normal(op.shape[1:])
    gl = rng.standard_normal(lp.shape[1:])
    do_p, dl_p = orc.lse_merge_backward(op, lp, g, gl)
    live = np.isfinite(lp).any(axis=0)
    np.testing.assert_allclose(dl_p.sum(0)[live], gl[live], atol=1e-12)
    np.testing.assert_allclose(do_p.sum(0)[live], g[live], atol=1e-12)
    d1, l1 = orc.lse_merge_backward(op[:1], lp[:1], g, gl)
    f1 = np.isfinite(lp[0])
    np.testing.assert_allclose(d1[0][f1], g[f1], atol=0)
    np.testing.assert_allclose(l1[0][f1], gl[f1], atol=1e-12)


def _torch_partial(q, k, v, allow):
    # o_p, l_p of Eq. 3 for one key subset, in torch fp64 (masked softmax)
    import torch
    z = torch.einsum("rhd,xhd->hrx", q, k) / np.sqrt(q.shape[-1])
    z = z.masked_fill(~allow[None], float("-inf"))
    l = torch.logsumexp(z, dim=-1)                                  # [H, R]
    p = torch.exp(z - torch.where(torch.isfinite(l), l, torch.zeros_like(l))[..., None])
    p = torch.where(allow[None], p, torch.zeros_like(p))
    o = torch.einsum("hrx,xhd->rhd", p, v)
    return o, l.transpose(0, 1)


def test_merge_backward_chain_rule_through_the_partials():
    # Chain rule pin with torch autograd (fp64): pushing each partial's
    # (d o_p, d l_p) from this function through that partial's own vjp, and
    # summing over partials, gives the gradient of the single-device attention.
    import torch
    rng = np.random.default_rng(3)
    B, H, d, S, m, P = 2, 2, 3, 16, 4, 3
    s, a = np.array([0, 0, 0, 8]), np.array([6, 10, 16, 13])
    R = len(s) * B
    q = torch.tensor(rng.standard_normal((R, H, d)), requires_grad=True)
    k = torch.tensor(rng.standard_normal((S, H, d)), requires_grad=True)
    v = torch.tensor(rng.standard_normal((S, H, d)), requires_grad=True)
    g = rng.standard_normal((R, H, d))
    gl = rng.standard_normal((R, H))
    roc = np.array([0, 2, 1, 2])
    x = np.arange(S)
    win = np.stack([(s[r // B] <= x) & (x < a[r // B]) for r in range(R)])
    o, l = _torch_partial(q, k, v, torch.tensor(win))
    ref = torch.autograd.grad([o, l], [q, k, v], [torch.tensor(g), torch.tensor(gl)])
    ops, lps = [], []
    for p in range(P):
        allow = torch.tensor(win & (roc[x // m] == p)[None])
        o_p, l_p = _torch_partial(q, k, v, allow)
        ops.append(o_p)
        lps.append(l_p)
    op = np.stack([t.detach().numpy() for t in ops])
    lp = np.stack([t.detach().numpy() for t in lps])
    do_p, dl_p = orc.lse_merge_backward(op, lp, g, gl)
    tot = [torch.zeros_like(t) for t in (q, k, v)]
    for p in range(P):
        fin = torch.tensor(np.isfinite(lp[p]))
        lq = torch.where(fin, lps[p], torch.zeros_like(lps[p]))
        gr = torch.autograd.grad([ops[p], lq], [q, k, v], [torch.tensor(do_p[p]), torch.tensor(dl_p[p])],
                                 allow_unused=True)
        tot = [t + (x if x is not None else 0) for t, x in zip(tot, gr)]
    for t, r in zip(tot, ref):
        np.testing.assert_allclose(t.numpy(), r.numpy(), atol=1e-10)
