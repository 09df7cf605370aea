"""Parity at the full workload sizes, in the launch configuration bench.py
times: the oracle computes sampled outputs one query block / key at a time
(two heads, 0 and H-1), and properties that hold at any size are checked on
every output (the exact -inf pattern of the partials, finiteness)."""
import gc

import numpy as np
import pytest
import torch

import lse_merge_gb300 as skv
import oracle as orc
from gpu_helpers import TOL_BF16, TOL_BF16_LSE, assert_lse_equal, maxabs
from workloads import LONG_1M, PACKED, PACKED_KV8, make_inputs, qs_sweep

pytestmark = pytest.mark.gpu

# every Q:S ratio of the sweep once, the two chunk orders alternating
FULL = [PACKED, LONG_1M, qs_sweep(4, "contiguous"), qs_sweep(8, "lpt"), qs_sweep(16, "contiguous"),
        qs_sweep(32, "lpt"), PACKED_KV8]


def sample_blocks(N, seed):
    rng = np.random.default_rng(seed)
    fixed = [0, 7, 8, N // 2, N - 1]
    return sorted(set(fixed + rng.integers(0, N, size=3).tolist()))


def empty_pattern(s, a, roc, m, P, B, H):
    """Exact -inf pattern of lse_part: row of block i is empty on rank p iff no
    chunk of p meets [s_i, a_i)."""
    s = s.numpy().astype(np.int64)
    a = a.numpy().astype(np.int64)
    N = len(s)
    has = np.zeros((P, N), bool)
    for j, p in enumerate(roc):
        lo, hi = j * m, (j + 1) * m
        has[p] |= (np.minimum(a, hi) - np.maximum(s, lo)) > 0
    return np.repeat(~has, B, axis=1)[:, :, None].repeat(H, axis=2)


@pytest.fixture(scope="module", params=FULL, ids=lambda w: w.name)
def full_run(request):
    w = request.param
    inp = make_inputs(w, device="cuda")
    s, a = inp.s.cuda(), inp.a.cuda()
    prob = skv.Problem(s, a, w.B, w.H, w.d, w.S, w.m, w.P, torch.bfloat16, n_kv_heads=w.Hkv)
    costs, roc, _, _ = skv.plan(prob, w.order)
    o_part, lse_part = skv.attn_fwd(prob, inp.q, inp.k, inp.v, roc)
    o, lse = skv.lse_merge(o_part, lse_part, out_dtype=torch.bfloat16)
    dq, dk, dv = skv.attn_bwd(prob, inp.q, inp.k, inp.v, o, lse, inp.dO, roc)
    assert skv.stream_status() == 0
    # a list, emptied at teardown: whatever still holds it then no longer holds the
    # workload's ~140 GB of device tensors when the next workload is drawn
    run = [w, inp, prob, roc.cpu().numpy(), o_part, lse_part, o, lse, dq, dk, dv]
    yield run
    run.clear()
    del inp, prob, o_part, lse_part, o, lse, dq, dk, dv, s, a, costs, roc
    gc.collect()
    torch.cuda.empty_cache()


def test_full_partials_pattern_and_finiteness(full_run):
    w, inp, prob, roc, o_part, lse_part, o, lse, _, _, _ = full_run
    lp = lse_part.cpu().numpy()
    assert np.array_equal(np.isneginf(lp), empty_pattern(inp.s, inp.a, roc, w.m, w.P, w.B, w.H))
    assert not np.isnan(lp).any() and not np.isposinf(lp).any()
    assert torch.isfinite(o.float()).all()
    assert torch.isfinite(lse).all()          # every block of these workloads sees some context
    # merge never lowers the log-sum-exp below a partial
    assert bool((lse[None] >= lse_part - 1e-4).all())


def test_full_merged_sampled_blocks(full_run):
    w, inp, prob, roc, o_part, lse_part, o, lse, _, _, _ = full_run
    heads = [0, w.H - 1]
    blocks = sample_blocks(w.N, w.seed)
    r_o, r_l = orc.attention_forward(inp.q, inp.k, inp.v, inp.s, inp.a, w.B, blocks=blocks, heads=heads)
    rows = np.concatenate([np.arange(i * w.B, (i + 1) * w.B) for i in blocks])
    rt = torch.as_tensor(rows, device="cuda")
    g_o = o[rt][:, heads].float().cpu().numpy()
    g_l = lse[rt][:, heads].cpu().numpy()
    assert_lse_equal(g_l, r_l[rows][:, heads], TOL_BF16_LSE)
    err = maxabs(g_o, r_o[rows][:, heads])
    assert err <= TOL_BF16, err


def test_full_partials_sampled_ranks(full_run):
    w, inp, prob, roc, o_part, lse_part, o, lse, _, _, _ = full_run
    heads = [0, w.H - 1]
    blocks = sample_blocks(w.N, w.seed + 1)[:4]
    rows = np.concatenate([np.arange(i * w.B, (i + 1) * w.B) for i in blocks])
    lp = lse_part.cpu().numpy()
    # the two ranks with the most finite partials among the sampled rows
    fin = np.isfinite(lp[:, rows][:, :, heads]).sum(axis=(1, 2))
    for p in np.argsort(-fin)[:2]:
        km = orc.chunk_key_mask(roc, int(p), w.m, w.S)
        r_o, r_l = orc.attention_forward(inp.q, inp.k, inp.v, inp.s, inp.a, w.B, key_mask=km, blocks=blocks,
                                         heads=heads)
        assert_lse_equal(lp[p][rows][:, heads], r_l[rows][:, heads], TOL_BF16_LSE)
        g = o_part[int(p)][torch.as_tensor(rows, device="cuda")][:, heads].cpu().numpy()
        mask = np.isfinite(r_l[rows][:, heads])[..., None].repeat(w.d, axis=-1)
        assert maxabs(g, r_o[rows][:, heads], mask) <= TOL_BF16


def few_attender_keys(s, a, limit=12):
    """Keys seen by at most `limit` blocks (cheap for the oracle), plus one key
    past every window of its sample."""
    s = s.numpy().astype(np.int64)
    a = a.numpy().astype(np.int64)
    keys = []
    for st in np.unique(s)[:2]:
        aa = np.sort(a[s == st])
        if len(aa) > limit:
            keys += [int(aa[-limit]), int(aa[-limit // 2]) + 1, int(aa[-1]) - 1]
        keys.append(int(aa[-1]) + 3)
    return sorted(set(k for k in keys if 0 <= k))


def test_full_dq_sampled_blocks(full_run):
    w, inp, prob, _, _, _, _, _, dq, dk, dv = full_run
    heads = [0, w.H - 1]
    blocks = sample_blocks(w.N, w.seed + 2)[:5]
    r_dq, _, _ = orc.attention_backward(inp.q, inp.k, inp.v, inp.s, inp.a, w.B, inp.dO, blocks=blocks, heads=heads)
    rows = np.concatenate([np.arange(i * w.B, (i + 1) * w.B) for i in blocks])
    g = dq[torch.as_tensor(rows, device="cuda")][:, heads].cpu().numpy()
    assert maxabs(g, r_dq[rows][:, heads]) <= TOL_BF16


def test_full_dkdv_sampled_keys(full_run):
    w, inp, prob, _, _, _, _, _, dq, dk, dv = full_run
    heads = [0, w.KVH - 1]                    # key/value heads (each sums its query heads)
    keys = [k for k in few_attender_keys(inp.s, inp.a) if k < w.S]
    r_dk, r_dv = orc.backward_key_rows(inp.q, inp.k, inp.v, inp.s, inp.a, w.B, inp.dO, keys, heads)
    kt = torch.as_tensor(keys, device="cuda")
    assert maxabs(dk[kt][:, heads].cpu().numpy(), r_dk) <= TOL_BF16
    assert maxabs(dv[kt][:, heads].cpu().numpy(), r_dv) <= TOL_BF16


def test_full_dkdv_prompt_keys(full_run):
    """Keys of the first sample's prompt quarter: every block of the sample sees
    them, so their key tiles walk every query tile of the sample in the
    key-stationary pass (the path that dominates the backward).  Key/value head
    0 only, on the workloads whose samples the oracle walks in seconds."""
    w, inp, prob, _, _, _, _, _, dq, dk, dv = full_run
    if w.name not in ("packed_4x128k", "qs_1to32_lpt"):
        pytest.skip("the oracle's walk over every block of a sample is too long here")
    L = w.sample_len
    keys = [0, 131, L // 8 + 77, L // 4 - 1]
    r_dk, r_dv = orc.backward_key_rows(inp.q, inp.k, inp.v, inp.s, inp.a, w.B, inp.dO, keys, [0])
    kt = torch.as_tensor(keys, device="cuda")
    assert maxabs(dk[kt][:, [0]].cpu().numpy(), r_dk) <= TOL_BF16
    assert maxabs(dv[kt][:, [0]].cpu().numpy(), r_dv) <= TOL_BF16


def test_full_gradient_properties(full_run):
    w, inp, prob, _, _, _, _, _, dq, dk, dv = full_run
    for t in (dq, dk, dv):
        assert bool(torch.isfinite(t).all())
    # keys no window covers get exactly zero gradient
    seen = torch.zeros(w.S, dtype=torch.bool)
    for si, ai in zip(inp.s.tolist(), inp.a.tolist()):
        seen[si:ai] = True
    unseen = (~seen).nonzero().flatten().cuda()
    if unseen.numel():
        assert float(dk[unseen].abs().max()) == 0.0 and float(dv[unseen].abs().max()) == 0.0
    # softmax rows sum to one: sum_x dv_x = sum_r dO_r over the key/value head's
    # query heads (every row sees some key here)
    g = w.H // w.KVH
    for c in (0, w.KVH - 1):
        lhs = dv[:, c].double().sum(0)
        grp = inp.dO[:, c * g:(c + 1) * g].double()
        rhs = grp.sum((0, 1))
        scale = grp.abs().sum((0, 1))
        assert float(((lhs - rhs).abs() / scale).max()) < 1e-2
