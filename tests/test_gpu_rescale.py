"""GPU parity with scores that rise steeply along the keys, against the CPU fp64
oracle on the same inputs.

Query feature 0 gets a constant and key feature 0 a ramp over the position in
its sample, so a row's scores grow by about 17 (natural-log units) per 128 keys
and by about 100 across its window:
  - the forward's running max grows at nearly every key tile, so O and l are
    rescaled on every step, not once at the first tile;
  - the per-rank partials' lse differ by tens, so the merge weights span many
    orders of magnitude;
  - the backward's P is concentrated on the last keys of each window; it is
    checked with the forward's own (o, lse) as given, the library's contract.
The workloads are otherwise those of the other parity tests. The forward's
tolerances are those tests' absolute bounds, taken relative to the largest
reference value (at least 1), since the ramp makes q and k up to tens. The
backward is held element by element to a bound derived from the relative error
of P and dS (see rounding_bounds)."""
import numpy as np
import pytest
import torch

import lse_merge_gb300 as skv
import oracle as orc
from gpu_helpers import TOL_BF16, TOL_BF16_LSE, TOL_FP32, assert_lse_equal, maxabs
from workloads import make_inputs, random_small

pytestmark = pytest.mark.gpu


def rising_inputs(w, gain_q, gain_k):
    inp = make_inputs(w, with_grad=True)
    pos = (torch.arange(w.S) % w.sample_len).double() / w.sample_len
    q, k = inp.q.double(), inp.k.double()
    q[:, :, 0] += gain_q
    k[:, :, 0] += gain_k * pos[:, None]
    inp.q, inp.k = q.to(inp.q.dtype), k.to(inp.k.dtype)
    return inp


def rounding_bounds(inp, B, o, lse, u):
    """Bounds on what a relative error u in each P and dS can move dq, dk, dv,
    in fp64 from the same inputs: |d dq_r| <= u scale sum_x |dS_rx| |k_x|,
    |d dk_x| <= u scale sum_r |dS_rx| |q_r|, |d dv_x| <= u sum_r P_rx |dO_r|.
      - bf16 path: u = 2^-8, the unit roundoff of the one rounding of P and dS
        to bf16 before the tensor-core MMAs.
      - fp32 path: u = 2^-16, the spacing of fp32 numbers at the exponent
        arguments' size (|z| up to ~200 in log2 units), which bounds P's error.
    Steep scores concentrate P on a few keys whose k share a large offset, so
    dq = scale sum_x dS_x k_x cancels (sum_x dS_x = 0): the bound on dq exceeds
    2e-2 of max |dq| for bf16."""
    q, k, v, dO = (np.asarray(x.double().numpy()) for x in (inp.q, inp.k, inp.v, inp.dO))
    s, a = inp.s.numpy().astype(np.int64), inp.a.numpy().astype(np.int64)
    Qn, H, d = q.shape
    S, Hkv = k.shape[0], k.shape[1]
    scale = 1.0 / np.sqrt(d)
    bq, bk, bv = np.zeros_like(q), np.zeros((S, Hkv, d)), np.zeros((S, Hkv, d))
    keys = np.arange(S)
    for h in range(H):
        c = h // (H // Hkv)
        for i in range(len(s)):
            rows = slice(i * B, (i + 1) * B)
            vis = (keys >= s[i]) & (keys < a[i])
            if not vis.any():
                continue
            kk, vv = k[vis, c, :], v[vis, c, :]
            z = q[rows, h, :] @ kk.T * scale
            P = np.exp(z - lse[rows, h][:, None])
            dS = P * (dO[rows, h, :] @ vv.T - np.sum(dO[rows, h, :] * o[rows, h, :], axis=1)[:, None])
            bq[rows, h, :] = u * scale * (np.abs(dS) @ np.abs(kk))
            bk[vis, c, :] += u * scale * (np.abs(dS).T @ np.abs(q[rows, h, :]))
            bv[vis, c, :] += u * (P.T @ np.abs(dO[rows, h, :]))
    return bq, bk, bv


def rel_err(g, r):
    r = np.asarray(r, np.float64)
    return maxabs(g, r) / max(1.0, float(np.abs(r).max()) if r.size else 1.0)


@pytest.mark.parametrize("cfg", [
    # (seed, samples, L, anchors/sample, B, H, Hkv, d, m, P, dtype, gain_q, gain_k)
    (71, 2, 1024, 6, 16, 2, 2, 128, 256, 4, "bf16", 32.0, 48.0),
    (72, 1, 1024, 8, 16, 2, 2, 64, 128, 4, "fp32", 32.0, 32.0),
    (73, 1, 1024, 9, 16, 8, 2, 128, 256, 4, "bf16", 32.0, 48.0),   # 4 query heads stacked a tile
])
def test_rising_scores(cfg):
    seed, b, L, A, B, H, Hkv, dd, m, P, dt, gq, gk = cfg
    w = random_small(seed, b, L, A, B, H, dd, m, P, dt, order="lpt").with_(Hkv=Hkv)
    inp = rising_inputs(w, gq, gk)
    tol = TOL_FP32 if dt == "fp32" else TOL_BF16
    tol_l = TOL_FP32 if dt == "fp32" else TOL_BF16_LSE
    d = {n: getattr(inp, n).cuda() for n in ("s", "a", "q", "k", "v", "dO")}
    prob = skv.Problem(d["s"], d["a"], w.B, w.H, w.d, w.S, w.m, w.P, d["q"].dtype, n_kv_heads=w.Hkv)
    _, roc, _, _ = skv.plan(prob, "lpt")
    o_part, lse_part = skv.attn_fwd(prob, d["q"], d["k"], d["v"], roc)
    o, lse = skv.lse_merge(o_part, lse_part, out_dtype=d["q"].dtype)
    dq, dk, dv = skv.attn_bwd(prob, d["q"], d["k"], d["v"], o, lse, d["dO"], roc)
    assert skv.stream_status() == 0

    r_o, r_l = orc.attention_forward(inp.q, inp.k, inp.v, inp.s, inp.a, w.B)
    fin = np.isfinite(r_l)
    # the ramp really is steep: each row's scores span tens of natural-log units
    assert float(np.ptp(r_l[fin])) > 20.0
    assert_lse_equal(lse.cpu().numpy(), r_l, tol_l)
    assert rel_err(o.float().cpu().numpy(), r_o) <= tol

    r_op, r_lp = orc.partition_forward(inp.q, inp.k, inp.v, inp.s, inp.a, w.B, roc.cpu().numpy(), w.m, w.P)
    assert_lse_equal(lse_part.cpu().numpy(), r_lp, tol_l)
    pf = np.broadcast_to(np.isfinite(r_lp)[..., None], r_op.shape)
    scale = max(1.0, float(np.abs(r_op[pf]).max()))
    assert maxabs(o_part.cpu().numpy(), r_op, pf) <= tol * scale

    # The backward takes (o, lse) as given, as the library does (Alg. 1's MERGE_BWD in
    # merged form: D = dO . o): both sides read the same o, rounded to the input dtype.
    # With P concentrated on one key, dP - D is a small difference of two terms of
    # size |dO||v|, so the rounding of o alone would move dq by a few per cent.
    r_dq, r_dk, r_dv = orc.context_backward_given(inp.q, inp.k, inp.v, inp.s, inp.a, w.B, inp.dO,
                                                  o.float().cpu().double().numpy(),
                                                  lse.cpu().double().numpy())
    # element by element within twice the rounding bound, plus a small absolute term
    # for the fp32 sums (1e-3 bf16, 1e-5 fp32); and within 10 % of the output's scale
    u, slack = (2.0 ** -16, 1e-5) if dt == "fp32" else (2.0 ** -8, 1e-3)
    bounds = rounding_bounds(inp, w.B, o.float().cpu().double().numpy(), lse.cpu().double().numpy(), u)
    for name, g, r, bd in (("dq", dq, r_dq, bounds[0]), ("dk", dk, r_dk, bounds[1]), ("dv", dv, r_dv, bounds[2])):
        gg = g.cpu().numpy().astype(np.float64)
        excess = np.abs(gg - r) - (2.0 * bd + slack)
        assert float(excess.max()) <= 0.0, f"{name} exceeds the rounding bound by {float(excess.max())}"
        assert rel_err(gg, r) <= 0.1, name
