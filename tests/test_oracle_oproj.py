"""Pins of the oracle's merge with the output projection [Split-KV §4.1, Eq. 5;
the MERGE_AR -> OProj -> RS_sum steps of Alg. 1's forward] (CPU only):
a scalar brute force on a tiny case, Eq. 5's linearity against Eq. 4's merge
followed by one projection, the one-partial and identity-projection special
cases, and the empty-partial conventions."""
import math

import numpy as np
import pytest

import oracle as orc


def _partials(seed, P, Q, H, d, frac_empty=0.25):
    rng = np.random.default_rng(seed)
    o_part = rng.standard_normal((P, Q, H, d))
    lse_part = 3.0 * rng.standard_normal((P, Q, H))
    lse_part[rng.random((P, Q, H)) < frac_empty] = -np.inf
    lse_part[:, -1, 0] = -np.inf                       # one (row, head) with no visible key at all
    return o_part, lse_part


def test_brute_force_scalar_loops():
    P, Q, H, d, dm = 3, 4, 2, 3, 5
    o_part, lse_part = _partials(1, P, Q, H, d)
    w = np.random.default_rng(2).standard_normal((dm, H * d))
    y, lse = orc.merge_oproj(o_part, lse_part, w)
    for r in range(Q):
        for j in range(dm):
            acc = 0.0
            for h in range(H):
                ls = [lse_part[p, r, h] for p in range(P) if math.isfinite(lse_part[p, r, h])]
                if not ls:
                    continue
                mx = max(ls)
                tot = mx + math.log(sum(math.exp(x - mx) for x in ls))
                for p in range(P):
                    if not math.isfinite(lse_part[p, r, h]):
                        continue
                    wp = math.exp(lse_part[p, r, h] - tot)
                    for c in range(d):
                        acc += wp * o_part[p, r, h, c] * w[j, h * d + c]
            assert abs(y[r, j] - acc) < 1e-12
    assert np.isneginf(lse[-1, 0])
    assert np.all(y[-1] == y[-1])                      # finite: the empty head adds nothing


def test_linearity_equals_merge_then_project():
    # Eq. 5: the sum of the projected weighted partials is the projection of
    # Eq. 4's merged output
    P, Q, H, d, dm = 5, 7, 3, 8, 11
    o_part, lse_part = _partials(3, P, Q, H, d)
    w = np.random.default_rng(4).standard_normal((dm, H * d))
    y, lse = orc.merge_oproj(o_part, lse_part, w)
    o, l2 = orc.lse_merge(o_part, lse_part)
    assert np.array_equal(np.isneginf(lse), np.isneginf(l2))
    assert np.allclose(y, o.reshape(Q, H * d) @ w.T, rtol=0, atol=1e-12)
    # a partial dropped from the sum is seen
    lp2 = lse_part.copy()
    lp2[1] = -np.inf
    y2, _ = orc.merge_oproj(o_part, lp2, w)
    assert np.abs(y2 - y).max() > 1e-3


def test_single_partial_and_identity_projection():
    o_part, lse_part = _partials(5, 1, 6, 2, 4, frac_empty=0.0)
    lse_part[0, -1, 0] = 0.7                            # every partial visible: the weight is 1
    w = np.random.default_rng(6).standard_normal((3, 8))
    y, _ = orc.merge_oproj(o_part, lse_part, w)
    assert np.allclose(y, o_part[0].reshape(6, 8) @ w.T, rtol=0, atol=1e-12)
    o_part, lse_part = _partials(7, 4, 5, 2, 4)
    y, lse = orc.merge_oproj(o_part, lse_part, np.eye(8))
    o, _ = orc.lse_merge(o_part, lse_part)
    assert np.allclose(y, o.reshape(5, 8), rtol=0, atol=1e-12)
