"""Shared helpers of the GPU parity tests (GPU side through the C-ABI binding,
expected values from the CPU oracle only)."""
import numpy as np
import torch

import lse_merge_gb300 as skv
from workloads import Workload, make_inputs

# Tolerances (max abs error) for floating outputs.
TOL_FP32 = 1e-4
TOL_BF16 = 2e-2          # o, dq, dk, dv
TOL_BF16_LSE = 1e-3      # lse


def dev_inputs(w: Workload, with_grad=None):
    inp = make_inputs(w, with_grad=with_grad)
    d = {"s": inp.s.cuda(), "a": inp.a.cuda(), "q": inp.q.cuda(), "k": inp.k.cuda(), "v": inp.v.cuda(),
         "dO": inp.dO.cuda() if inp.dO is not None else None}
    tdt = torch.float32 if w.dtype == "fp32" else torch.bfloat16
    prob = skv.Problem(d["s"], d["a"], w.B, w.H, w.d, w.S, w.m, w.P, tdt, n_kv_heads=w.Hkv)
    return inp, d, prob


def maxabs(a, b, mask=None):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    if mask is not None:
        a, b = a[mask], b[mask]
    diff = np.abs(a - b)
    return float(diff.max()) if diff.size else 0.0


def assert_lse_equal(gpu_lse, ref_lse, tol):
    """Same -inf pattern; finite entries within tol."""
    g = np.asarray(gpu_lse, np.float64)
    r = np.asarray(ref_lse, np.float64)
    assert np.array_equal(np.isneginf(g), np.isneginf(r)), "different empty-partial pattern"
    fin = np.isfinite(r)
    assert np.all(np.isfinite(g[fin]))
    err = maxabs(g, r, fin)
    assert err <= tol, f"lse max abs err {err} > {tol}"
    return err
