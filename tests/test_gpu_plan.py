"""GPU parity of the planning calls (chunk prices, LPT, contiguous, Zigzag):
bit-exact against the oracle and the printed Fig. 5 values of "Split-KV:
Efficient Context Parallelism for Training Diffusion Drafters"."""
import json
import os
import random

import numpy as np
import pytest
import torch

import lse_merge_gb300 as skv
import oracle as orc
from workloads import WORKLOADS, draw_anchors

pytestmark = pytest.mark.gpu

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def fig5_problem():
    with open(os.path.join(GOLD, "fig5_example.json")) as f:
        g = json.load(f)
    s, a = [], []
    for st, anc in zip(g["sample_starts"], g["anchors_in_sample"]):
        for x in anc:
            s.append(st)
            a.append(st + x)
    S = sum(g["sample_lens"])
    st = torch.tensor(s, dtype=torch.int32, device="cuda")
    at = torch.tensor(a, dtype=torch.int32, device="cuda")
    prob = skv.Problem(st, at, g["B"], 1, 64, S, g["m"], g["P"], torch.float32)
    return g, prob


def test_fig5_on_gpu():
    g, prob = fig5_problem()
    costs = skv.chunk_costs(prob)
    assert costs.cpu().tolist() == g["chunk_costs"]
    roc, order, load = skv.lpt_order(costs, g["P"], g["J"])
    assert load.cpu().tolist() == g["lpt_loads"]
    zz = skv.zigzag_loads(prob, torch.tensor(g["sample_starts"], dtype=torch.int32, device="cuda"),
                          torch.tensor(g["sample_lens"], dtype=torch.int32, device="cuda"))
    assert zz.cpu().tolist() == g["zigzag_loads"]
    assert skv.stream_status() == 0


@pytest.mark.parametrize("name", sorted(WORKLOADS))
def test_costs_and_lpt_every_workload(name):
    w = WORKLOADS[name]
    gen = torch.Generator().manual_seed(w.seed)
    s, a = draw_anchors(w, gen)
    prob = skv.Problem(s.cuda(), a.cuda(), w.B, w.H, w.d, w.S, w.m, w.P, torch.bfloat16)
    costs = skv.chunk_costs(prob).cpu().numpy()
    ref = orc.chunk_costs(s.numpy(), a.numpy(), w.B, w.S, w.m)
    assert np.array_equal(costs, ref)
    roc, order, load = skv.lpt_order(torch.from_numpy(costs).cuda(), w.P, w.J)
    r_roc, r_order, r_load = orc.lpt_assign(ref, w.P, w.J)
    assert np.array_equal(roc.cpu().numpy(), r_roc)
    assert np.array_equal(order.cpu().numpy(), r_order)
    assert np.array_equal(load.cpu().numpy(), r_load)
    c_roc, c_order, c_load = skv.contiguous_order(w.n_chunks, w.P, w.J, torch.from_numpy(costs).cuda())
    e_roc, e_order, e_load = orc.contiguous_assign(w.n_chunks, w.P, w.J, ref)
    assert np.array_equal(c_roc.cpu().numpy(), e_roc)
    assert np.array_equal(c_order.cpu().numpy(), e_order)
    assert np.array_equal(c_load.cpu().numpy(), e_load)
    assert skv.stream_status() == 0


@pytest.mark.parametrize("seed", range(10))
def test_lpt_random_with_ties(seed):
    rng = random.Random(seed)
    P = rng.choice([1, 2, 3, 7, 32, 33, 64, 100, 1024])
    J = rng.choice([1, 2, 3, 8])
    n = P * J
    hi = rng.choice([1, 3, 1000, 10**12])          # small ranges force many ties
    costs = np.array([rng.randint(0, hi) for _ in range(n)], np.int64)
    roc, order, load = skv.lpt_order(torch.from_numpy(costs).cuda(), P, J)
    e_roc, e_order, e_load = orc.lpt_assign(costs, P, J)
    assert np.array_equal(roc.cpu().numpy(), e_roc)
    assert np.array_equal(order.cpu().numpy(), e_order)
    assert np.array_equal(load.cpu().numpy(), e_load)


def test_lpt_max_size():
    P, J = 1024, 16
    costs = np.random.default_rng(0).integers(0, 5000, size=P * J).astype(np.int64)
    roc, order, load = skv.lpt_order(torch.from_numpy(costs).cuda(), P, J)
    e_roc, e_order, e_load = orc.lpt_assign(costs, P, J)
    assert np.array_equal(roc.cpu().numpy(), e_roc)
    assert np.array_equal(load.cpu().numpy(), e_load)


def test_costs_random_and_empty():
    rng = random.Random(5)
    for _ in range(5):
        n_samples = rng.randint(1, 5)
        L = 256 * rng.randint(1, 4)
        s, a = [], []
        for u in range(n_samples):
            for x in sorted(rng.sample(range(0, L + 1), rng.randint(0, 20))):
                s.append(u * L)
                a.append(u * L + x)
        S = n_samples * L
        m = 128
        B = rng.randint(1, 16)
        st = torch.tensor(s, dtype=torch.int32, device="cuda")
        at = torch.tensor(a, dtype=torch.int32, device="cuda")
        prob = skv.Problem(st, at, B, 1, 64, S, m, S // m)
        got = skv.chunk_costs(prob).cpu().numpy()
        assert np.array_equal(got, orc.chunk_costs(s, a, B, S, m))


def test_bad_anchors_raise_device_status():
    s = torch.tensor([0, 0], dtype=torch.int32, device="cuda")
    a = torch.tensor([5, 9000], dtype=torch.int32, device="cuda")   # a_1 > S
    prob = skv.Problem(s, a, 16, 1, 64, 4096, 1024, 4, torch.bfloat16)
    costs = skv.chunk_costs(prob).cpu().numpy()
    assert skv.stream_status() == 5          # SKV_ERR_BAD_ANCHORS
    # the offending block is clamped to [0, S)
    assert np.array_equal(costs, orc.chunk_costs([0, 0], [5, 4096], 16, 4096, 1024))
    assert skv.stream_status() == 0          # cleared by the previous read
