"""GPU parity of the per-partial merge backward (MERGE_BWD of Alg. 1, the
derivative of Eq. 4) against the CPU fp64 oracle on the same seeded partials.

Element by element at small sizes (every head_dim the kernel dispatches, fp32
and bf16 upstream gradients, empty partials, an all-empty row, with and
without dlse); at the packed workload's merge size (P = 16, Q*H rows, d = 128)
on sampled rows plus the invariants sum_p dlse_p = dlse and sum_p do_p = dO on
every row.  fp32 arithmetic: 1e-4 max abs error on dlse_part, 1e-5 on do_part
relative to |dO| (a product of two fp32 values)."""
import numpy as np
import pytest
import torch

import lse_merge_gb300 as skv
import oracle as orc
from workloads import PACKED, merge_partials

pytestmark = pytest.mark.gpu

TOL_DL = 1e-4
TOL_DO = 1e-5


def check(seed, P, rows, d, dt, with_dlse, want_do):
    op, lp, g, gl = merge_partials(seed, P, rows, d, dt)
    do_p, dl_p = skv.lse_merge_bwd(op.cuda(), lp.cuda(), g.cuda(), gl.cuda() if with_dlse else None,
                                   want_do_part=want_do)
    assert skv.stream_status() == 0
    r_do, r_dl = orc.lse_merge_backward(op.numpy(), lp.numpy(), g.float().numpy(), gl.numpy() if with_dlse else None)
    err = np.abs(dl_p.cpu().numpy() - r_dl).max()
    assert err <= TOL_DL, f"dlse_part err {err}"
    if want_do:
        err = np.abs(do_p.cpu().numpy() - r_do).max()
        assert err <= TOL_DO * max(1.0, float(np.abs(g.float().numpy()).max())), f"do_part err {err}"
    else:
        assert do_p is None


@pytest.mark.parametrize("d", [4, 8, 16, 32, 64, 128, 256])
@pytest.mark.parametrize("dt", ["fp32", "bf16"])
def test_merge_bwd_every_head_dim(d, dt):
    check(11 + d, 5, 67, d, dt, True, True)


@pytest.mark.parametrize("with_dlse,want_do", [(False, True), (True, False), (False, False)])
def test_merge_bwd_optional_arguments(with_dlse, want_do):
    check(3, 7, 45, 128, "bf16", with_dlse, want_do)


@pytest.mark.parametrize("P", [1, 2, 33, 70])
def test_merge_bwd_partial_counts(P):
    # P = 1 passes the gradients straight through; P > 32 takes several rounds of lanes
    check(20 + P, P, 29, 64, "fp32", True, True)


def test_merge_bwd_zero_rows_and_errors():
    op, lp, g, gl = merge_partials(1, 3, 0, 64)
    do_p, dl_p = skv.lse_merge_bwd(op.cuda(), lp.cuda(), g.cuda(), None)
    assert do_p.numel() == 0 and dl_p.numel() == 0
    op, lp, g, gl = merge_partials(1, 3, 8, 48)
    with pytest.raises(skv.SkvError):
        skv.lse_merge_bwd(op.cuda(), lp.cuda(), g.cuda(), None)     # head_dim 48 is not dispatched


def test_merge_bwd_from_oracle_partials():
    # partials of a real anchor-attention problem (the oracle's Eq. 3 per rank)
    rng = np.random.default_rng(5)
    B, H, d, S, m, P = 4, 2, 64, 512, 128, 4
    s = np.array([0, 0, 0, 256, 256], np.int32)
    a = np.array([100, 250, 256, 300, 512], np.int32)
    q = rng.standard_normal((len(s) * B, H, d))
    k = rng.standard_normal((S, H, d))
    v = rng.standard_normal((S, H, d))
    gO = rng.standard_normal((len(s) * B, H, d))
    op, lp = orc.partition_forward(q, k, v, s, a, B, np.array([0, 1, 2, 3]), m, P)
    t = lambda x: torch.tensor(np.ascontiguousarray(x), dtype=torch.float32).cuda()
    do_p, dl_p = skv.lse_merge_bwd(t(op), t(lp), t(gO), None)
    r_do, r_dl = orc.lse_merge_backward(op.astype(np.float32), lp.astype(np.float32), gO.astype(np.float32))
    assert np.abs(dl_p.cpu().numpy() - r_dl).max() <= TOL_DL
    assert np.abs(do_p.cpu().numpy() - r_do).max() <= TOL_DO * 10


def test_merge_bwd_packed_size():
    # the packed workload's merge: P = 16 partials of Q*H rows, d = 128, bf16 dO
    P, rows, d = PACKED.P, PACKED.Q * PACKED.H, PACKED.d
    op, lp, g, gl = merge_partials(77, P, rows, d, "bf16", frac_empty=0.3, device="cuda")
    do_p, dl_p = skv.lse_merge_bwd(op, lp, g, gl)
    assert skv.stream_status() == 0
    live = torch.isfinite(lp).any(dim=0)
    # sum_p w_p = 1: the partials' gradients add up to the upstream ones
    assert (dl_p.sum(0) - gl)[live].abs().max().item() <= 1e-3
    assert (do_p.sum(0) - g.float())[live].abs().max().item() <= 1e-4 * 8
    assert dl_p[:, ~live].abs().max().item() == 0.0
    idx = torch.randperm(rows, generator=torch.Generator().manual_seed(1))[:400].sort().values
    sel = idx.cuda()
    r_do, r_dl = orc.lse_merge_backward(op[:, sel].cpu().numpy(), lp[:, sel].cpu().numpy(), g[sel].float().cpu().numpy(),
                                        gl[sel].cpu().numpy())
    assert np.abs(dl_p[:, sel].cpu().numpy() - r_dl).max() <= TOL_DL
    assert np.abs(do_p[:, sel].cpu().numpy() - r_do).max() <= TOL_DO * 8
