"""GPU parity of the merge with the output projection [Split-KV §4.1, Eq. 5]
against the CPU fp64 oracle (merge_oproj: Eq. 5's sum of the projected
weighted partials) on the same seeded partials and weight: y at the bf16
tolerance 2e-2 (the projection reads the merged o in bf16), o at 2e-2, lse at
1e-3, empty partials and rows with no partial at all included, ragged rows
and output columns, and Table 2's hidden sizes (2048, 5120) over 32 x 128
attention columns."""
import numpy as np
import pytest
import torch

import lse_merge_gb300 as skv
import oracle as orc
from gpu_helpers import TOL_BF16, TOL_BF16_LSE, assert_lse_equal, maxabs
from workloads import merge_partials, oproj_weight

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("P,Q,H,d,d_model", [
    (4, 300, 4, 64, 272),         # ragged rows (300 = 2 x 128 + 44) and columns (256 + 16)
    (1, 128, 2, 128, 256),        # one partial: y = o_0 W_o^T
    (6, 520, 32, 128, 2048),      # Table 2: d_model 2048 over 32 x 128
    (3, 384, 32, 128, 5120),      # Table 2: d_model 5120
    (3, 77, 2, 256, 64),          # head_dim 256, one ragged row tile
])
def test_merge_oproj_matches_oracle(P, Q, H, d, d_model):
    o_part, lse_part, _, _ = merge_partials(900 + Q, P, Q * H, d)
    o_part = o_part.view(P, Q, H, d)
    lse_part = lse_part.view(P, Q, H)
    w = oproj_weight(17 + d_model, d_model, H * d)
    y, o, lse = skv.lse_merge_oproj(o_part.cuda(), lse_part.cuda(), w.cuda())
    assert skv.stream_status() == 0
    r_y, r_l = orc.merge_oproj(o_part, lse_part, w)
    r_o, _ = orc.lse_merge(o_part.double().numpy(), lse_part.double().numpy())
    assert_lse_equal(lse.cpu().numpy(), r_l, TOL_BF16_LSE)
    assert maxabs(o.float().cpu().numpy(), r_o) <= TOL_BF16
    err = maxabs(y.cpu().numpy(), r_y)
    assert err <= TOL_BF16, f"y err {err}"


def test_merge_oproj_twice_same_buffers():
    # a second call into the same buffers gives the same bits (nothing is accumulated)
    o_part, lse_part, _, _ = merge_partials(77, 4, 256 * 4, 128)
    o_part = o_part.view(4, 256, 4, 128).cuda()
    lse_part = lse_part.view(4, 256, 4).cuda()
    w = oproj_weight(5, 512, 512).cuda()
    y1, o1, l1 = skv.lse_merge_oproj(o_part, lse_part, w)
    y1 = y1.clone()
    y2, _, _ = skv.lse_merge_oproj(o_part, lse_part, w, o=o1, lse=l1)
    assert skv.stream_status() == 0
    assert torch.equal(y1, y2)
