"""GPU parity where each key tile walks many query tiles: every output element
against the CPU fp64 oracle.

One sample of 16384 context with 256 anchors in its last 3/4 (B = 16, so 32
query tiles of 128 rows): a key tile of the prompt quarter is seen by every
block, so the key-stationary backward walks all 32 query tiles for it, many
times round its operand rings and barrier phases, and the query-stationary
pass walks up to 128 key tiles per query tile.  Checked element by element: o,
lse, dq, dk, dv (multi-head, and a grouped-query variant with four query heads
on one key/value head, which makes the key-stationary walk 4 x 32 tiles long).
Tolerances: bf16 2e-2 (o, dq, dk, dv) and 1e-3 (lse)."""
import pytest

from gpu_helpers import TOL_BF16, TOL_BF16_LSE
from test_gpu_attn import check_backward, check_forward
from workloads import random_small

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("w", [
    random_small(61, 1, 16384, 256, 16, 2, 128, 4096, 4, "bf16", order="lpt"),
    random_small(62, 1, 16384, 256, 16, 4, 128, 4096, 4, "bf16", order="contiguous").with_(Hkv=1),
], ids=["mha_h2", "gqa_h4_kv1"])
def test_long_walks_every_element(w):
    inp, d, prob, roc, o, lse = check_forward(w, TOL_BF16, TOL_BF16_LSE, order=w.order, check_parts=False)
    check_backward(w, inp, d, prob, roc, o, lse, TOL_BF16)
