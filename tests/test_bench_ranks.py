"""The multi-rank rules of bench.py, on CPU with two gloo ranks (127.0.0.1):
every rank runs its own replica (its own seed, same shape), the reported time
is the slowest rank's, and the job's throughput counts the work of every rank
over that time (weak scaling, no collective on the data path)."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
from workloads import PACKED


def _free_port():
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        return sk.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        mine = [10.0 + 5.0 * rank, 3.0 - rank]        # rank 1 is slower on the first, faster on the second
        got = bench.slowest(mine, world, "cpu")
        dist.barrier()
        q.put((rank, got, bench.replica(PACKED, rank).seed))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = {}
    for _ in range(world):
        rank, got, seed = q.get(timeout=120)
        res[rank] = (got, seed)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank in range(world):
        assert res[rank][0] == [15.0, 3.0]           # the maximum of each entry over ranks
    assert res[0][1] == PACKED.seed and res[1][1] != res[0][1]


def test_single_rank_and_job_throughput():
    assert bench.slowest([4.0, 2.0], 1, "cpu") == [4.0, 2.0]
    assert bench.replica(PACKED, 0) is PACKED
    r3 = bench.replica(PACKED, 3)
    assert (r3.S, r3.Q, r3.H, r3.d, r3.P) == (PACKED.S, PACKED.Q, PACKED.H, PACKED.d, PACKED.P)
    # 2 TFLOP per rank-step, 4 ranks, 10 ms for the slowest: 800 TFLOP/s for the job
    assert bench.job_tflops(2e12, 4, 10.0) == pytest.approx(800.0)


def test_merge_bytes_match_the_oracle_count():
    """The bench's merge bytes count the partials it is given, as the oracle's
    count does: the block-local slot kept after the context partials is not
    part of the context merge and must be sliced off by the caller."""
    import numpy as np
    import oracle as orc
    g = torch.Generator().manual_seed(5)
    lse = torch.randn(5, 7, 3, generator=g)
    lse[torch.rand(5, 7, 3, generator=g) < 0.3] = float("-inf")
    for out_b in (2, 4):
        assert bench.merge_algorithmic_bytes(lse[:4], 16, out_b) == orc.merge_bytes(lse[:4].numpy(), 16, out_b)
        assert bench.merge_algorithmic_bytes(lse, 16, out_b) == orc.merge_bytes(lse.numpy(), 16, out_b)
    assert bench.merge_algorithmic_bytes(lse[:4], 16, 2) < bench.merge_algorithmic_bytes(lse, 16, 2)


def test_traffic_digest_follows_code_not_comments(tmp_path, monkeypatch):
    """The digest that gates the captured DRAM traffic ignores comment and
    blank-line edits of the tensor-core kernels' sources and changes with any
    code edit."""
    import shutil
    src = os.path.join(bench.ROOT, "lse_merge_gb300", "csrc")
    dst = tmp_path / "lse_merge_gb300" / "csrc"
    dst.mkdir(parents=True)
    for f in bench.TC_SOURCES:
        shutil.copy(os.path.join(src, f), dst / f)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    base = bench.csrc_digest()
    f0 = dst / bench.TC_SOURCES[0]
    text = f0.read_text()
    f0.write_text("// a reworded comment\n\n/* and a block\n   comment */\n" + text)
    assert bench.csrc_digest() == base
    f0.write_text(text + "\nstatic const int digest_probe = 1;\n")   # one line of code more
    assert bench.csrc_digest() != base


def test_pinned_buffer_check():
    # the default workload's 106 GB of pinned buffers and its 17 GB staging copy fit one
    # rank on a 199 GB box, not eight ranks; an unreadable meminfo does not block the pass
    need, staging = 105_800_000_000, 17_200_000_000
    assert bench.pinned_buffers_fit(need, staging, 1, 190_000_000_000)
    assert not bench.pinned_buffers_fit(need, staging, 8, 900_000_000_000)
    assert bench.pinned_buffers_fit(need, staging, 8, None)
    avail = bench.host_mem_available()
    assert avail is None or avail > 0
