#!/usr/bin/env python3
"""Benchmark of the Split-KV anchor-attention hot path on GB300.

One step = one pass of the whole path over one synthetic batch, all through
the C ABI: chunk prices (Eq. 6) -> LPT plan -> per-rank partial attention
(Eq. 3) -> LSE merge (Eq. 4) -> backward (Alg. 1), with the inputs resident in
HBM.  Prints ONE JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the CPU fp64 oracle, timed on the host cores

With N > 1 (torchrun) every rank runs an independent replica of the workload
(weak scaling, no collective on the data path); value = work of all ranks /
the slowest rank's time.
"""
import os

# BLAS threads of the oracle legs: every host core (set before numpy loads).
os.environ.setdefault("OPENBLAS_NUM_THREADS", str(os.cpu_count() or 1))

import argparse
import ctypes
import json
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "anchor-attn fwd+bwd useful TFLOP/s and % BF16 tensor peak; merge HBM GB/s"
UNIT = "TFLOP/s"
DEFAULT_WORKLOAD = "qs_1to32_lpt"   # the largest single-GPU configuration (S = 2M keys, Q = 64k)
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# Sources the three tensor-core attention kernels compile from: the DRAM
# traffic captured for them with ncu holds while these files are unchanged.
TC_SOURCES = ("skv_attn_tc.cu", "skv_attn_bwd_tc.cu", "skv_ptx.cuh", "skv_tc.h", "skv_tc_common.cuh",
              "skv_common.cuh")


def csrc_digest():
    """sha256 over the tensor-core kernels' sources with comments and blank
    lines left out: DRAM-traffic figures captured with ncu are reported only
    while the kernels' code is the code that was captured."""
    import hashlib
    import re
    h = hashlib.sha256()
    d = os.path.join(ROOT, "lse_merge_gb300", "csrc")
    for f in TC_SOURCES:
        with open(os.path.join(d, f), encoding="utf-8") as fh:
            text = fh.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        code = "\n".join(ln.rstrip() for ln in text.splitlines() if ln.strip())
        h.update(f.encode() + b"\0" + code.encode())
    return h.hexdigest()


def merge_algorithmic_bytes(lse_merged, d: int, out_b: int) -> int:
    """HBM bytes of one merge of the partials whose l is lse_merged [P, ...]:
    every l_p, the o_p rows with a finite l_p, and the merged o (out_b bytes an
    element) and l per row."""
    P = lse_merged.shape[0]
    rows = lse_merged[0].numel()
    finite = int(lse_merged.isfinite().sum().item())
    return P * rows * 4 + finite * d * 4 + rows * (d * out_b + 4)


def host_mem_available():
    """MemAvailable of /proc/meminfo in bytes, or None where it cannot be read."""
    try:
        with open("/proc/meminfo", encoding="ascii") as fh:
            for ln in fh:
                if ln.startswith("MemAvailable:"):
                    return int(ln.split()[1]) * 1024
    except (OSError, ValueError, IndexError):
        pass
    return None


def pinned_buffers_fit(need: int, staging: int, ranks_on_node: int, avail) -> bool:
    """Whether every rank of a node can pin its end-to-end buffers (need bytes)
    beside one pageable staging copy, within the node's available host memory
    (None: unknown, assumed to fit)."""
    return avail is None or (need + staging) * ranks_on_node <= avail


def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


# Multi-rank rules of the measurement (weak scaling: one independent replica
# per rank, no collective on the data path).

def replica(w, rank: int):
    """Rank r's replica: the same workload shape with its own seed."""
    return w.with_(seed=w.seed + 1000 * rank) if rank else w


def slowest(values, world: int, device):
    """Per-rank times -> the slowest rank's (the job ends with its last replica)."""
    if world == 1:
        return list(values)
    import torch
    import torch.distributed as dist
    t = torch.tensor(list(values), dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.tolist()]


def job_tflops(flop_per_rank_step: float, world: int, ms: float) -> float:
    """Whole-job throughput: the work of every rank over the slowest rank's time."""
    return flop_per_rank_step * world / (ms * 1e-3) / 1e12


class ClockSampler:
    """nvidia-smi samples (200 ms) of SM clock and throttle reasons."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if not self.proc:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.t:
            self.t.join(timeout=2)
        sms, mx, reasons, watts = [], None, set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sms.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            try:
                watts.append(float(parts[3]))
            except ValueError:
                pass
            for nm, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(nm)
        if not sms:
            return None
        out = {"sm_mhz": statistics.median(sms), "sm_max_mhz": mx, "reasons": sorted(reasons),
               "samples": len(sms)}
        if watts:
            out["power_w"] = statistics.median(watts)
        return out


def useful_pairs_per_head(s, a, B):
    """Unmasked (query, context key) pairs of one head (the block-local B x B
    pairs of each block are counted separately)."""
    return int(B * (a.long() - s.long()).clamp(min=0).sum().item())


# ------------------------------------------------------------------ oracle legs

def oracle_sample(w, inp, budget_s: float, block_offset: int = 0):
    """Times the CPU oracle (as it stands) on a bounded sample of the workload:
    forward (+ backward when the workload has one) of whole query blocks of one
    head, until ~budget_s seconds of work.  A block's window lies inside its own
    sample, so each block is given its sample's keys and values (the oracle's
    mask row covers those L keys; every key outside them is masked for the
    block) and the backward keeps dk, dv of the one key/value head in use.
    Returns (useful TFLOP/s, description, seconds, extrapolated step seconds)."""
    import oracle as orc
    N, L = w.N, w.sample_len
    stride = max(1, N // 64)
    order = [(block_offset + t * stride) % N for t in range(N)]
    head = 0
    s_all, a_all = inp.s.long(), inp.a.long()
    t0 = time.perf_counter()
    pairs = 0
    done = []
    for i in order:
        u0 = int(s_all[i]) // L * L                  # the block's sample: keys [u0, u0 + L)
        k_u, v_u = inp.k[u0:u0 + L], inp.v[u0:u0 + L]
        s_u, a_u = s_all - u0, a_all - u0
        orc.attention_forward(inp.q, k_u, v_u, s_u, a_u, w.B, blocks=[i], heads=[head])
        if w.backward:
            orc.attention_backward(inp.q, k_u, v_u, s_u, a_u, w.B, inp.dO, blocks=[i], heads=[head],
                                   kv_heads_only=True)
        pairs += w.B * max(0, int(inp.a[i]) - int(inp.s[i]))
        done.append(i)
        if time.perf_counter() - t0 >= budget_s:
            break
    dt = time.perf_counter() - t0
    flops = pairs * w.d * (12 if w.backward else 4)
    desc = (f"{len(done)} query blocks (B={w.B} rows each) x head {head} of {w.name}, each over its "
            f"sample's {L} keys, {'fwd+bwd' if w.backward else 'fwd'}, {pairs} useful pairs, {dt:.1f} s")
    # the oracle's cost per (block, head) does not depend on the window (it forms
    # the explicit mask row and the scores over all L keys of the sample), so the
    # whole step scales with the number of (block, head) pairs
    extrap_s = dt * (w.N * w.H) / max(1, len(done))
    return flops / dt / 1e12, desc, dt, extrap_s


def blas_threads():
    v = os.environ.get("OPENBLAS_NUM_THREADS") or os.environ.get("OMP_NUM_THREADS")
    try:
        return int(v)
    except (TypeError, ValueError):
        return os.cpu_count() or 1


def run_planner_study(args):
    """Planner quality and latency on the shapes of the pages' planner study
    [Split-KV §5.5, Figs. 9 and 10]: b = 4 samples with a 1:3 prompt-to-response
    split, anchors at one per 256 context positions in the response (the
    density of the packed workload), B = 16, m = 4096.  Context per sample
    16k..256k at P = 8, then P = 8..64 at 256k.  For LPT, contiguous ("no
    balance") and Zigzag on the GPU: rho = max_p W_p / mean_p W_p with
    W_p = C_p + (N/P) B^2, and the latency of costs + LPT (CUDA events, warm).
    Prints one JSON line per shape."""
    import torch
    import lse_merge_gb300 as skv
    from lse_merge_gb300.build import build
    from workloads import Workload, draw_anchors
    build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    shapes = [(L, 8) for L in (16384, 32768, 65536, 131072, 262144)] + [(262144, P) for P in (16, 32, 64)]
    B, m, b = 16, 4096, 4
    for L, P in shapes:
        A = L // 256
        w = Workload(f"planner_{L // 1024}k_P{P}", 77, b, L, A, L // 4, L, B, 1, 128, m, P, "bf16", 0.5, 1.0,
                     "lpt", False)
        g = torch.Generator().manual_seed(w.seed)
        s, a = draw_anchors(w, g)
        s, a = s.to(dev), a.to(dev)
        prob = skv.Problem(s, a, B, 1, 128, w.S, m, P, torch.bfloat16)
        n = w.n_chunks
        costs = torch.empty(n, dtype=torch.int64, device=dev)
        starts = torch.arange(b, dtype=torch.int32, device=dev) * L
        lens = torch.full((b,), L, dtype=torch.int32, device=dev)
        D = (w.N / P) * B * B

        def rho(load):
            W = load.double() + D
            return float(W.max() / W.mean())

        for _ in range(3):                      # warm-up
            skv.chunk_costs(prob, costs)
            skv.lpt_order(costs, P, w.J)
        reps = 20
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            skv.chunk_costs(prob, costs)
            _, _, load_lpt = skv.lpt_order(costs, P, w.J)
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / reps
        _, _, load_con = skv.contiguous_order(n, P, w.J, costs)
        load_zz = skv.zigzag_loads(prob, starts, lens)
        if skv.stream_status() != 0:
            raise RuntimeError("device status set by the planners")
        print(json.dumps({"study": "planners", "shape": {"context_per_sample": L, "samples": b, "P": P,
                                                         "anchors_per_sample": A, "B": B, "m": m, "J": w.J},
                          "imbalance_pct": {"lpt": 100 * (rho(load_lpt) - 1), "contiguous": 100 * (rho(load_con) - 1),
                                            "zigzag": 100 * (rho(load_zz) - 1)},
                          "plan_ms_costs_plus_lpt": ms}), flush=True)
    return 0


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    from workloads import WORKLOADS, make_inputs
    import torch
    w = WORKLOADS[args.workload]
    # the same draw as our arm (device generator when a GPU is present); the
    # oracle itself runs on the host cores only
    inp = make_inputs(w, device="cuda" if torch.cuda.is_available() else "cpu")
    per_step = []
    for t in range(args.warmup + args.steps):
        tf, desc, dt, _ = oracle_sample(w, inp, args.ref_step_s, block_offset=7 * t)
        if t >= args.warmup:
            per_step.append((tf, dt, desc))
    value = statistics.mean(x[0] for x in per_step)
    ms = statistics.mean(x[1] for x in per_step) * 1e3
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "S": w.S, "Q": w.Q, "H": w.H, "d": w.d, "P": w.P, "order": w.order,
                   "sample": "bounded oracle sample per step"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": blas_threads(), "kind": "oracle",
                         "sample": per_step[-1][2]},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# --------------------------------------------------------------------- our arm

def run_ours(args):
    import torch
    import torch.distributed as dist

    rank, world, local_rank = dist_env()
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    torch.cuda.set_device(local_rank)
    from lse_merge_gb300.build import build
    if rank == 0 or world == 1:
        build()
    if world > 1:
        dist.barrier()
    import lse_merge_gb300 as skv
    from lse_merge_gb300 import _lib
    from workloads import WORKLOADS, block_kv, make_inputs, oproj_weight

    lib = _lib.load()
    w = WORKLOADS[args.workload]
    w = replica(w, rank)                           # independent replica per rank
    dev = torch.device("cuda", local_rank)
    inp = make_inputs(w, with_grad=w.backward, device=str(dev))
    tdt = torch.float32 if w.dtype == "fp32" else torch.bfloat16
    s, a = inp.s.to(dev), inp.a.to(dev)
    q, k, v = inp.q, inp.k, inp.v
    kb, vb = block_kv(w, device=str(dev))       # the block tokens' own keys / values
    dO = inp.dO if w.backward else None
    prob = skv.Problem(s, a, w.B, w.H, w.d, w.S, w.m, w.P, tdt, n_kv_heads=w.Hkv)
    P, Q, H, d = w.P, w.Q, w.H, w.d
    # P rank partials (+ slot P for the block-local partial of the separate pass)
    o_part = torch.empty(P + 1, Q, H, d, dtype=torch.float32, device=dev)
    lse_part = torch.empty(P + 1, Q, H, dtype=torch.float32, device=dev)
    o = torch.empty(Q, H, d, dtype=tdt, device=dev)
    lse = torch.empty(Q, H, dtype=torch.float32, device=dev)
    if w.backward:
        dq = torch.empty(Q, H, d, dtype=torch.float32, device=dev)
        dk = torch.empty(w.S, w.KVH, d, dtype=torch.float32, device=dev)
        dv = torch.empty(w.S, w.KVH, d, dtype=torch.float32, device=dev)
        dkb = torch.empty(Q, w.KVH, d, dtype=torch.float32, device=dev)
        dvb = torch.empty(Q, w.KVH, d, dtype=torch.float32, device=dev)
        ws_b = torch.empty(skv.workspace_bytes(prob, 1), dtype=torch.uint8, device=dev)
    ws_f = torch.empty(skv.workspace_bytes(prob, 0), dtype=torch.uint8, device=dev)
    costs = torch.empty(w.n_chunks, dtype=torch.int64, device=dev)

    def path(ev=None):
        if ev: ev[0].record()
        skv.chunk_costs(prob, costs)
        if w.order == "lpt":
            roc, _, _ = skv.lpt_order(costs, P, w.J)
        else:
            roc, _, _ = skv.contiguous_order(w.n_chunks, P, w.J, costs)
        if ev: ev[1].record()
        skv.attn_fwd(prob, q, k, v, roc, o_part[:P], lse_part[:P], ws_f)
        if ev: ev[2].record()
        skv.lse_merge(o_part[:P], lse_part[:P], o=o, lse=lse)
        if ev: ev[3].record()
        if w.backward:
            skv.attn_bwd(prob, q, k, v, o, lse, dO, roc, dq, dk, dv, ws_b)
        if ev: ev[4].record()
        return roc

    def local_pass(roc):
        # the block-local term of the mask (the first widening past the context
        # path): its partial in slot P, the P + 1 merge, its backward on top of dq
        skv.attn_fwd(prob, q, k, v, roc, o_part[:P], lse_part[:P], ws_f)
        skv.block_local_fwd(prob, q, kb, vb, o_part[P], lse_part[P])
        skv.lse_merge(o_part, lse_part, o=o, lse=lse)
        if w.backward:
            skv.attn_bwd(prob, q, k, v, o, lse, dO, roc, dq, dk, dv, ws_b)
            skv.block_local_bwd(prob, q, kb, vb, o, lse, dO, dq, dkb, dvb)

    kt_names = ["attn_fwd_tc_kernel", "lse_merge_kernel", "attn_bwd_dkdv_tc_kernel", "attn_bwd_dq_tc_kernel",
                "block_local_fwd_kernel", "block_local_bwd_kernel"]
    kt_buf = (ctypes.c_float * 7)()
    for _ in range(args.warmup):
        path()
    torch.cuda.synchronize()
    st = skv.stream_status()
    if st != 0:
        raise RuntimeError(f"device status {st} after warm-up")

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(args.steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local_rank)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    n0 = lib.skv_launch_count()
    clocks.start()
    time.sleep(0.3)
    start.record()
    for t in range(args.steps):
        path(evs[t])
    end.record()
    torch.cuda.synchronize()
    launches = lib.skv_launch_count() - n0
    clk = clocks.stop()
    if world > 1:
        dist.barrier()
    ms = start.elapsed_time(end) / args.steps
    ph = {"plan": [], "fwd": [], "merge": [], "bwd": []}
    for e in evs:
        ph["plan"].append(e[0].elapsed_time(e[1]))
        ph["fwd"].append(e[1].elapsed_time(e[2]))
        ph["merge"].append(e[2].elapsed_time(e[3]))
        ph["bwd"].append(e[3].elapsed_time(e[4]))
    ph = {kk: statistics.mean(vv) for kk, vv in ph.items()}
    ms = slowest([ms], world, dev)[0]
    if skv.stream_status() != 0:
        raise RuntimeError("device status set during the timed region")
    # a short step is bound by its launches: the same step captured once in a CUDA
    # graph and replayed (its own pass, reported beside the eager number)
    graph = None
    if ms < 20.0 and world == 1:
        try:
            gr = torch.cuda.CUDAGraph()
            side = torch.cuda.Stream(device=dev)
            side.wait_stream(torch.cuda.current_stream(dev))
            with torch.cuda.stream(side):
                path()                                  # warm the allocations of the captured stream
            torch.cuda.current_stream(dev).wait_stream(side)
            torch.cuda.synchronize()
            with torch.cuda.graph(gr, capture_error_mode="thread_local"):
                path()
            gr.replay()
            torch.cuda.synchronize()
            g_s, g_e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            g_s.record()
            for _ in range(args.steps):
                gr.replay()
            g_e.record()
            torch.cuda.synchronize()
            if skv.stream_status() != 0:
                raise RuntimeError("device status set by the graph replays")
            g_ms = g_s.elapsed_time(g_e) / args.steps
            graph = {"ms_per_step": g_ms, "value": job_tflops(4.0 * d * useful_pairs_per_head(inp.s, inp.a, w.B) * H
                                                             * (3.0 if w.backward else 1.0), world, g_ms),
                     "mode": "the whole step captured once in a CUDA graph and replayed"}
            del gr
        except Exception as exc:                        # reported, never fatal
            graph = {"error": f"{type(exc).__name__}: {exc}"[:200]}
    # per-kernel durations: the library's own CUDA events on the launching
    # stream, read after each step of a separate pass of the same steps
    kt_ms = [[] for _ in kt_names]
    lib.skv_set_kernel_timing(1)
    n_kt = max(3, min(args.steps, 5))
    for t in range(n_kt):
        roc_t = path()
        if lib.skv_kernel_times(kt_buf, 4) == 0:
            for i in range(4):
                if kt_buf[i] >= 0:
                    kt_ms[i].append(kt_buf[i])
        local_pass(roc_t)
        if lib.skv_kernel_times(kt_buf, 6) == 0:
            for i in (4, 5):
                if kt_buf[i] >= 0:
                    kt_ms[i].append(kt_buf[i])
    lib.skv_set_kernel_timing(0)
    torch.cuda.synchronize()
    # the whole mask (context + block-local term) as one step, outside the headline
    roc_l = path()
    local_pass(roc_l)
    torch.cuda.synchronize()
    if skv.stream_status() != 0:
        raise RuntimeError("device status set by the block-local pass")
    l_s, l_e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    l_s.record()
    for _ in range(n_kt):
        local_pass(roc_l)
    l_e.record()
    torch.cuda.synchronize()
    whole_ms = l_s.elapsed_time(l_e) / n_kt

    # the per-partial merge backward (MERGE_BWD of Alg. 1, the route a multi-GPU
    # build takes) on this step's context partials: timed on its own, not in the step
    # Eq. 5: the merge with the output projection (Table 2's d_model = 2048) on this
    # step's context partials, its own pass
    oproj = None
    if tdt == torch.bfloat16:
        d_model = 2048
        w_o = oproj_weight(w.seed + 11, d_model, H * d, device=str(dev))
        y_o = torch.empty(Q, d_model, dtype=torch.float32, device=dev)
        skv.lse_merge_oproj(o_part[:P], lse_part[:P], w_o, o=o, lse=lse, y=y_o)
        torch.cuda.synchronize()
        lib.skv_set_kernel_timing(1)
        skv.lse_merge_oproj(o_part[:P], lse_part[:P], w_o, o=o, lse=lse, y=y_o)
        g_ms = kt_buf[6] if lib.skv_kernel_times(kt_buf, 7) == 0 and kt_buf[6] >= 0 else None
        lib.skv_set_kernel_timing(0)
        o_s, o_e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        o_s.record()
        for _ in range(n_kt):
            skv.lse_merge_oproj(o_part[:P], lse_part[:P], w_o, o=o, lse=lse, y=y_o)
        o_e.record()
        torch.cuda.synchronize()
        if skv.stream_status() != 0:
            raise RuntimeError("device status set by the merge with the output projection")
        op_ms = o_s.elapsed_time(o_e) / n_kt
        gflop = 2.0 * Q * d_model * H * d
        oproj = {"d_model": d_model, "ms": op_ms, "gemm_ms": g_ms,
                 "gemm_tflops": gflop / (g_ms * 1e-3) / 1e12 if g_ms else None,
                 "route": "Eq. 4 merge into o (bf16), then y = o W_o^T on the tensor cores (one C-ABI call)"}
        del w_o, y_o

    mbwd = None
    if w.backward:
        do_part = torch.empty(P, Q, H, d, dtype=torch.float32, device=dev)
        dlse_part = torch.empty(P, Q, H, dtype=torch.float32, device=dev)
        op_c, lp_c = o_part[:P], lse_part[:P]
        skv.lse_merge_bwd(op_c, lp_c, dO, None, do_part=do_part, dlse_part=dlse_part)
        torch.cuda.synchronize()
        m_s, m_e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        m_s.record()
        for _ in range(n_kt):
            skv.lse_merge_bwd(op_c, lp_c, dO, None, do_part=do_part, dlse_part=dlse_part)
        m_e.record()
        torch.cuda.synchronize()
        if skv.stream_status() != 0:
            raise RuntimeError("device status set by the merge backward")
        mb_ms = m_s.elapsed_time(m_e) / n_kt
        fin_c = int(torch.isfinite(lp_c).sum().item())
        eb_do = 2 if tdt == torch.bfloat16 else 4
        # lse_part and the finite o_part rows, dO in; dlse_part and do_part out
        mb_bytes = P * Q * H * 4 + fin_c * d * 4 + Q * H * d * eb_do + P * Q * H * 4 + P * Q * H * d * 4
        mbwd = {"ms": mb_ms, "bytes": mb_bytes, "gbs": mb_bytes / (mb_ms * 1e-3) / 1e9}
        del do_part, dlse_part
        torch.cuda.empty_cache()

    pairs = useful_pairs_per_head(inp.s, inp.a, w.B) * H
    fwd_flops = 4.0 * d * pairs
    bwd_flops = 8.0 * d * pairs if w.backward else 0.0
    step_flops = fwd_flops + bwd_flops
    value = job_tflops(step_flops, world, ms)
    pk, pk_kind = peaks()
    sustained = pk.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"])
    hbm = pk.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])
    out_b = 2 if tdt == torch.bfloat16 else 4
    merge_bytes = merge_algorithmic_bytes(lse_part[:P], d, out_b)   # the P context partials the step merges
    merge_gbs = merge_bytes / (ph["merge"] * 1e-3) / 1e9
    # credited (useful) FLOP of each main kernel per launch: forward 4d per pair;
    # the backward's 8d per pair (dV, dP, dQ, dK) is credited 6d to the dK/dV
    # kernel (dV, dP, dK) and 2d to the dQ kernel (dQ; its S and dP are recompute)
    credit = {"attn_fwd_tc_kernel": 4.0 * d * pairs, "attn_bwd_dkdv_tc_kernel": 6.0 * d * pairs,
              "attn_bwd_dq_tc_kernel": 2.0 * d * pairs}
    # the block-local kernels are HBM-bound: their algorithmic bytes per launch
    # (q, k_blk, v_blk in, o, lse out; backward also o, dO in and dq read+write,
    # dk_blk, dv_blk out)
    eb = 2 if tdt == torch.bfloat16 else 4
    rows_h = Q * H
    rows_kv = Q * w.KVH                      # k_blk, v_blk, dk_blk, dv_blk rows (grouped heads)
    local_bytes = {"block_local_fwd_kernel": rows_h * (d * eb + d * 4 + 4) + rows_kv * 2 * d * eb,
                   "block_local_bwd_kernel": rows_h * (3 * d * eb + 4 + 2 * d * 4) + rows_kv * (2 * d * eb + 2 * d * 4)}
    kernels = {}
    for i, nm in enumerate(kt_names):
        if kt_ms[i]:
            km = statistics.mean(kt_ms[i])
            kernels[nm] = {"ms": km}
            if nm in credit:
                kernels[nm]["useful_tflops"] = credit[nm] / (km * 1e-3) / 1e12
            if nm in local_bytes:
                kernels[nm]["gbs"] = local_bytes[nm] / (km * 1e-3) / 1e9
    tensor_k = {k: v for k, v in kernels.items() if k in credit}
    dom = max(tensor_k, key=lambda k: tensor_k[k]["ms"]) if tensor_k else None
    dom_tf = tensor_k[dom]["useful_tflops"] if dom else 0.0
    # DRAM bytes of one launch of the dominant kernel, read with ncu on this very
    # workload (profiles/traffic.json); null for a workload without a capture, and
    # once the kernels differ from the ones the counters were taken on
    traffic = None
    tr_path = os.path.join(ROOT, "profiles", "traffic.json")
    if dom and os.path.exists(tr_path):
        with open(tr_path) as f:
            tr = json.load(f)
        per_launch = tr.get("per_launch", {}).get(w.name, {}).get(dom, {}).get("dram_bytes")
        if per_launch and tr.get("csrc_sha256") == csrc_digest():
            traffic = per_launch

    # the CPU baseline before the end-to-end pass: the pinned host buffers of the
    # largest workloads and the oracle's arrays do not fit in host memory together
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        tf, desc, _, extrap_s = oracle_sample(w, inp, args.cpu_budget_s)
        cpu = {"value": tf, "unit": UNIT, "cores": blas_threads(), "kind": "oracle", "sample": desc,
               "extrapolated_full_step_s": extrap_s,
               "extrapolation": f"sample time x (N x H = {w.N} x {w.H}) / blocks sampled: the oracle's "
                                "cost per (block, head) is the same for every block (explicit mask row over "
                                "its sample's L keys); extrapolated, not measured"}

    # end to end through the public API with host buffers (pinned), copies inside
    e2e = None
    e2e_fits = True
    if not args.no_e2e and w.backward:
        # the pinned host buffers of every rank on this node must fit in its free memory
        # (all ranks take the same decision)
        need = sum(x.numel() * x.element_size() for x in (s, a, q, k, v, dO, o, lse, dq, dk, dv))
        staging = max(x.numel() * x.element_size() for x in (q, k, v, dO))   # one pageable copy at a time
        local_world = int(os.environ.get("LOCAL_WORLD_SIZE", str(world)))
        avail = host_mem_available()
        e2e_fits = pinned_buffers_fit(need, staging, local_world, avail)
        if world > 1:
            flag = torch.tensor([1 if e2e_fits else 0], device=dev)
            dist.all_reduce(flag, op=dist.ReduceOp.MIN)
            e2e_fits = bool(flag.item())
        if not e2e_fits:
            e2e = {"skipped": f"the pinned host buffers ({need / 1e9:.0f} GB a rank, {local_world} ranks on this "
                              f"node) exceed the host memory available ({(avail or 0) / 1e9:.0f} GB)"}
    if not args.no_e2e and w.backward and e2e_fits:
        h_o = torch.empty(Q, H, d, dtype=tdt, pin_memory=True)
        h_lse = torch.empty(Q, H, dtype=torch.float32, pin_memory=True)
        h_dq = torch.empty(Q, H, d, dtype=torch.float32, pin_memory=True)
        h_dk = torch.empty(w.S, w.KVH, d, dtype=torch.float32, pin_memory=True)
        h_dv = torch.empty(w.S, w.KVH, d, dtype=torch.float32, pin_memory=True)
        h_in = [(x.cpu().pin_memory(), x) for x in (s, a, q, k, v, dO)]
        h_out = [(o, h_o), (lse, h_lse), (dq, h_dq), (dk, h_dk), (dv, h_dv)]
        bi = sum(x.numel() * x.element_size() for x, _ in h_in)
        bo = sum(x.numel() * x.element_size() for x, _ in h_out)

        def e2e_step():
            for hsrc, ddst in h_in:
                ddst.copy_(hsrc, non_blocking=True)
            path()
            for dsrc, hdst in h_out:
                hdst.copy_(dsrc, non_blocking=True)

        e2e_step()
        torch.cuda.synchronize()
        ke = max(1, min(args.steps, 3))
        t_s, t_e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t_s.record()
        for _ in range(ke):
            e2e_step()
        t_e.record()
        torch.cuda.synchronize()
        serial_ms = t_s.elapsed_time(t_e) / ke

        # pipelined: the inputs and the results each have two device sets (the resident
        # one and a second).  Step t+1's inputs go up on one copy stream while step t
        # computes; step t's results come down on another while step t+1 computes into
        # the other result set.  A set is reused two steps later, once its inputs have
        # been read and its results are down.  Every step still copies all of its
        # inputs in and all of its results out.
        names_in = ("s", "a", "q", "k", "v", "dO")
        in_sets = [dict(zip(names_in, (s, a, q, k, v, dO)))]
        in_sets.append({nm: torch.empty_like(x) for nm, x in in_sets[0].items()})
        probs = [skv.Problem(st["s"], st["a"], w.B, H, d, w.S, w.m, P, tdt, n_kv_heads=w.Hkv) for st in in_sets]
        h_src = [hsrc for hsrc, _ in h_in]
        out_sets = [(o, lse, dq, dk, dv)]
        out_sets.append(tuple(torch.empty_like(x) for x in out_sets[0]))
        h_dst = (h_o, h_lse, h_dq, h_dk, h_dv)
        up, down = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
        comp = torch.cuda.current_stream(dev)
        ev_in = [torch.cuda.Event() for _ in range(2)]
        ev_used = [torch.cuda.Event() for _ in range(2)]
        ev_done = [torch.cuda.Event() for _ in range(2)]
        ev_down = [torch.cuda.Event() for _ in range(2)]

        def pipelined(n_steps):
            for t in range(n_steps):
                b = t % 2
                st, pr = in_sets[b], probs[b]
                o_b, lse_b, dq_b, dk_b, dv_b = out_sets[b]
                with torch.cuda.stream(up):
                    up.wait_event(ev_used[b])            # step t-2 has finished with these inputs
                    for hs, nm in zip(h_src, names_in):
                        st[nm].copy_(hs, non_blocking=True)
                    ev_in[b].record(up)
                comp.wait_event(ev_in[b])
                skv.chunk_costs(pr, costs)
                if w.order == "lpt":
                    roc_s, _, _ = skv.lpt_order(costs, P, w.J)
                else:
                    roc_s, _, _ = skv.contiguous_order(w.n_chunks, P, w.J, costs)
                skv.attn_fwd(pr, st["q"], st["k"], st["v"], roc_s, o_part[:P], lse_part[:P], ws_f)
                comp.wait_event(ev_down[b])              # step t-2's results are down
                skv.lse_merge(o_part[:P], lse_part[:P], o=o_b, lse=lse_b)
                skv.attn_bwd(pr, st["q"], st["k"], st["v"], o_b, lse_b, st["dO"], roc_s, dq_b, dk_b, dv_b, ws_b)
                ev_used[b].record(comp)
                ev_done[b].record(comp)
                with torch.cuda.stream(down):
                    down.wait_event(ev_done[b])
                    for dsrc, hdst in zip(out_sets[b], h_dst):
                        hdst.copy_(dsrc, non_blocking=True)
                    ev_down[b].record(down)
            comp.wait_stream(up)
            comp.wait_stream(down)

        pipelined(2)
        torch.cuda.synchronize()
        kp = max(2, args.steps)                  # the same K steps as the device-timed line
        t_s.record()
        pipelined(kp)
        t_e.record()
        torch.cuda.synchronize()
        if skv.stream_status() != 0:
            raise RuntimeError("device status set during the end-to-end pass")
        e_ms = t_s.elapsed_time(t_e) / kp
        # Every step had the same inputs, and the kernels are deterministic: the last
        # step's host copies equal its device set, and both device sets agree (bit for
        # bit, on rows sampled evenly over each result).
        b_last = (kp - 1) % 2
        for x0, x1, hx in zip(out_sets[0], out_sets[1], h_dst):
            idx = torch.linspace(0, x0.shape[0] - 1, steps=min(x0.shape[0], 4096)).long()
            idx_d = idx.to(dev)
            got = (x0, x1)[b_last][idx_d].cpu()
            if not (torch.equal(got, hx[idx]) and torch.equal(x0[idx_d], x1[idx_d])):
                raise RuntimeError("end-to-end results differ from the device-resident results")
        del in_sets, probs, out_sets, h_in, h_src, h_dst, h_out, h_o, h_lse, h_dq, h_dk, h_dv
        e_ms, serial_ms = slowest([e_ms, serial_ms], world, dev)
        e2e = {"value": job_tflops(step_flops, world, e_ms), "unit": UNIT, "ms_per_step": e_ms,
               "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo,
               "mode": f"pipelined over {kp} steps: step t+1's inputs go up on one copy stream while "
                       "step t computes, step t's results come down on another while step t+1 computes "
                       "(two device sets of inputs and of results, each reused two steps later); the "
                       "first upload and the last download are inside the timed region",
               "serial": {"ms_per_step": serial_ms, "value": job_tflops(step_flops, world, serial_ms)}}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16" if tdt == torch.bfloat16 else "f32", "data": "synthetic",
            "config": {"workload": w.name, "b": w.n_samples, "S": w.S, "Q": w.Q, "B": w.B, "H": H, "Hkv": w.KVH,
                       "d": d,
                       "m": w.m, "P": P, "J": w.J, "order": w.order,
                       "l2": "inputs larger than L2 (K+V alone exceed 129 MB)",
                       "mask": "context windows (block-local term: block_local object)",
                       "parallelism": f"{world} independent replica(s)"},
            "pct_bf16_peak": {"measured_sustained": value / world / sustained,
                              "nominal_2250": value / world / 2250.0},
            "phases_ms": ph,
            "useful_tflop_per_step": step_flops / 1e12,
            "fa_convention": ({"label": "secondary: FlashAttention convention, backward credited 10 d FLOP per "
                                        "pair (its recomputed Q K^T counted), forward 4 d",
                               "tflop_per_step": (fwd_flops + 10.0 * d * pairs) / 1e12,
                               "value": job_tflops(fwd_flops + 10.0 * d * pairs, world, ms)}
                              if w.backward else None),
            "merge": {"gbs": merge_gbs, "bytes": merge_bytes, "frac_of_hbm": merge_gbs / hbm,
                      "peak_gbs": hbm, "peak_kind": pk_kind},
            "roofline": {"kernel": dom, "bound": "tensor", "achieved": dom_tf,
                         "peak": sustained, "unit": "TFLOP/s", "frac": dom_tf / sustained,
                         "peak_kind": f"{pk_kind} sustained bf16", "traffic": traffic},
            "kernels": kernels,
            "block_local": {"term": "each block's rows over its own B keys (one more merged partial)",
                            "whole_mask_ms_per_step": whole_ms,
                            "fwd": kernels.get("block_local_fwd_kernel"),
                            "bwd": kernels.get("block_local_bwd_kernel")},
            "merge_oproj": oproj,
            "merge_bwd": (dict(mbwd, frac_of_hbm=mbwd["gbs"] / hbm, peak_kind=pk_kind,
                               route="per-partial MERGE_BWD on this step's partials (own pass)")
                          if mbwd else None),
            "gpu_launches": int(launches),
            "cuda_graph": graph,
            "clocks": clk,
            "e2e": e2e,
            "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--cpu-budget-s", type=float, default=15.0)
    ap.add_argument("--ref-step-s", type=float, default=4.0)
    ap.add_argument("--study", choices=["planners"], default=None,
                    help="instead of the step benchmark: the planner rho / latency study")
    args = ap.parse_args()
    if args.study == "planners":
        return run_planner_study(args)
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
