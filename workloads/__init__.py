"""Seeded synthetic inputs for the Split-KV anchor-attention path.

This module is shared by the CPU oracle and the CUDA path, and it holds none of
the method's arithmetic: it only draws anchors and tensors.  The workloads stand
in for the paper's evaluation inputs, which were themselves randomly generated
fixed-length samples with a 1:3 prompt-to-response ratio and block size B=16
(Split-KV: Efficient Context Parallelism for Training Diffusion Drafters,
§5.1 "Evaluation protocol").

Reading of the anchor sampling (the paper says "A response positions per
sequence", §3.1, and 1:3 prompt-to-response, §5.1): anchors are integers drawn
uniformly without replacement from the last 3/4 of each sample, sorted
ascending inside the sample; blocks are ordered by (sample, anchor).  Block i of
sample u has s_i = u*L (the sample start) and a_i its anchor.

Draw order for one workload (one torch CPU generator seeded once):
anchors (sample by sample) -> q -> k -> v -> dO.  The block tokens' own keys
and values (the block-local term of the mask) come from a second generator
seeded with seed + 1000003, so adding them changes none of the draws above:
k_blk -> v_blk, [Q, H, d], distributed like q.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    seed: int
    n_samples: int          # b
    sample_len: int         # L (per-sample context length)
    anchors_per_sample: int # A
    anchor_lo: int          # anchors drawn from [s + anchor_lo, s + anchor_hi) ...
    anchor_hi: int          # ... (half-open, offsets inside the sample)
    B: int                  # block size (rows per anchor)
    H: int                  # heads
    d: int                  # head dim
    m: int                  # chunk length
    P: int                  # virtual ranks
    dtype: str              # "fp32" or "bf16"
    qkv_std: float          # q, k, v ~ N(0,1) * qkv_std
    do_std: float           # dO ~ N(0,1) * do_std
    order: str              # "contiguous" or "lpt"
    backward: bool          # whether the workload runs the backward pass
    Hkv: int = 0            # key/value heads (grouped queries); 0 means H

    @property
    def KVH(self) -> int:
        return self.Hkv or self.H

    @property
    def S(self) -> int:
        return self.n_samples * self.sample_len

    @property
    def N(self) -> int:
        return self.n_samples * self.anchors_per_sample

    @property
    def Q(self) -> int:
        return self.N * self.B

    @property
    def n_chunks(self) -> int:
        return self.S // self.m

    @property
    def J(self) -> int:
        return self.n_chunks // self.P

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


def _resp(L: int):
    """Offsets of the response (last 3/4) of a sample of length L."""
    return L // 4, L


# The five evaluation workloads (sizes of the paper's step-time studies, §5):
# q, k, v ~ N(0, 1) * qkv_std and dO ~ N(0, 1) * do_std, as listed below.
TINY_FP32 = Workload("tiny_fp32", 1, 1, 2048, 8, 256, 2049, 16, 4, 64, 512, 4,
                     "fp32", 1.0, 1.0, "contiguous", True)
BF16_FWD = Workload("bf16_fwd", 2, 1, 32768, 64, *_resp(32768), 16, 16, 128, 4096, 8,
                    "bf16", 0.5, 0.5, "contiguous", False)
PACKED = Workload("packed_4x128k", 3, 4, 131072, 512, *_resp(131072), 16, 32, 128, 4096, 16,
                  "bf16", 0.5, 1.0, "lpt", True)
LONG_1M = Workload("long_1m", 4, 1, 1048576, 512, *_resp(1048576), 16, 32, 128, 4096, 64,
                   "bf16", 0.5, 0.5, "lpt", True)


def qs_sweep(ratio: int, order: str = "lpt") -> Workload:
    """Q:S sweep point 1:ratio, ratio in {4, 8, 16, 32}: per-sample context 128k,
    packed queries fixed at 64k (Split-KV §5.4), P=32."""
    assert ratio in (4, 8, 16, 32)
    b = ratio // 2                     # S = 2^17 * b, Q = 2^16  =>  S/Q = 2b
    A = 65536 // 16 // b
    return Workload(f"qs_1to{ratio}_{order}", 5, b, 131072, A, *_resp(131072), 16, 32, 128,
                    4096, 32, "bf16", 0.5, 0.5, order, True)


# A reduced packed case for ncu captures (inputs > L2, a few GB on the device).
PROFILE_SMALL = Workload("profile_1x128k", 6, 1, 131072, 512, *_resp(131072), 16, 8, 128, 4096, 8,
                         "bf16", 0.5, 1.0, "lpt", True)

# Grouped-query layouts of the paper's drafters (Table 2: 32 query heads over 8
# or 4 key/value heads, head dim 128) on the packed shape.
PACKED_KV8 = PACKED.with_(name="packed_4x128k_kv8", Hkv=8)
PACKED_KV4 = PACKED.with_(name="packed_4x128k_kv4", Hkv=4)

WORKLOADS = {w.name: w for w in (TINY_FP32, BF16_FWD, PACKED, LONG_1M, PROFILE_SMALL, PACKED_KV8, PACKED_KV4)}
for _r in (4, 8, 16, 32):
    for _o in ("lpt", "contiguous"):
        _w = qs_sweep(_r, _o)
        WORKLOADS[_w.name] = _w


def draw_anchors(w: Workload, g: torch.Generator):
    """Returns (s, a) as int32 CPU tensors of length N, ordered by (sample, a)."""
    s_list, a_list = [], []
    span = w.anchor_hi - w.anchor_lo
    assert w.anchors_per_sample <= span
    for u in range(w.n_samples):
        start = u * w.sample_len
        pick = torch.randperm(span, generator=g)[: w.anchors_per_sample]
        a_u = torch.sort(pick).values + (start + w.anchor_lo)
        s_list.append(torch.full((w.anchors_per_sample,), start, dtype=torch.int64))
        a_list.append(a_u)
    s = torch.cat(s_list).to(torch.int32)
    a = torch.cat(a_list).to(torch.int32)
    return s, a


@dataclasses.dataclass
class Inputs:
    w: Workload
    s: torch.Tensor          # int32 [N]
    a: torch.Tensor          # int32 [N]
    q: torch.Tensor          # [Q, H, d] fp32 or bf16 (exactly what the GPU receives)
    k: torch.Tensor          # [S, Hkv, d]
    v: torch.Tensor          # [S, Hkv, d]
    dO: Optional[torch.Tensor]  # [Q, H, d] or None


def make_inputs(w: Workload, with_grad: Optional[bool] = None, pin: bool = False,
                device: str = "cpu") -> Inputs:
    """Draws one workload's inputs.  bf16 workloads round the fp32 draws to
    bf16 (round to nearest even); the oracle widens exactly those values to
    fp64.  Anchors always come from the seeded CPU generator; q, k, v, dO come
    from a generator on ``device`` ("cpu", or "cuda" for the large workloads,
    whose host draw would take minutes) -- both sides of a parity check read
    the same tensors, so the device only changes which values are drawn."""
    g = torch.Generator(device="cpu")
    g.manual_seed(w.seed)
    s, a = draw_anchors(w, g)
    tdt = torch.float32 if w.dtype == "fp32" else torch.bfloat16
    if device != "cpu":
        g = torch.Generator(device=device)
        g.manual_seed(w.seed)

    def draw(shape, std):
        out = torch.empty(shape, dtype=tdt, device=device)
        flat = out.view(-1)
        step = 1 << 26                      # bounded fp32 temporaries
        for i in range(0, flat.numel(), step):
            n = min(step, flat.numel() - i)
            x = torch.randn(n, generator=g, dtype=torch.float32, device=device)
            if std != 1.0:
                x.mul_(std)
            flat[i:i + n] = x.to(tdt)
        return out.pin_memory() if (pin and device == "cpu") else out

    q = draw((w.Q, w.H, w.d), w.qkv_std)
    k = draw((w.S, w.KVH, w.d), w.qkv_std)
    v = draw((w.S, w.KVH, w.d), w.qkv_std)
    want = w.backward if with_grad is None else with_grad
    dO = draw((w.Q, w.H, w.d), w.do_std) if want else None
    return Inputs(w, s, a, q, k, v, dO)


def block_kv(w: Workload, device: str = "cpu"):
    """(k_blk, v_blk) [Q, Hkv, d]: the block tokens' own keys and values for the
    block-local term, drawn like q from their own seeded generator."""
    tdt = torch.float32 if w.dtype == "fp32" else torch.bfloat16
    g = torch.Generator(device=device)
    g.manual_seed(w.seed + 1000003)
    out = []
    for _ in range(2):
        x = torch.empty(w.Q, w.KVH, w.d, dtype=tdt, device=device)
        flat = x.view(-1)
        step = 1 << 26
        for i in range(0, flat.numel(), step):
            n = min(step, flat.numel() - i)
            r = torch.randn(n, generator=g, dtype=torch.float32, device=device)
            if w.qkv_std != 1.0:
                r.mul_(w.qkv_std)
            flat[i:i + n] = r.to(tdt)
        out.append(x)
    return out[0], out[1]


def random_small(seed: int, n_samples: int, sample_len: int, anchors_per_sample: int,
                 B: int, H: int, d: int, m: int, P: int, dtype: str = "fp32",
                 anchor_lo: Optional[int] = None, anchor_hi: Optional[int] = None,
                 order: str = "contiguous") -> Workload:
    """A small ad-hoc workload for tests (ragged tails, several tiles)."""
    lo = sample_len // 4 if anchor_lo is None else anchor_lo
    hi = sample_len if anchor_hi is None else anchor_hi
    return Workload(f"small_{seed}", seed, n_samples, sample_len, anchors_per_sample, lo, hi,
                    B, H, d, m, P, dtype, 1.0 if dtype == "fp32" else 0.5, 1.0, order, True)


def merge_partials(seed: int, P: int, rows: int, d: int, do_dtype: str = "fp32", frac_empty: float = 0.2,
                   device: str = "cpu"):
    """Seeded inputs of the merge and its backward: (o_part fp32 [P, rows, d],
    lse_part fp32 [P, rows], dO [rows, d] in do_dtype, dlse fp32 [rows]).
    A share frac_empty of the partials is empty (lse_part = -inf), and the last
    row has every partial empty.  Draw order: o_part -> lse_part -> empty mask ->
    dO -> dlse, one torch generator on `device` (large cases draw on the GPU)."""
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    o_part = torch.randn(P, rows, d, generator=g, device=device)
    lse_part = torch.randn(P, rows, generator=g, device=device) * 3.0
    empty = torch.rand(P, rows, generator=g, device=device) < frac_empty
    if rows > 0:
        empty[:, rows - 1] = True
    lse_part = lse_part.masked_fill(empty, float("-inf"))
    dO = torch.randn(rows, d, generator=g, device=device).to(torch.float32 if do_dtype == "fp32" else torch.bfloat16)
    dlse = torch.randn(rows, generator=g, device=device)
    return o_part, lse_part, dO, dlse


def oproj_weight(seed: int, d_model: int, hd: int, device: str = "cpu") -> torch.Tensor:
    """A seeded synthetic output-projection weight W_o, bf16 [d_model, hd] (the
    drafters' hidden sizes of Split-KV Table 2 are 2048 and 5120 over
    32 x 128 = 4096 attention columns): N(0, 1) / sqrt(hd), so each output has
    the scale of one attention row."""
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    w = torch.randn(d_model, hd, generator=g, device=device) / (hd ** 0.5)
    return w.to(torch.bfloat16)
