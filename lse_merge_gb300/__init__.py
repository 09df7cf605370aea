"""lse_merge_gb300 -- Split-KV anchor-sampled attention on one GB300 (sm_103a).

Thin Python binding of libskv (include/skv.h): every function below marshals
torch tensors (device memory) and the current CUDA stream into one C-ABI call;
all arithmetic runs in the library's CUDA kernels.  There is no CPU fallback:
a missing libskv.so raises.

Method: "Split-KV: Efficient Context Parallelism for Training Diffusion
Drafters" -- chunk prices (§4.2 Eq. 6), cost-aware LPT (§4.2), per-rank
partial attention (§4.1 Eq. 3), LSE merge (§4.1 Eq. 4), backward (Alg. 1).
"""
from __future__ import annotations

import ctypes
from typing import Optional, Tuple

import torch

from . import _lib
from ._lib import SKV_BF16, SKV_FP32, SkvProblem

__all__ = ["SkvError", "Problem", "chunk_costs", "lpt_order", "contiguous_order", "zigzag_loads",
           "workspace_bytes", "attn_fwd", "attn_fwd_static", "lse_merge", "lse_merge_bwd", "lse_merge_oproj", "attn_bwd", "stream_status", "set_wait_limit",
           "forward", "plan", "block_local_fwd", "block_local_bwd"]


class SkvError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what}: {_lib.load().skv_status_str(code).decode()} (status {code})")


def _check(code: int, what: str):
    if code != 0:
        raise SkvError(code, what)


def _stream() -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensor must live on the GPU")
    if not t.is_contiguous():
        raise ValueError("tensor must be contiguous")
    return t.data_ptr()


def _dtype_code(dt: torch.dtype) -> int:
    if dt == torch.float32:
        return SKV_FP32
    if dt == torch.bfloat16:
        return SKV_BF16
    raise ValueError(f"unsupported dtype {dt}")


class Problem:
    """One anchor-attention problem (struct skv_problem).  s, a: int32 device
    tensors [N] (sample start and anchor of each block)."""

    def __init__(self, s: torch.Tensor, a: torch.Tensor, B: int, n_heads: int, head_dim: int, S: int, m: int,
                 P: int, dtype: torch.dtype = torch.bfloat16, scale: float = 0.0, n_kv_heads: int = 0):
        if s.dtype != torch.int32 or a.dtype != torch.int32:
            raise ValueError("anchors must be int32")
        if s.numel() != a.numel():
            raise ValueError("s and a differ in length")
        n_chunks = S // m
        J = n_chunks // P if P else 0
        self.s, self.a = s, a          # keep the device buffers alive
        self.B, self.N, self.H, self.d, self.S, self.m, self.P, self.J = B, s.numel(), n_heads, head_dim, S, m, P, J
        self.Hkv = n_kv_heads or n_heads     # heads of k, v, dk, dv (grouped-query layouts)
        self.dtype = dtype
        self.c = SkvProblem(B, s.numel(), n_heads, head_dim, S, m, P, J,
                            _ptr(s) if s.numel() else None, _ptr(a) if a.numel() else None,
                            _dtype_code(dtype), float(scale), int(n_kv_heads))

    @property
    def Q(self) -> int:
        return self.N * self.B

    @property
    def n_chunks(self) -> int:
        return self.S // self.m

    def ref(self):
        return ctypes.byref(self.c)


def chunk_costs(prob: Problem, out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """c_j of Eq. 6 for every chunk (int64 [S/m])."""
    dev = prob.s.device
    out = torch.empty(prob.n_chunks, dtype=torch.int64, device=dev) if out is None else out
    _check(_lib.load().skv_chunk_costs(prob.ref(), _ptr(out), _stream()), "skv_chunk_costs")
    return out


def lpt_order(costs: torch.Tensor, P: int, J: int) -> Tuple[torch.Tensor, torch.Tensor, torch.Tensor]:
    """Cost-aware LPT: (rank_of_chunk int32, order int32 rank-major, load int64 [P])."""
    n = costs.numel()
    roc = torch.empty(n, dtype=torch.int32, device=costs.device)
    order = torch.empty(n, dtype=torch.int32, device=costs.device)
    load = torch.empty(P, dtype=torch.int64, device=costs.device)
    _check(_lib.load().skv_lpt_order(_ptr(costs), n, P, J, _ptr(roc), _ptr(order), _ptr(load), _stream()),
           "skv_lpt_order")
    return roc, order, load


def contiguous_order(n_chunks: int, P: int, J: int, costs: Optional[torch.Tensor] = None,
                     device="cuda") -> Tuple[torch.Tensor, torch.Tensor, Optional[torch.Tensor]]:
    dev = costs.device if costs is not None else torch.device(device)
    roc = torch.empty(n_chunks, dtype=torch.int32, device=dev)
    order = torch.empty(n_chunks, dtype=torch.int32, device=dev)
    load = torch.empty(P, dtype=torch.int64, device=dev) if costs is not None else None
    _check(_lib.load().skv_contiguous_order(_ptr(costs), n_chunks, P, J, _ptr(roc), _ptr(order), _ptr(load),
                                            _stream()), "skv_contiguous_order")
    return roc, order, load


def zigzag_loads(prob: Problem, sample_start: torch.Tensor, sample_len: torch.Tensor) -> torch.Tensor:
    load = torch.empty(prob.P, dtype=torch.int64, device=prob.s.device)
    _check(_lib.load().skv_zigzag_loads(prob.ref(), _ptr(sample_start), _ptr(sample_len), sample_start.numel(),
                                        _ptr(load), _stream()), "skv_zigzag_loads")
    return load


def workspace_bytes(prob: Problem, which: int) -> int:
    return int(_lib.load().skv_workspace_bytes(prob.ref(), which))


def _workspace(prob: Problem, which: int, ws: Optional[torch.Tensor]) -> torch.Tensor:
    need = workspace_bytes(prob, which)
    if need == 0:
        raise SkvError(_lib.SKV_ERR_INVALID_ARG, "skv_workspace_bytes")
    if ws is None or ws.numel() < need:
        ws = torch.empty(need, dtype=torch.uint8, device=prob.s.device)
    return ws


def attn_fwd(prob: Problem, q, k, v, rank_of_chunk, o_part=None, lse_part=None, workspace=None):
    """Per-rank partials (o_part fp32 [P,Q,H,d], lse_part fp32 [P,Q,H]) of Eq. 3."""
    dev = q.device
    if o_part is None:
        o_part = torch.empty(prob.P, prob.Q, prob.H, prob.d, dtype=torch.float32, device=dev)
    if lse_part is None:
        lse_part = torch.empty(prob.P, prob.Q, prob.H, dtype=torch.float32, device=dev)
    ws = _workspace(prob, 0, workspace)
    _check(_lib.load().skv_attn_fwd(prob.ref(), _ptr(q), _ptr(k), _ptr(v), _ptr(rank_of_chunk), _ptr(o_part),
                                    _ptr(lse_part), _ptr(ws), ws.numel(), _stream()), "skv_attn_fwd")
    return o_part, lse_part


def attn_fwd_static(prob: Problem, q, k, v, rank_of_chunk, o_part=None, lse_part=None):
    """attn_fwd without a workspace: the library's fixed device scratch is used
    instead, for callers that must not allocate device memory.  Calls that
    overlap on the GPU race on that shared scratch."""
    dev = q.device
    if o_part is None:
        o_part = torch.empty(prob.P, prob.Q, prob.H, prob.d, dtype=torch.float32, device=dev)
    if lse_part is None:
        lse_part = torch.empty(prob.P, prob.Q, prob.H, dtype=torch.float32, device=dev)
    _check(_lib.load().skv_attn_fwd_static(prob.ref(), _ptr(q), _ptr(k), _ptr(v), _ptr(rank_of_chunk),
                                           _ptr(o_part), _ptr(lse_part), _stream()), "skv_attn_fwd_static")
    return o_part, lse_part


def lse_merge(o_part: torch.Tensor, lse_part: torch.Tensor, out_dtype: torch.dtype = torch.float32,
              o: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None):
    """Eq. 4 over the leading (rank) dimension: returns (o, lse)."""
    P = o_part.shape[0]
    d = o_part.shape[-1]
    rows = lse_part[0].numel()
    if o is None:
        o = torch.empty(o_part.shape[1:], dtype=out_dtype, device=o_part.device)
    if lse is None:
        lse = torch.empty(lse_part.shape[1:], dtype=torch.float32, device=o_part.device)
    _check(_lib.load().skv_lse_merge(_ptr(o_part), _ptr(lse_part), P, rows, d, _ptr(o), _dtype_code(o.dtype),
                                     _ptr(lse), _stream()), "skv_lse_merge")
    return o, lse


def lse_merge_oproj(o_part: torch.Tensor, lse_part: torch.Tensor, w_o: torch.Tensor,
                    o: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                    y: Optional[torch.Tensor] = None):
    """Eq. 5: the merge of the partials [P, Q, H, d] and the output projection
    y = o W_o^T (w_o bf16 [d_model, H*d]).  Returns (y fp32 [Q, d_model],
    o bf16 [Q, H, d], lse fp32 [Q, H])."""
    P, Q, H, d = o_part.shape
    d_model = w_o.shape[0]
    dev = o_part.device
    o = torch.empty(Q, H, d, dtype=torch.bfloat16, device=dev) if o is None else o
    lse = torch.empty(Q, H, dtype=torch.float32, device=dev) if lse is None else lse
    y = torch.empty(Q, d_model, dtype=torch.float32, device=dev) if y is None else y
    if w_o.dtype != torch.bfloat16 or o.dtype != torch.bfloat16 or y.dtype != torch.float32:
        raise ValueError("w_o and o are bf16, y is fp32")
    _check(_lib.load().skv_lse_merge_oproj(_ptr(o_part), _ptr(lse_part), P, Q, H, d, _ptr(w_o), d_model, _ptr(o),
                                           _ptr(lse), _ptr(y), _stream()), "skv_lse_merge_oproj")
    return y, o, lse


def lse_merge_bwd(o_part: torch.Tensor, lse_part: torch.Tensor, dO: torch.Tensor, dlse: Optional[torch.Tensor] = None,
                  want_do_part: bool = True, do_part: Optional[torch.Tensor] = None,
                  dlse_part: Optional[torch.Tensor] = None):
    """Per-partial backward of Eq. 4 (MERGE_BWD): returns (do_part or None, dlse_part)."""
    P = o_part.shape[0]
    d = o_part.shape[-1]
    rows = lse_part[0].numel()
    if do_part is None and want_do_part:
        do_part = torch.empty(o_part.shape, dtype=torch.float32, device=o_part.device)
    if dlse_part is None:
        dlse_part = torch.empty(lse_part.shape, dtype=torch.float32, device=o_part.device)
    _check(_lib.load().skv_lse_merge_bwd(_ptr(o_part), _ptr(lse_part), P, rows, d, _ptr(dO), _dtype_code(dO.dtype),
                                         _ptr(dlse), _ptr(do_part), _ptr(dlse_part), _stream()),
           "skv_lse_merge_bwd")
    return do_part, dlse_part


def attn_bwd(prob: Problem, q, k, v, o, lse, dO, rank_of_chunk, dq=None, dk=None, dv=None, workspace=None):
    """(dq, dk, dv) fp32 of L = sum(dO * o)."""
    dev = k.device
    dq = torch.empty(prob.Q, prob.H, prob.d, dtype=torch.float32, device=dev) if dq is None else dq
    dk = torch.empty(prob.S, prob.Hkv, prob.d, dtype=torch.float32, device=dev) if dk is None else dk
    dv = torch.empty(prob.S, prob.Hkv, prob.d, dtype=torch.float32, device=dev) if dv is None else dv
    ws = _workspace(prob, 1, workspace)
    _check(_lib.load().skv_attn_bwd(prob.ref(), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dO),
                                    _ptr(rank_of_chunk), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(ws), ws.numel(),
                                    _stream()), "skv_attn_bwd")
    return dq, dk, dv


def block_local_fwd(prob: Problem, q, k_blk, v_blk, o_loc=None, lse_loc=None):
    """(o_loc fp32 [Q,H,d], lse_loc fp32 [Q,H]): each block's rows over its own B keys,
    one more partial for lse_merge."""
    dev = q.device
    o_loc = torch.empty(prob.Q, prob.H, prob.d, dtype=torch.float32, device=dev) if o_loc is None else o_loc
    lse_loc = torch.empty(prob.Q, prob.H, dtype=torch.float32, device=dev) if lse_loc is None else lse_loc
    _check(_lib.load().skv_block_local_fwd(prob.ref(), _ptr(q), _ptr(k_blk), _ptr(v_blk), _ptr(o_loc),
                                           _ptr(lse_loc), _stream()), "skv_block_local_fwd")
    return o_loc, lse_loc


def block_local_bwd(prob: Problem, q, k_blk, v_blk, o, lse, dO, dq, dk_blk=None, dv_blk=None):
    """Adds the block-local part to dq (fp32, holding the context part) and returns
    (dq, dk_blk, dv_blk); o, lse are the merged results of the whole mask."""
    dev = q.device
    dk_blk = torch.empty(prob.Q, prob.Hkv, prob.d, dtype=torch.float32, device=dev) if dk_blk is None else dk_blk
    dv_blk = torch.empty(prob.Q, prob.Hkv, prob.d, dtype=torch.float32, device=dev) if dv_blk is None else dv_blk
    _check(_lib.load().skv_block_local_bwd(prob.ref(), _ptr(q), _ptr(k_blk), _ptr(v_blk), _ptr(o), _ptr(lse),
                                           _ptr(dO), _ptr(dq), _ptr(dk_blk), _ptr(dv_blk), _stream()),
           "skv_block_local_bwd")
    return dq, dk_blk, dv_blk


def stream_status() -> int:
    """Synchronises the current stream; returns and clears the device status word."""
    return int(_lib.load().skv_stream_status(_stream()))


def set_wait_limit(limit: int) -> None:
    _check(_lib.load().skv_set_wait_limit(int(limit)), "skv_set_wait_limit")


def plan(prob: Problem, order: str = "lpt"):
    """Eq. 6 prices and a chunk assignment: (costs, rank_of_chunk, order, load)."""
    costs = chunk_costs(prob)
    if order == "lpt":
        roc, ordr, load = lpt_order(costs, prob.P, prob.J)
    elif order == "contiguous":
        roc, ordr, load = contiguous_order(prob.n_chunks, prob.P, prob.J, costs)
    else:
        raise ValueError(order)
    return costs, roc, ordr, load


def forward(prob: Problem, q, k, v, order: str = "lpt"):
    """Whole forward path: prices, plan, per-rank partials, merge -> (o, lse, plan)."""
    costs, roc, ordr, load = plan(prob, order)
    o_part, lse_part = attn_fwd(prob, q, k, v, roc)
    o, lse = lse_merge(o_part, lse_part, out_dtype=q.dtype)
    return o, lse, (costs, roc, ordr, load)
