"""Plain, slow, fp64 CPU definitions of the Split-KV anchor-attention path.

TEST INFRASTRUCTURE ONLY: imported by tests, by ``__graft_entry__.smoke()``
and by the CPU-baseline leg of ``bench.py``; never by the product path.

Source: "Split-KV: Efficient Context Parallelism for Training Diffusion
Drafters" (Zhang, Zhang, Xie, Fan, You), cited below as [Split-KV ...].

Notation (paper's): B block size, N blocks, Q = N*B query rows, S packed
context, H heads, d head dim, m chunk length, P ranks, J chunks per rank,
anchor metadata A = {(s_i, a_i)}.  Query row r belongs to block floor(r/B).
Tensors: q, dO [Q, H, d]; k, v [S, Hkv, d] (Hkv = H, or fewer key/value heads
in a grouped-query layout, see kv_head); outputs o [Q, H, d], lse [Q, H].

Everything here is written as the definition reads: the mask is materialised
as an explicit boolean row over all S context keys, the softmax is the
textbook max-shifted one, and no blocking beyond "the B rows of one block share
one mask row" is applied (rows are independent in the definition).

Parity status: every function is pinned (tests/test_oracle_pins.py).
"""
from __future__ import annotations

import math
from typing import Iterable, Optional, Sequence

import numpy as np

NEG_INF = -np.inf


def _np64(x) -> np.ndarray:
    """torch tensor (any dtype, incl. bf16) or array -> float64 numpy (exact widening)."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            return x.detach().to("cpu").double().numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.asarray(x, dtype=np.float64)


def _npi(x) -> np.ndarray:
    try:
        import torch
        if isinstance(x, torch.Tensor):
            return x.detach().to("cpu").to(torch.int64).numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.asarray(x, dtype=np.int64)


# ---------------------------------------------------------------------------
# Planning: per-position load, chunk cost, LPT, baselines, imbalance
# ---------------------------------------------------------------------------

def anchor_profile(s, a, B: int, S: int) -> np.ndarray:
    """Per-position context load c_anchor(x) = B * sum_i 1[s_i <= x < a_i]
    for x in [0, S)  [Split-KV §3.3, Eq. 2].  int64."""
    s, a = _npi(s), _npi(a)
    c = np.zeros(S, dtype=np.int64)
    for si, ai in zip(s.tolist(), a.tolist()):
        if ai > si:
            c[si:ai] += B
    return c


def rank_load(profile: np.ndarray, keys: Iterable[int]) -> int:
    """C_p = sum of c_anchor(x) over the context positions K_p of rank p
    [Split-KV §3.3]."""
    return int(sum(int(profile[x]) for x in keys))


def chunk_costs(s, a, B: int, S: int, m: int) -> np.ndarray:
    """Chunk price, closed form  c_j = B * sum_i (min(a_i, l_j + m) - max(s_i, l_j))^+
    with l_j = j*m the chunk's left bound, for j < S/m  [Split-KV §4.2, Eq. 6].
    int64."""
    s, a = _npi(s), _npi(a)
    n = S // m
    out = np.zeros(n, dtype=np.int64)
    for j in range(n):
        lam = j * m
        overlap = np.minimum(a, lam + m) - np.maximum(s, lam)
        out[j] = B * int(np.clip(overlap, 0, None).sum())
    return out


def chunk_costs_from_profile(s, a, B: int, S: int, m: int) -> np.ndarray:
    """The same prices obtained the second way: summing the Eq. 2 profile over
    each chunk's positions [Split-KV §3.3 Eq. 2 with §4.2 chunks]."""
    prof = anchor_profile(s, a, B, S)
    return prof[: (S // m) * m].reshape(S // m, m).sum(axis=1)


def lpt_assign(costs, P: int, J: int):
    """Cost-aware LPT [Split-KV §4.2 "Cost-aware LPT"]: take chunks from the
    costliest down; give each to the least-loaded rank that still holds fewer
    than J chunks.  Tie-breaks (unstated on the page): equal costs are taken
    in ascending chunk index; equal loads go to the lowest rank index.  The
    final locality matching is the identity (bundle p stays on rank p).

    Returns (rank_of_chunk int32[n], order int32[P*J] rank-major in assignment
    order, load int64[P])."""
    costs = [int(c) for c in _npi(costs).tolist()]
    n = len(costs)
    if n != P * J:
        raise ValueError("LPT needs exactly P*J chunks")
    by_cost = sorted(range(n), key=lambda j: (-costs[j], j))
    load = [0] * P
    held = [0] * P
    bundles = [[] for _ in range(P)]
    rank_of_chunk = [-1] * n
    for j in by_cost:
        best = -1
        for p in range(P):
            if held[p] < J and (best < 0 or load[p] < load[best]):
                best = p
        rank_of_chunk[j] = best
        load[best] += costs[j]
        held[best] += 1
        bundles[best].append(j)
    order = [j for p in range(P) for j in bundles[p]]
    return (np.asarray(rank_of_chunk, np.int32), np.asarray(order, np.int32),
            np.asarray(load, np.int64))


def contiguous_assign(n_chunks: int, P: int, J: int, costs=None):
    """"No balance" baseline: contiguous chunks, rank p gets chunks
    [pJ, (p+1)J)  [Split-KV §5.1 Baselines].  Returns the same triple as
    lpt_assign (load is zeros when costs is None)."""
    if n_chunks != P * J:
        raise ValueError("need exactly P*J chunks")
    rank_of_chunk = np.asarray([j // J for j in range(n_chunks)], np.int32)
    order = np.arange(n_chunks, dtype=np.int32)
    load = np.zeros(P, np.int64)
    if costs is not None:
        c = _npi(costs)
        for j in range(n_chunks):
            load[j // J] += int(c[j])
    return rank_of_chunk, order, load


def zigzag_loads(profile: np.ndarray, sample_starts: Sequence[int],
                 sample_lens: Sequence[int], P: int) -> np.ndarray:
    """Zigzag baseline: each sample is cut independently into 2P equal chunks
    Z_0..Z_{2P-1}; rank p receives Z_p and Z_{2P-1-p} of every sample
    [Split-KV §4.2 "A concrete example", Fig. 5b].  Returns C_p (int64[P])."""
    load = np.zeros(P, np.int64)
    for st, L in zip(sample_starts, sample_lens):
        if L % (2 * P):
            raise ValueError("sample length must split into 2P chunks")
        w = L // (2 * P)
        for p in range(P):
            for z in (p, 2 * P - 1 - p):
                load[p] += int(profile[st + z * w: st + (z + 1) * w].sum())
    return load


def imbalance(loads, N: int, P: int, B: int) -> float:
    """rho = max_p W_p / mean_p W_p with W_p = C_p + D, D = (N/P) B^2
    [Split-KV §4.2, last paragraph before "A concrete example"]."""
    D = (N / P) * B * B
    W = np.asarray(_npi(loads), np.float64) + D
    return float(W.max() / W.mean())


def useful_pairs(s, a, B: int) -> int:
    """Unmasked context (query, key) pairs per head: B * sum_i (a_i - s_i),
    the context term of T_attn [Split-KV §4.1, last paragraph]."""
    s, a = _npi(s), _npi(a)
    return int(B * np.clip(a - s, 0, None).sum())


# ---------------------------------------------------------------------------
# Attention: the mask, local partial attention, the LSE merge, the backward
# ---------------------------------------------------------------------------

def mask_row(s_i: int, a_i: int, S: int) -> np.ndarray:
    """Boolean context mask of block i's rows: key x is visible iff
    s_i <= x < a_i (the context window W_i)  [Split-KV §3.1, Fig. 1]."""
    row = np.zeros(S, dtype=bool)
    if a_i > s_i:
        row[max(s_i, 0):min(a_i, S)] = True
    return row


def chunk_key_mask(rank_of_chunk, p: int, m: int, S: int) -> np.ndarray:
    """K_p as a boolean row: the positions of the chunks [j*m, (j+1)*m) held by
    rank p [Split-KV §4.2]."""
    roc = _npi(rank_of_chunk)
    keys = np.zeros(S, dtype=bool)
    for j in range(len(roc)):
        if roc[j] == p:
            keys[j * m:(j + 1) * m] = True
    return keys


def kv_head(h: int, H: int, Hkv: int) -> int:
    """Grouped-query layouts [Split-KV Table 2: 32 query heads over 4 or 8
    key/value heads]: query head h attends with key/value head h // (H / Hkv);
    with Hkv = H this is the identity."""
    return h // (H // Hkv)


class _Heads:
    """Per-head fp64 copies of k, v (converted lazily, one head at a time),
    indexed by query head (k, v may hold fewer, grouped, heads)."""

    def __init__(self, k, v, H: Optional[int] = None):
        self.k, self.v = k, v
        self.H = k.shape[1] if H is None else H
        self._h, self._kh, self._vh = None, None, None

    def head(self, h):
        return kv_head(h, self.H, self.k.shape[1])

    def get(self, h):
        c = self.head(h)
        if self._h != c:
            self._kh = _np64(self.k[:, c, :])
            self._vh = _np64(self.v[:, c, :])
            self._h = c
        return self._kh, self._vh


def _softmax_stats(z: np.ndarray):
    """Textbook max-shifted log-sum-exp of each row of z (masked entries -inf).
    Rows that are entirely -inf get lse = -inf and weights 0."""
    mx = z.max(axis=1)
    empty = ~np.isfinite(mx)
    mx_safe = np.where(empty, 0.0, mx)
    e = np.exp(z - mx_safe[:, None])
    ssum = e.sum(axis=1)
    with np.errstate(divide="ignore"):
        lse = np.where(empty, NEG_INF, mx_safe + np.log(np.where(empty, 1.0, ssum)))
    return e, ssum, lse, empty


def attention_forward(q, k, v, s, a, B: int, scale: Optional[float] = None,
                      key_mask: Optional[np.ndarray] = None,
                      blocks: Optional[Sequence[int]] = None,
                      heads: Optional[Sequence[int]] = None):
    """Masked attention of the query rows over the context keys:
    z = scale * q k^T + M (M = 0 on s_i <= x < a_i, -inf elsewhere, and -inf
    outside ``key_mask`` when given), lse = log sum_x exp z,
    o = sum_x exp(z - lse) v_x  [Split-KV §4.1, Eq. 3; mask of Fig. 1].

    With key_mask = K_p this is rank p's local partial (o_p, l_p); without it,
    the single-device result.  Rows with no visible key get lse = -inf, o = 0.
    ``blocks``/``heads`` restrict the rows/heads computed (others stay 0/-inf).
    Returns (o [Q,H,d], lse [Q,H]) float64."""
    s, a = _npi(s), _npi(a)
    N = len(s)
    Qn, H, d = q.shape
    S = k.shape[0]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    o = np.zeros((Qn, H, d))
    lse = np.full((Qn, H), NEG_INF)
    kv = _Heads(k, v, H)
    for h in (range(H) if heads is None else heads):
        kh, vh = kv.get(h)
        for i in (range(N) if blocks is None else blocks):
            rows = slice(i * B, (i + 1) * B)
            mrow = mask_row(int(s[i]), int(a[i]), S)
            if key_mask is not None:
                mrow &= key_mask
            z = scale * (_np64(q[rows, h, :]) @ kh.T)
            z = np.where(mrow[None, :], z, NEG_INF)
            e, ssum, l_rows, empty = _softmax_stats(z)
            lse[rows, h] = l_rows
            num = e @ vh
            o[rows, h, :] = np.where(empty[:, None], 0.0,
                                     num / np.where(empty, 1.0, ssum)[:, None])
    return o, lse


def partition_forward(q, k, v, s, a, B: int, rank_of_chunk, m: int, P: int,
                      scale: Optional[float] = None,
                      blocks: Optional[Sequence[int]] = None,
                      heads: Optional[Sequence[int]] = None):
    """Per-rank partials (o_p, l_p) for p < P over K_p  [Split-KV §4.1 Eq. 3,
    the per-rank attention of Alg. 1].  Returns (o_part [P,Q,H,d], lse_part [P,Q,H])."""
    S = k.shape[0]
    outs, lses = [], []
    for p in range(P):
        km = chunk_key_mask(rank_of_chunk, p, m, S)
        o_p, l_p = attention_forward(q, k, v, s, a, B, scale, key_mask=km,
                                     blocks=blocks, heads=heads)
        outs.append(o_p)
        lses.append(l_p)
    return np.stack(outs), np.stack(lses)


def lse_merge(o_part, lse_part):
    """Exact reconstruction from disjoint partials  [Split-KV §4.1, Eq. 4]:
    l = log sum_p exp(l_p), o = sum_p exp(l_p - l) o_p.
    Partials with l_p = -inf contribute nothing; a row whose partials are all
    -inf gets o = 0, l = -inf.  Inputs [P, ...rows..., d] and [P, ...rows...]."""
    o_part = np.asarray(o_part, np.float64)
    lse_part = np.asarray(lse_part, np.float64)
    mx = lse_part.max(axis=0)
    empty = ~np.isfinite(mx)
    mx_safe = np.where(empty, 0.0, mx)
    w = np.exp(lse_part - mx_safe[None])            # exp(-inf) = 0 for empty partials
    tot = w.sum(axis=0)
    with np.errstate(divide="ignore"):
        lse = np.where(empty, NEG_INF, mx_safe + np.log(np.where(empty, 1.0, tot)))
    # exp(l_p - l) per partial; zero where l_p = -inf (o_p unspecified there)
    coef = np.where(np.isfinite(lse_part), np.exp(lse_part - np.where(empty, 0.0, lse)[None]), 0.0)
    o_clean = np.where(np.isfinite(lse_part)[..., None], o_part, 0.0)
    o = (coef[..., None] * o_clean).sum(axis=0)
    return o, lse


def lse_merge_backward(o_part, lse_part, dO, dlse=None):
    """Backward of the exact merge, per partial  [Split-KV §4.1, Eq. 4; the
    MERGE_BWD step of Alg. 1's backward].  For a loss with gradients dO (of o)
    and dlse (of l; None means zero), differentiate o = sum_p w_p o_p and
    l = log sum_p exp(l_p), where w_p = exp(l_p - l) and dl/dl_p = w_p:
        d o_p = w_p dO,
        d l_p = w_p (dO . o_p) - w_p (dO . o) + w_p dlse,
    the middle term from dw_p/dl_q = w_p (delta_pq - w_q) summed against
    dO . o_p.  Partials with l_p = -inf get zeros.  Shapes as lse_merge; returns
    (do_part [P, ...rows..., d], dlse_part [P, ...rows...])."""
    o_part = np.asarray(o_part, np.float64)
    lse_part = np.asarray(lse_part, np.float64)
    g = np.asarray(dO, np.float64)
    o, lse = lse_merge(o_part, lse_part)
    fin = np.isfinite(lse_part)
    lse_safe = np.where(np.isfinite(lse), lse, 0.0)
    w = np.where(fin, np.exp(np.where(fin, lse_part, 0.0) - lse_safe[None]), 0.0)
    o_clean = np.where(fin[..., None], o_part, 0.0)
    dot_p = (g[None] * o_clean).sum(axis=-1)         # dO . o_p
    dot_o = (g * o).sum(axis=-1)                     # dO . o
    dl = 0.0 if dlse is None else np.asarray(dlse, np.float64)[None]
    dlse_part = w * (dot_p - dot_o[None] + dl)
    do_part = w[..., None] * g[None]
    return do_part, dlse_part


def merge_oproj(o_part, lse_part, w_o):
    """The output projection fused with the merge  [Split-KV §4.1, Eq. 5; the
    MERGE_AR, OProj and RS_sum steps of Alg. 1's forward]: every rank scales its
    partial by its merge weight, o_bar_p = exp(l_p - l) o_p (zero where
    l_p = -inf), projects it, OProj(x) = x W_o^T over the concatenated heads,
    and the projected outputs are summed over the ranks:
        Y = sum_p OProj(o_bar_p).
    Taken in that order here (one projection per partial).  o_part
    [P, Q, H, d], lse_part [P, Q, H], w_o [d_model, H*d]; returns
    (Y [Q, d_model], l [Q, H])."""
    o_part = np.asarray(_np64(o_part), np.float64)
    lse_part = np.asarray(_np64(lse_part), np.float64)
    w = np.asarray(_np64(w_o), np.float64)
    P, Qn, H, d = o_part.shape
    _, lse = lse_merge(o_part, lse_part)
    fin = np.isfinite(lse_part)
    lse_safe = np.where(np.isfinite(lse), lse, 0.0)
    y = np.zeros((Qn, w.shape[0]))
    for p in range(P):
        wp = np.where(fin[p], np.exp(np.where(fin[p], lse_part[p], 0.0) - lse_safe), 0.0)   # [Q, H]
        o_bar = np.where(fin[p][..., None], wp[..., None] * o_part[p], 0.0)                # [Q, H, d]
        y += o_bar.reshape(Qn, H * d) @ w.T
    return y, lse


def attention_backward(q, k, v, s, a, B: int, dO, scale: Optional[float] = None,
                       blocks: Optional[Sequence[int]] = None,
                       heads: Optional[Sequence[int]] = None,
                       kv_heads_only: bool = False):
    """Gradients of L = sum(dO * o) for the single-device masked attention
    (lse receives no gradient), textbook softmax backward:
      P_rx = exp(z_rx - l_r), dv_x = sum_r P_rx dO_r, dP_rx = dO_r . v_x,
      D_r = sum_x P_rx dP_rx, dS = P * (dP - D), dq_r = scale sum_x dS_rx k_x,
      dk_x = scale sum_r dS_rx q_r.
    Split-KV computes the same gradients per rank (Alg. 1's backward) and sums
    dq over ranks; the partitioned route is ``partitioned_backward``.
    ``blocks`` restricts which query blocks contribute (dk/dv then hold only
    their contributions).  Returns (dq [Q,H,d], dk [S,Hkv,d], dv [S,Hkv,d]);
    with ``kv_heads_only`` dk and dv hold just the key/value heads of ``heads``,
    in order of first use ([S, n, d]; the same sums, smaller arrays)."""
    s, a = _npi(s), _npi(a)
    N = len(s)
    Qn, H, d = q.shape
    S = k.shape[0]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dq = np.zeros((Qn, H, d))
    kv = _Heads(k, v, H)
    hs = list(range(H) if heads is None else heads)
    slot = {}
    for h in hs:
        slot.setdefault(kv.head(h), len(slot))
    n_kv = len(slot) if kv_heads_only else k.shape[1]
    dk = np.zeros((S, n_kv, d))
    dv = np.zeros((S, n_kv, d))
    for h in hs:
        kh, vh = kv.get(h)
        c = slot[kv.head(h)] if kv_heads_only else kv.head(h)
        for i in (range(N) if blocks is None else blocks):
            rows = slice(i * B, (i + 1) * B)
            mrow = mask_row(int(s[i]), int(a[i]), S)
            qb = _np64(q[rows, h, :])
            gb = _np64(dO[rows, h, :])
            z = np.where(mrow[None, :], scale * (qb @ kh.T), NEG_INF)
            e, ssum, l_rows, empty = _softmax_stats(z)
            Pm = np.where(empty[:, None], 0.0, e / np.where(empty, 1.0, ssum)[:, None])
            dv[:, c, :] += Pm.T @ gb
            dP = gb @ vh.T
            D = (Pm * dP).sum(axis=1)
            dS = Pm * (dP - D[:, None])
            dq[rows, h, :] = scale * (dS @ kh)
            dk[:, c, :] += scale * (dS.T @ qb)
    return dq, dk, dv


def backward_key_rows(q, k, v, s, a, B: int, dO, keys: Sequence[int],
                      heads: Sequence[int], scale: Optional[float] = None):
    """dk, dv at the listed context keys only, for the listed key/value heads
    (same definition as attention_backward, each head summed over its query
    heads; only the blocks whose window holds one of the keys contribute, and
    each of those rows needs its full-row l_r and D_r).
    Returns (dk [len(keys), len(heads), d], dv [...])."""
    s, a = _npi(s), _npi(a)
    N = len(s)
    H, d = q.shape[1], q.shape[2]
    S = k.shape[0]
    g = H // k.shape[1]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    keys = list(keys)
    kidx = np.asarray(keys, np.int64)
    dk = np.zeros((len(keys), len(heads), d))
    dv = np.zeros((len(keys), len(heads), d))
    kv = _Heads(k, v, H)
    for hi, h in ((hi, h) for hi, c in enumerate(heads) for h in range(c * g, (c + 1) * g)):
        kh, vh = kv.get(h)
        for i in range(N):
            if not np.any((s[i] <= kidx) & (kidx < a[i])):
                continue
            rows = slice(i * B, (i + 1) * B)
            # the block's visible keys: the columns its mask row leaves open (a key
            # outside them has exp(-inf) = 0 weight, so the row statistics are sums
            # over these columns alone)
            cols = np.flatnonzero(mask_row(int(s[i]), int(a[i]), S))
            c0, c1 = int(cols[0]), int(cols[-1]) + 1      # one run of columns: the window [s_i, a_i)
            assert c1 - c0 == len(cols)
            qb = _np64(q[rows, h, :])
            gb = _np64(dO[rows, h, :])
            z = scale * (qb @ kh[c0:c1].T)
            e, ssum, _, _ = _softmax_stats(z)
            Pm = e / ssum[:, None]
            dP = gb @ vh[c0:c1].T
            D = (Pm * dP).sum(axis=1)
            pos = np.searchsorted(cols, kidx)          # the listed keys' columns among the visible ones
            seen = (pos < len(cols)) & (cols[np.minimum(pos, len(cols) - 1)] == kidx)
            Pk = np.where(seen[None, :], Pm[:, np.minimum(pos, len(cols) - 1)], 0.0)
            dSk = Pk * (dP[:, np.minimum(pos, len(cols) - 1)] - D[:, None])
            dv[:, hi, :] += Pk.T @ gb
            dk[:, hi, :] += scale * (dSk.T @ qb)
    return dk, dv


def partitioned_backward(q, k, v, s, a, B: int, dO, rank_of_chunk, m: int, P: int,
                         scale: Optional[float] = None):
    """The backward along Alg. 1's own route [Split-KV Alg. 1, backward pass;
    Eq. 4]: with every rank's dō_p = dO (o = sum_p ō_p), MERGE_BWD gives
    do_p = w_p dO and dl_p = w_p (dO . o_p - dO . o), w_p = exp(l_p - l); each
    rank then back-propagates through its local partial (o_p, l_p) of Eq. 3:
    dz = P^p * (do_p . v - do_p . o_p) + dl_p P^p, dq^(p) = scale dz k,
    dk_p = scale dz^T q, dv_p = P^p^T do_p; finally dq = sum_p dq^(p).
    Returns (dq, dk, dv, dq_parts [P,Q,H,d])."""
    s, a = _npi(s), _npi(a)
    N = len(s)
    Qn, H, d = q.shape
    S = k.shape[0]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    o_part, lse_part = partition_forward(q, k, v, s, a, B, rank_of_chunk, m, P, scale)
    o, lse = lse_merge(o_part, lse_part)
    g = _np64(dO)
    dq_parts = np.zeros((P, Qn, H, d))
    dk = np.zeros((S, k.shape[1], d))
    dv = np.zeros((S, k.shape[1], d))
    kv = _Heads(k, v, H)
    for p in range(P):
        km = chunk_key_mask(rank_of_chunk, p, m, S)
        for h in range(H):
            kh, vh = kv.get(h)
            for i in range(N):
                rows = slice(i * B, (i + 1) * B)
                l_p = lse_part[p, rows, h]
                if not np.any(np.isfinite(l_p)):
                    continue
                mrow = mask_row(int(s[i]), int(a[i]), S) & km
                qb = _np64(q[rows, h, :])
                z = np.where(mrow[None, :], scale * (qb @ kh.T), NEG_INF)
                Pp = np.exp(z - l_p[:, None])                    # local softmax
                w = np.exp(l_p - lse[rows, h])                   # w_p
                do_p = w[:, None] * g[rows, h, :]
                dl_p = w * ((g[rows, h, :] * o_part[p, rows, h, :]).sum(1)
                            - (g[rows, h, :] * o[rows, h, :]).sum(1))
                dz = Pp * (do_p @ vh.T - (do_p * o_part[p, rows, h, :]).sum(1)[:, None]) \
                    + dl_p[:, None] * Pp
                dq_parts[p, rows, h, :] = scale * (dz @ kh)
                dk[:, kv.head(h), :] += scale * (dz.T @ qb)
                dv[:, kv.head(h), :] += Pp.T @ do_p
    return dq_parts.sum(axis=0), dk, dv, dq_parts


# ---------------------------------------------------------------------------
# The block-local term: each block's rows over the block's own B keys
# ---------------------------------------------------------------------------
#
# Reading: besides its context window, block i attends bidirectionally to the B
# tokens of its own block [Split-KV §3.1, Fig. 1 caption; the N B^2 term of
# T_attn in §4.1].  Those tokens' keys and values are the drafter's own
# projections of the block positions, so they arrive as two more tensors with
# q's rows: k_blk, v_blk [Q, Hkv, d], rows [iB, iB+B) belonging to block i (Hkv
# key/value heads, = H without grouped queries).
# They are disjoint from every context chunk, so their (o, l) is one more
# partial of Eq. 4.

def block_local_forward(q, k_blk, v_blk, B: int, scale: Optional[float] = None,
                        heads: Optional[Sequence[int]] = None):
    """Rows of block i over the block's own keys, unmasked:
    z = scale q k_blk^T, l = log sum exp z, o = sum exp(z - l) v_blk.
    Returns (o [Q,H,d], lse [Q,H]) float64."""
    Qn, H, d = q.shape
    N = Qn // B
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    o = np.zeros((Qn, H, d))
    lse = np.full((Qn, H), NEG_INF)
    for h in (range(H) if heads is None else heads):
        for i in range(N):
            rows = slice(i * B, (i + 1) * B)
            c = kv_head(h, H, k_blk.shape[1])
            z = scale * (_np64(q[rows, h, :]) @ _np64(k_blk[rows, c, :]).T)
            e, ssum, l_rows, _ = _softmax_stats(z)
            lse[rows, h] = l_rows
            o[rows, h, :] = (e @ _np64(v_blk[rows, c, :])) / ssum[:, None]
    return o, lse


def full_mask_forward(q, k, v, k_blk, v_blk, s, a, B: int, scale: Optional[float] = None,
                      blocks: Optional[Sequence[int]] = None, heads: Optional[Sequence[int]] = None):
    """The whole anchor mask at once, as its definition reads: block i's rows
    see the context keys of W_i and their block's own B keys; one softmax over
    that concatenated key set [Split-KV §3.1, Fig. 1].  ``blocks``/``heads``
    restrict the rows/heads computed (others stay 0/-inf).  Returns (o, lse)."""
    s, a = _npi(s), _npi(a)
    N = len(s)
    Qn, H, d = q.shape
    S = k.shape[0]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    o = np.zeros((Qn, H, d))
    lse = np.full((Qn, H), NEG_INF)
    kv = _Heads(k, v, H)
    for h in (range(H) if heads is None else heads):
        kh, vh = kv.get(h)
        c = kv.head(h)
        for i in (range(N) if blocks is None else blocks):
            rows = slice(i * B, (i + 1) * B)
            keys = np.concatenate([kh, _np64(k_blk[rows, c, :])])
            vals = np.concatenate([vh, _np64(v_blk[rows, c, :])])
            visible = np.concatenate([mask_row(int(s[i]), int(a[i]), S), np.ones(B, dtype=bool)])
            z = np.where(visible[None, :], scale * (_np64(q[rows, h, :]) @ keys.T), NEG_INF)
            e, ssum, l_rows, _ = _softmax_stats(z)
            lse[rows, h] = l_rows
            o[rows, h, :] = (e @ vals) / ssum[:, None]
    return o, lse


def _given_backward(qb, kb, vb, gb, ob, lb, visible, scale):
    """Gradients through one row block for keys kb/vb, given the merged output
    ob and log-sum-exp lb of those rows: P = exp(z - l), D = dO . o,
    dS = P (dP - D); returns (dq, dk, dv) of this key set."""
    z = np.where(visible, scale * (qb @ kb.T), NEG_INF)
    finite = np.isfinite(lb)
    Pm = np.where(finite[:, None], np.exp(z - np.where(finite, lb, 0.0)[:, None]), 0.0)
    dP = gb @ vb.T
    D = (gb * ob).sum(axis=1)
    dS = Pm * (dP - D[:, None])
    return scale * (dS @ kb), scale * (dS.T @ qb), Pm.T @ gb


def context_backward_given(q, k, v, s, a, B: int, dO, o, lse, scale: Optional[float] = None,
                           blocks: Optional[Sequence[int]] = None, heads: Optional[Sequence[int]] = None):
    """The context part of the gradients of L = sum(dO * o) when o and lse are
    the merged results of a larger key set (Alg. 1's MERGE_BWD in merged form):
    P_rx = exp(z_rx - l_r) over W_i, D_r = dO_r . o_r, dS = P (dP - D).
    With o, lse of the context alone this is ``attention_backward``.
    ``blocks``/``heads`` restrict which query rows contribute.  Returns (dq, dk, dv)."""
    s, a = _npi(s), _npi(a)
    N = len(s)
    Qn, H, d = q.shape
    S = k.shape[0]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    o, lse, g = _np64(o), _np64(lse), _np64(dO)
    dq = np.zeros((Qn, H, d))
    dk = np.zeros((S, k.shape[1], d))
    dv = np.zeros((S, k.shape[1], d))
    kv = _Heads(k, v, H)
    for h in (range(H) if heads is None else heads):
        kh, vh = kv.get(h)
        c = kv.head(h)
        for i in (range(N) if blocks is None else blocks):
            rows = slice(i * B, (i + 1) * B)
            mrow = mask_row(int(s[i]), int(a[i]), S)[None, :]
            gq, gk, gv = _given_backward(_np64(q[rows, h, :]), kh, vh, g[rows, h, :], o[rows, h, :],
                                         lse[rows, h], mrow, scale)
            dq[rows, h, :] = gq
            dk[:, c, :] += gk
            dv[:, c, :] += gv
    return dq, dk, dv


def block_local_backward(q, k_blk, v_blk, dO, o, lse, B: int, scale: Optional[float] = None,
                         blocks: Optional[Sequence[int]] = None, heads: Optional[Sequence[int]] = None):
    """The block-local part of the same gradients: rows of block i over the
    block's own keys with the merged o, lse.  Returns (dq_local [Q,H,d],
    dk_blk [Q,Hkv,d], dv_blk [Q,Hkv,d]; a key/value head sums its query heads);
    the full dq is the context dq plus dq_local."""
    Qn, H, d = q.shape
    N = Qn // B
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    o, lse, g = _np64(o), _np64(lse), _np64(dO)
    Hkv = k_blk.shape[1]
    dq = np.zeros((Qn, H, d))
    dk = np.zeros((Qn, Hkv, d))
    dv = np.zeros((Qn, Hkv, d))
    allvis = np.ones((1, B), dtype=bool)
    for h in (range(H) if heads is None else heads):
        c = kv_head(h, H, Hkv)
        for i in (range(N) if blocks is None else blocks):
            rows = slice(i * B, (i + 1) * B)
            gq, gk, gv = _given_backward(_np64(q[rows, h, :]), _np64(k_blk[rows, c, :]),
                                         _np64(v_blk[rows, c, :]), g[rows, h, :], o[rows, h, :],
                                         lse[rows, h], allvis, scale)
            dq[rows, h, :] = gq
            dk[rows, c, :] += gk
            dv[rows, c, :] += gv
    return dq, dk, dv


def merge_bytes(lse_part, d: int, out_elem_bytes: int) -> int:
    """Algorithmic HBM bytes of one LSE merge: every l_p (4 B), the o_p rows
    whose l_p is finite (d*4 B each), and the outputs o (d*out_elem_bytes) and
    l (4 B) per row."""
    lp = np.asarray(lse_part)
    P = lp.shape[0]
    rows = int(np.prod(lp.shape[1:]))
    finite = int(np.isfinite(lp).sum())
    return P * rows * 4 + finite * d * 4 + rows * (d * out_elem_bytes + 4)
