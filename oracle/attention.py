"""Exact masked softmax attention in fp64 (oracle; test infrastructure only).

The quantity every sequence-parallel scheme on the pages must reproduce is
plain full attention: the ring is correct because merging per-chunk partials
"equals full attention" ("Long Context Attention" notes, "Ring Attention":
blocks may be computed in any order; "Tree Attention": logsumexp and max are
associative). This module is that plain definition, written with no chunking,
no layout and no merge, so the ring/zigzag/stripe machinery can be checked
against it.

Definition. For a query at position i and a key at position j of the same
sequence (positions relative to the start of that sequence in a packed batch):

    visible(i, j) = (not causal or j <= i)
                    and (window <= 0 or i - j < window or j < sink_tokens)

`window` counts visible keys including the query's own position: the ring
sliding-window README ("Arguments": window_size is the number of tokens each
query attends to) with the problem statement's "previous 1000 tokens
including itself". `sink_tokens` are the first tokens of every sequence,
visible to every later query regardless of the window (the README's "Ring
Streaming LLM Attention": every query attends to the first token).

    s_ij = scale * <q_i, k_j>                       (visible j only)
    LSE_i = log sum_j exp(s_ij)                      (natural log; -inf if none)
    O_i   = sum_j exp(s_ij - LSE_i) v_j              (0 if no key is visible)

GQA: query head h reads key/value head h // (Hq // Hkv) (contiguous groups).

Gradient by direct differentiation of the above (the LSE is kept for the
backward pass, "Long Context Attention" notes, "Motivation"):

    P_ij  = exp(s_ij - LSE_i)
    dV_j  = sum_i P_ij dO_i
    dP_ij = <dO_i, v_j>
    dS_ij = P_ij (dP_ij - sum_k P_ik dP_ik)          (softmax Jacobian)
    dQ_i  = scale * sum_j dS_ij k_j
    dK_j  = scale * sum_i dS_ij q_i
with dK, dV summed over the query heads that share a key/value head.
"""
from __future__ import annotations

from typing import Iterable, Optional, Tuple

import numpy as np


def visibility(qpos: np.ndarray, kpos: np.ndarray, causal: bool, window: int,
               sink_tokens: int) -> np.ndarray:
    """Boolean [len(qpos), len(kpos)] mask from positions within one sequence."""
    i = np.asarray(qpos, dtype=np.int64)[:, None]
    j = np.asarray(kpos, dtype=np.int64)[None, :]
    vis = np.ones((i.shape[0], j.shape[1]), dtype=bool)
    if causal:
        vis &= j <= i
    if window > 0:
        vis &= (i - j < window) | (j < sink_tokens)
    return vis


def _f64(x) -> np.ndarray:
    if hasattr(x, "detach"):  # torch tensor (possibly bf16) -> exact fp64
        x = x.detach().to("cpu")
        import torch
        x = x.to(torch.float64).numpy()
    return np.asarray(x, dtype=np.float64)


def softmax_rows(q: np.ndarray, k: np.ndarray, v: np.ndarray, vis: np.ndarray,
                 scale: float) -> Tuple[np.ndarray, np.ndarray]:
    """O [Nq, D] and LSE [Nq] of one head over the visible keys (fp64)."""
    s = scale * (q @ k.T)
    s = np.where(vis, s, -np.inf)
    m = s.max(axis=1, initial=-np.inf)
    empty = ~np.isfinite(m)
    m_safe = np.where(empty, 0.0, m)
    e = np.where(vis, np.exp(s - m_safe[:, None]), 0.0)
    ssum = e.sum(axis=1)
    lse = np.where(empty, -np.inf, m_safe + np.log(np.where(empty, 1.0, ssum)))
    p = np.where(empty[:, None], 0.0, e / np.where(empty, 1.0, ssum)[:, None])
    return p @ v, lse


def _segments(S: int, cu_seqlens) -> list:
    if cu_seqlens is None:
        return [(0, S)]
    cu = [int(x) for x in np.asarray(cu_seqlens).tolist()]
    return [(cu[n], cu[n + 1]) for n in range(len(cu) - 1)]


def _as_batched(x: np.ndarray, packed: bool) -> np.ndarray:
    return x[None] if packed else x


def attn_fwd(q, k, v, scale: float, causal: bool = True, window: int = 0,
             sink_tokens: int = 0, cu_seqlens=None,
             heads: Optional[Iterable[int]] = None,
             block: int = 1024) -> Tuple[np.ndarray, np.ndarray]:
    """Full attention forward.

    q [B,S,Hq,D] (or packed [T,Hq,D] with cu_seqlens); k, v [B,S,Hkv,D] (or
    [T,Hkv,D]). Returns O in q's shape (fp64) and LSE [B,Hq,S] (packed:
    [Hq,T]). `heads` restricts the computation to those query heads (others
    are left NaN): heads are independent, so a subset is checked exactly.
    """
    packed = cu_seqlens is not None
    q, k, v = (_as_batched(_f64(t), packed) for t in (q, k, v))
    B, S, Hq, D = q.shape
    Hkv = k.shape[2]
    G = Hq // Hkv
    heads = range(Hq) if heads is None else list(heads)
    O = np.full(q.shape, np.nan)
    L = np.full((B, Hq, S), np.nan)
    for b in range(B):
        for (a, e) in _segments(S, cu_seqlens):
            pos = np.arange(e - a)
            for h in heads:
                g = h // G
                kk, vv = k[b, a:e, g], v[b, a:e, g]
                for r0 in range(0, e - a, block):
                    r1 = min(e - a, r0 + block)
                    # keys beyond the block's last query are never visible
                    # when causal; cutting them only saves time.
                    kend = r1 if causal else e - a
                    vis = visibility(pos[r0:r1], pos[:kend], causal, window,
                                     sink_tokens)
                    o, lse = softmax_rows(q[b, a + r0:a + r1, h], kk[:kend],
                                          vv[:kend], vis, scale)
                    O[b, a + r0:a + r1, h] = o
                    L[b, h, a + r0:a + r1] = lse
    if packed:
        return O[0], L[0]
    return O, L


def attn_bwd(q, k, v, dout, scale: float, causal: bool = True, window: int = 0,
             sink_tokens: int = 0, cu_seqlens=None,
             kv_heads: Optional[Iterable[int]] = None,
             block: int = 1024):
    """Gradient of attn_fwd's O with respect to q, k, v given dO.

    Recomputes P from its own forward (no GPU value enters). Returns
    (dq, dk, dv) in the input shapes, fp64. `kv_heads` restricts to those
    key/value heads and the query heads of their groups (others NaN).
    """
    packed = cu_seqlens is not None
    q, k, v, do = (_as_batched(_f64(t), packed) for t in (q, k, v, dout))
    B, S, Hq, D = q.shape
    Hkv = k.shape[2]
    G = Hq // Hkv
    kv_heads = range(Hkv) if kv_heads is None else list(kv_heads)
    dq = np.full(q.shape, np.nan)
    dk = np.full(k.shape, np.nan)
    dv = np.full(v.shape, np.nan)
    for b in range(B):
        for g in kv_heads:
            dk[b, :, g] = 0.0
            dv[b, :, g] = 0.0
            for h in range(g * G, (g + 1) * G):
                dq[b, :, h] = 0.0
        for (a, e) in _segments(S, cu_seqlens):
            n = e - a
            pos = np.arange(n)
            for g in kv_heads:
                kk, vv = k[b, a:e, g], v[b, a:e, g]
                for h in range(g * G, (g + 1) * G):
                    for r0 in range(0, n, block):
                        r1 = min(n, r0 + block)
                        kend = r1 if causal else n
                        vis = visibility(pos[r0:r1], pos[:kend], causal,
                                         window, sink_tokens)
                        qb = q[b, a + r0:a + r1, h]
                        dob = do[b, a + r0:a + r1, h]
                        _, lse = softmax_rows(qb, kk[:kend], vv[:kend], vis,
                                              scale)
                        s = scale * (qb @ kk[:kend].T)
                        lse_safe = np.where(np.isfinite(lse), lse, 0.0)
                        P = np.where(vis, np.exp(s - lse_safe[:, None]), 0.0)
                        dP = dob @ vv[:kend].T
                        dS = P * (dP - (P * dP).sum(axis=1, keepdims=True))
                        dq[b, a + r0:a + r1, h] = scale * (dS @ kk[:kend])
                        dk[b, a:a + kend, g] += scale * (dS.T @ qb)
                        dv[b, a:a + kend, g] += P.T @ dob
    if packed:
        return dq[0], dk[0], dv[0]
    return dq, dk, dv


def attn_fwd_rows(q, k, v, scale: float, b: int, h: int, rows: Iterable[int],
                  causal: bool = True, window: int = 0, sink_tokens: int = 0,
                  cu_seqlens=None) -> Tuple[np.ndarray, np.ndarray]:
    """O and LSE of selected query rows (natural positions) of one head.

    For spot checks at full problem size: each row is computed on its own
    from the definition. Packed inputs take b=0 and rows in packed positions.
    """
    packed = cu_seqlens is not None
    rows = np.asarray(list(rows), dtype=np.int64)
    qb = q[b] if not packed else q
    kb = k[b] if not packed else k
    vb = v[b] if not packed else v
    Hq, Hkv = qb.shape[1], kb.shape[1]
    g = h // (Hq // Hkv)
    S = qb.shape[0]
    segs = _segments(S, cu_seqlens)
    starts = np.array([s for s, _ in segs])
    O = np.zeros((len(rows), qb.shape[2]))
    L = np.zeros(len(rows))
    for n, r in enumerate(rows.tolist()):
        si = int(np.searchsorted(starts, r, side="right") - 1)
        a, e = segs[si]
        kend = r + 1 if causal else e
        vis = visibility(np.array([r - a]), np.arange(kend - a), causal,
                         window, sink_tokens)
        o, lse = softmax_rows(_f64(qb[r:r + 1, h]), _f64(kb[a:kend, g]),
                              _f64(vb[a:kend, g]), vis, scale)
        O[n], L[n] = o[0], lse[0]
    return O, L


def count_visible_pairs(S: int, causal: bool, window: int, sink_tokens: int,
                        cu_seqlens=None) -> int:
    """Number of visible (query, key) pairs of one head, by brute force."""
    total = 0
    for (a, e) in _segments(S, cu_seqlens):
        pos = np.arange(e - a)
        for r0 in range(0, e - a, 2048):
            r1 = min(e - a, r0 + 2048)
            total += int(visibility(pos[r0:r1], pos, causal, window,
                                    sink_tokens).sum())
    return total


def attn_bwd_sampled(q, k, v, dout, scale: float, b: int, g: int,
                     q_rows: Iterable[int], k_rows: Iterable[int],
                     causal: bool = True, window: int = 0, sink_tokens: int = 0,
                     cu_seqlens=None, block: int = 2048):
    """Gradient rows for spot checks at full problem size.

    Returns (dq [G, nq, D] for q_rows of every query head of KV group g,
    dk [nk, D], dv [nk, D] for k_rows of KV head g), batch b (packed: b=0).
    Uses the identity sum_j P_ij dP_ij = <dO_i, O_i> (the P row sums to one),
    with O and LSE from this module's own forward of the group's heads. That
    forward covers only the query rows the result needs: q_rows and every
    query that sees one of k_rows (the visibility rule decides which); the
    other rows enter no sampled gradient.
    """
    packed = cu_seqlens is not None
    sel = (lambda t: t) if packed else (lambda t: t[b])
    G = q.shape[-2] // k.shape[-2]
    heads = list(range(g * G, (g + 1) * G))
    # only the group's heads are converted (inputs can be several GB)
    qb = np.stack([_f64(sel(q)[:, h]) for h in heads], axis=1)
    dob = np.stack([_f64(sel(dout)[:, h]) for h in heads], axis=1)
    kk, vv = _f64(sel(k)[:, g]), _f64(sel(v)[:, g])
    S, _, D = qb.shape
    segs = _segments(S, cu_seqlens)
    starts = np.array([s for s, _ in segs])
    # full forward (O, LSE) of the group's heads, segment by segment; heads
    # are independent and run on threads (NumPy releases the GIL).
    O = np.zeros((G, S, D))
    L = np.zeros((G, S))
    q_rows = [int(r) for r in q_rows]
    k_rows = [int(r) for r in k_rows]
    # per segment: the local query positions whose O and LSE are needed
    need = []
    for (a, e) in segs:
        pos = np.arange(e - a)
        nd = np.zeros(e - a, dtype=bool)
        nd[[r - a for r in q_rows if a <= r < e]] = True
        ks = np.array([j - a for j in k_rows if a <= j < e], dtype=np.int64)
        if ks.size:
            nd |= visibility(pos, ks, causal, window, sink_tokens).any(axis=1)
        need.append(nd)

    def head_fwd(hi):
        for (a, e), nd in zip(segs, need):
            pos = np.arange(e - a)
            for r0 in range(0, e - a, block):
                r1 = min(e - a, r0 + block)
                rr = r0 + np.nonzero(nd[r0:r1])[0]
                if rr.size == 0:
                    continue
                # with causal, keys past the block's last needed query are
                # never visible to it; cutting them only saves time
                kend = int(rr[-1]) + 1 if causal else e - a
                vis = visibility(pos[rr], pos[:kend], causal, window,
                                 sink_tokens)
                o, lse = softmax_rows(qb[a + rr, hi], kk[a:a + kend],
                                      vv[a:a + kend], vis, scale)
                O[hi, a + rr] = o
                L[hi, a + rr] = lse

    from concurrent.futures import ThreadPoolExecutor
    with ThreadPoolExecutor(max_workers=G) as ex:
        list(ex.map(head_fwd, range(G)))
    delta = np.einsum("hsd,shd->hs", O, dob)
    dq = np.zeros((G, len(q_rows), D))
    for n, r in enumerate(q_rows):
        si = int(np.searchsorted(starts, r, side="right") - 1)
        a, e = segs[si]
        vis = visibility(np.array([r - a]), np.arange(e - a), causal, window,
                         sink_tokens)[0]
        js = a + np.nonzero(vis)[0]
        for hi in range(G):
            s = scale * (kk[js] @ qb[r, hi])
            P = np.exp(s - L[hi, r])
            dS = P * (vv[js] @ dob[r, hi] - delta[hi, r])
            dq[hi, n] = scale * (dS @ kk[js])
    dk = np.zeros((len(k_rows), D))
    dv = np.zeros((len(k_rows), D))
    for n, j in enumerate(k_rows):
        si = int(np.searchsorted(starts, j, side="right") - 1)
        a, e = segs[si]
        vis = visibility(np.arange(e - a), np.array([j - a]), causal, window,
                         sink_tokens)[:, 0]
        iis = a + np.nonzero(vis)[0]
        for hi in range(G):
            s = scale * (qb[iis, hi] @ kk[j])
            P = np.exp(s - L[hi, iis])
            dS = P * (dob[iis, hi] @ vv[j] - delta[hi, iis])
            dv[n] += P @ dob[iis, hi]
            dk[n] += scale * (dS @ qb[iis, hi])
    return dq, dk, dv
