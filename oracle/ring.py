"""Ring attention simulated rank by rank on the CPU (oracle; test infrastructure).

"Long Context Attention" notes, "Ring Attention": the QKV sequence is split
over cp hosts arranged in a ring; the KV segments travel around the ring and
a full cycle ends once every host has seen every KV segment. At step s, ring
rank rho holds the KV shard that started on rank (rho - s) mod cp. Each step
yields a partial (O_s, LSE_s) for rho's queries (attention restricted to that
shard's keys, with the mask taken on natural positions), and the partials are
combined with the log-sum-exp merge. This module runs that schedule literally
with NumPy, one virtual rank and one step at a time, so "chunk, then merge"
can be checked against the plain definition in `attention`.

With ulysses_degree > 1 (USP, YunChang README "2. Usage") the heads are first
exchanged by the simulated all-to-all in `layouts`, each Ulysses group runs
its own ring over its heads, and the outputs are exchanged back.

The backward pass uses the forward's final LSE: for every (rank, step) the
chunk pair contributes P = exp(s - LSE) restricted to that pair, and
dS = P * (dO.V - Delta) with Delta_i = <dO_i, O_i> (which equals
sum_j P_ij dP_ij because the P row sums to one over all chunks). dK/dV of a
shard accumulate across every query rank that visited it (the shard's ring
return).
"""
from __future__ import annotations

from typing import Dict, Optional, Tuple

import numpy as np

from . import attention, layouts, merge


def _f64(x):
    return attention._f64(x)


class _Seq:
    """Natural position, segment id and segment start for each token."""

    def __init__(self, S: int, cu_seqlens):
        self.S = S
        if cu_seqlens is None:
            self.start = np.zeros(S, np.int64)
            self.seg = np.zeros(S, np.int64)
        else:
            cu = np.asarray(cu_seqlens, dtype=np.int64)
            seg = np.searchsorted(cu, np.arange(S), side="right") - 1
            self.seg = seg
            self.start = cu[seg]

    def vis(self, qnat, knat, causal, window, sink):
        v = attention.visibility(qnat - self.start[qnat],
                                 knat - self.start[knat],
                                 causal, window, sink)
        # visibility() compares relative positions as an outer product; keys of
        # another segment are hidden outright.
        return v & (self.seg[qnat][:, None] == self.seg[knat][None, :])


def _group_tensors(x_perm: np.ndarray, cp: int, ud: int) -> np.ndarray:
    """[B,S,H,D] permuted -> [ud,B,S,H/ud,D] by the simulated all-to-all."""
    if ud == 1:
        return x_perm[None]
    return layouts.ulysses_seq2head(x_perm, cp, ud)


def _ungroup(y: np.ndarray, cp: int, ud: int) -> np.ndarray:
    if ud == 1:
        return y[0]
    return layouts.ulysses_head2seq(y, cp, ud)


def ring_attn_fwd(q, k, v, scale: float, layout: str, cp: int, ud: int = 1,
                  causal: bool = True, window: int = 0, sink_tokens: int = 0,
                  cu_seqlens=None, order: str = "ring",
                  record: Optional[Dict] = None) -> Tuple[np.ndarray, np.ndarray]:
    """Natural-order inputs -> natural-order (O, LSE) via the ring schedule.

    Shapes as attention.attn_fwd. `order` picks the merge order of the cp
    partials of each rank: "ring" (step order) or "tree" (pairwise levels).
    `record`, if given, receives record[(rho, s)] = number of visible pairs
    per head at that step (for checking the layouts' balance).
    """
    packed = cu_seqlens is not None
    q, k, v = (_f64(t) for t in (q, k, v))
    if packed:
        q, k, v = q[None], k[None], v[None]
    B, S, Hq, D = q.shape
    Hkv = k.shape[2]
    G = Hq // Hkv
    seq = _Seq(S, cu_seqlens)
    perm = layouts.permutation(layout, S, cp)
    Yq = _group_tensors(layouts.extract(q, layout, cp), cp, ud)
    Yk = _group_tensors(layouts.extract(k, layout, cp), cp, ud)
    Yv = _group_tensors(layouts.extract(v, layout, cp), cp, ud)
    n = S // cp
    Oy = np.zeros_like(Yq)
    Ly = np.zeros((ud, B, Hq // ud, S))
    for u in range(ud):
        for rho in range(cp):
            qrows = slice(rho * n, (rho + 1) * n)
            qnat = perm[qrows]
            parts = {}
            for s in range(cp):
                kap = (rho - s) % cp
                krows = slice(kap * n, (kap + 1) * n)
                vis = seq.vis(qnat, perm[krows], causal, window, sink_tokens)
                if record is not None:
                    record[(rho, s)] = int(vis.sum())
                for b in range(B):
                    for hl in range(Hq // ud):
                        gl = hl // G
                        o, lse = attention.softmax_rows(
                            Yq[u, b, qrows, hl], Yk[u, b, krows, gl],
                            Yv[u, b, krows, gl], vis, scale)
                        parts.setdefault((b, hl), []).append((o, lse))
            for (b, hl), plist in parts.items():
                fn = merge.merge_linear if order == "ring" else merge.merge_tree
                o, lse = fn(plist)
                Oy[u, b, qrows, hl] = o
                Ly[u, b, hl, qrows] = lse
    O_perm = _ungroup(Oy, cp, ud)
    # LSE [ud, B, Hq/ud, S] -> [B, Hq, S] (head h = u*Hq/ud + h')
    L_perm = np.concatenate([Ly[u] for u in range(ud)], axis=1)
    O = layouts.restore(O_perm, layout, cp, axis=1)
    L = layouts.restore(L_perm, layout, cp, axis=2)
    if packed:
        return O[0], L[0]
    return O, L


def ring_attn_bwd(q, k, v, dout, scale: float, layout: str, cp: int,
                  ud: int = 1, causal: bool = True, window: int = 0,
                  sink_tokens: int = 0, cu_seqlens=None):
    """Gradients via the ring schedule, using the forward's final (O, LSE)."""
    packed = cu_seqlens is not None
    O_nat, L_nat = ring_attn_fwd(q, k, v, scale, layout, cp, ud, causal,
                                 window, sink_tokens, cu_seqlens)
    q, k, v, do = (_f64(t) for t in (q, k, v, dout))
    if packed:
        q, k, v, do = q[None], k[None], v[None], do[None]
        O_nat, L_nat = O_nat[None], L_nat[None]
    B, S, Hq, D = q.shape
    Hkv = k.shape[2]
    G = Hq // Hkv
    seq = _Seq(S, cu_seqlens)
    perm = layouts.permutation(layout, S, cp)
    ex = lambda x: layouts.extract(x, layout, cp)  # noqa: E731
    Yq, Yk, Yv, Ydo, Yo = (_group_tensors(ex(t), cp, ud)
                           for t in (q, k, v, do, O_nat))
    Lp = layouts.extract(L_nat, layout, cp, axis=2)
    n = S // cp
    dYq = np.zeros_like(Yq)
    dYk = np.zeros_like(Yk)
    dYv = np.zeros_like(Yv)
    hq = Hq // ud
    for u in range(ud):
        for rho in range(cp):
            qrows = slice(rho * n, (rho + 1) * n)
            qnat = perm[qrows]
            for s in range(cp):
                kap = (rho - s) % cp
                krows = slice(kap * n, (kap + 1) * n)
                vis = seq.vis(qnat, perm[krows], causal, window, sink_tokens)
                for b in range(B):
                    for hl in range(hq):
                        gl = hl // G
                        qb, dob = Yq[u, b, qrows, hl], Ydo[u, b, qrows, hl]
                        kb, vb = Yk[u, b, krows, gl], Yv[u, b, krows, gl]
                        lse = Lp[b, u * hq + hl, qrows]
                        lse_s = np.where(np.isfinite(lse), lse, 0.0)
                        P = np.where(vis, np.exp(scale * (qb @ kb.T)
                                                 - lse_s[:, None]), 0.0)
                        delta = (dob * Yo[u, b, qrows, hl]).sum(axis=1)
                        dS = P * (dob @ vb.T - delta[:, None])
                        dYq[u, b, qrows, hl] += scale * (dS @ kb)
                        dYk[u, b, krows, gl] += scale * (dS.T @ qb)
                        dYv[u, b, krows, gl] += P.T @ dob
    res = []
    for y in (dYq, dYk, dYv):
        x = layouts.restore(_ungroup(y, cp, ud), layout, cp, axis=1)
        res.append(x[0] if packed else x)
    return tuple(res)


def step_pair_counts(layout: str, S: int, cp: int, causal: bool = True,
                     window: int = 0, sink_tokens: int = 0,
                     cu_seqlens=None) -> np.ndarray:
    """Visible (query, key) pairs of one head at each (rank, step): [cp, cp].

    Counts only; no attention is computed. Used to check which ring steps do
    work under each layout and mask.
    """
    seq = _Seq(S, cu_seqlens)
    perm = layouts.permutation(layout, S, cp)
    n = S // cp
    out = np.zeros((cp, cp), dtype=np.int64)
    for rho in range(cp):
        qnat = perm[rho * n:(rho + 1) * n]
        for s in range(cp):
            kap = (rho - s) % cp
            knat = perm[kap * n:(kap + 1) * n]
            for r0 in range(0, n, 1024):
                out[rho, s] += int(seq.vis(qnat[r0:r0 + 1024], knat, causal,
                                           window, sink_tokens).sum())
    return out
