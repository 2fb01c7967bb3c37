"""Useful-FLOP and algorithmic-byte accounting for the benchmark.

Only visible (query, key) pairs count: masked-out work is never useful. Per
visible pair and query head the forward does two D-long dot products
(q.k and p.v), i.e. 4*D FLOPs; the backward does five (recomputed q.k, dO.v,
and the dV, dQ, dK products), i.e. 2.5x the forward.
"""
from __future__ import annotations

from typing import Iterable, Optional


def visible_pairs_segment(L: int, causal: bool, window: int, sink: int) -> int:
    """Visible pairs of one head in one sequence of length L (closed form)."""
    if L <= 0:
        return 0
    if window <= 0 or (causal and window >= L):
        return L * (L + 1) // 2 if causal else L * L
    W = window
    if causal:
        # row i sees min(i+1, W) window keys ...
        n = W * (W + 1) // 2 + (L - W) * W
        # ... plus sink keys j < sink that fall out of the window (j <= i-W)
        if sink > 0:
            for i in range(W, L):
                n += min(sink, i - W + 1)
        return n
    # non-causal window: row i sees keys j >= i-W+1 (all later keys) ...
    n = 0
    for i in range(L):
        lo = max(0, i - W + 1)
        n += L - lo
        if sink > 0:
            n += max(0, min(sink, lo))
    return n


def visible_pairs(S: int, causal: bool, window: int, sink: int,
                  cu_seqlens: Optional[Iterable[int]] = None) -> int:
    """Visible pairs of one head over a dense sequence or a packed batch."""
    if cu_seqlens is None:
        return visible_pairs_segment(S, causal, window, sink)
    cu = [int(c) for c in cu_seqlens]
    return sum(visible_pairs_segment(cu[i + 1] - cu[i], causal, window, sink)
               for i in range(len(cu) - 1))


def attention_flops(w, cu_seqlens=None) -> dict:
    """Useful forward/backward FLOPs of one pass over workload `w`."""
    pairs = visible_pairs(w.S, w.causal, w.window, w.sink_tokens, cu_seqlens)
    batches = 1 if w.varlen else w.B
    fwd = 4.0 * w.D * pairs * w.Hq * batches
    bwd = 2.5 * fwd if w.backward else 0.0
    return {"pairs_per_head": pairs, "fwd": fwd, "bwd": bwd, "total": fwd + bwd}
