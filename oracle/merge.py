"""The log-sum-exp merge of attention partials (oracle; test infrastructure).

A partial (O_a, L_a) is attention restricted to a subset of keys: L_a is the
log-sum-exp of its scores and O_a its normalised output. Because logsumexp
and max are associative ("Long Context Attention" notes, "Tree Attention"),
two partials over disjoint key sets combine into the partial over their
union:

    L = log(exp(L_a) + exp(L_b))
    O = exp(L_a - L) O_a + exp(L_b - L) O_b

computed here with the larger of L_a, L_b factored out. An empty partial
(L = -inf, O = 0) is the identity. The order of merging is free ("Ring
Attention": the order of block computation is arbitrary).
"""
from __future__ import annotations

from typing import List, Sequence, Tuple

import numpy as np

Partial = Tuple[np.ndarray, np.ndarray]  # O [..., D], L [...]


def merge_pair(a: Partial, b: Partial) -> Partial:
    oa, la = np.asarray(a[0], np.float64), np.asarray(a[1], np.float64)
    ob, lb = np.asarray(b[0], np.float64), np.asarray(b[1], np.float64)
    m = np.maximum(la, lb)
    both_empty = ~np.isfinite(m)
    ms = np.where(both_empty, 0.0, m)
    ea = np.where(np.isfinite(la), np.exp(la - ms), 0.0)
    eb = np.where(np.isfinite(lb), np.exp(lb - ms), 0.0)
    tot = ea + eb
    L = np.where(both_empty, -np.inf, ms + np.log(np.where(both_empty, 1.0, tot)))
    wa = np.where(both_empty, 0.0, ea / np.where(both_empty, 1.0, tot))
    wb = np.where(both_empty, 0.0, eb / np.where(both_empty, 1.0, tot))
    O = wa[..., None] * oa + wb[..., None] * ob
    return O, L


def merge_linear(parts: Sequence[Partial]) -> Partial:
    """((p0 + p1) + p2) + ... : the order a ring visits its chunks."""
    acc = parts[0]
    for p in parts[1:]:
        acc = merge_pair(acc, p)
    return acc


def merge_tree(parts: Sequence[Partial]) -> Partial:
    """Pairwise levels: (p0+p1), (p2+p3), ...; an odd last one moves up as is."""
    level: List[Partial] = list(parts)
    while len(level) > 1:
        nxt = [merge_pair(level[i], level[i + 1])
               for i in range(0, len(level) - 1, 2)]
        if len(level) % 2:
            nxt.append(level[-1])
        level = nxt
    return level[0]
