"""Decode-step attention over a sharded KV cache (oracle; test infrastructure
only: tests, the smoke check and the bench's CPU baseline use it).

At inference the ring carries the KV cache instead of training chunks ("Long
Context Attention" notes, "Ring Attention": flash decoding is ring attention
at inference time; "Tree Attention": the partials that the devices compute
for one decoding step are combined by a tree reduction, which logsumexp's
associativity allows). What a decode step must produce is still plain
attention, of the newest Tq tokens against the whole cache of S keys:

    query t (t = 0 .. Tq-1) is the token at position S - Tq + t;
    visible(t, j) = (not causal) or j <= S - Tq + t
    s_tj = scale * <q_t, k_j>,  LSE_t = log sum_j exp(s_tj),
    O_t = sum_j exp(s_tj - LSE_t) v_j            (oracle.attention's rule)

GQA: query head h reads key/value head h // (Hq // Hkv).

decode_fwd is that definition. decode_partials cuts the keys into n equal
contiguous pieces in order (cp ranks holding `splits` pieces each; rank r
holds keys [r S / cp, (r + 1) S / cp)) and returns the partial of each piece,
so that merging them (oracle.merge, linear or tree order) can be checked
against decode_fwd.

Layouts: q [B, Tq, Hq, D]; k, v [B, S, Hkv, D]; O [B, Tq, Hq, D];
LSE [B, Tq, Hq].
"""
from __future__ import annotations

from typing import List, Tuple

import numpy as np

from oracle.attention import _f64, softmax_rows


def _decode(q, k, v, scale: float, causal: bool, k0: int, k1: int,
            S: int) -> Tuple[np.ndarray, np.ndarray]:
    """Partial of keys [k0, k1) for every query (the whole cache: 0, S)."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, Tq, Hq, D = q.shape
    G = Hq // k.shape[2]
    qpos = S - Tq + np.arange(Tq)
    kpos = np.arange(k0, k1)
    vis = np.ones((Tq, k1 - k0), dtype=bool)
    if causal:
        vis = kpos[None, :] <= qpos[:, None]
    O = np.zeros((B, Tq, Hq, D))
    L = np.zeros((B, Tq, Hq))
    for b in range(B):
        for h in range(Hq):
            g = h // G
            o, lse = softmax_rows(q[b, :, h], k[b, k0:k1, g], v[b, k0:k1, g], vis, scale)
            O[b, :, h] = o
            L[b, :, h] = lse
    return O, L


def decode_fwd(q, k, v, scale: float, causal: bool = True
               ) -> Tuple[np.ndarray, np.ndarray]:
    """Attention of the Tq newest tokens against all S cached keys."""
    S = int(np.asarray(k.shape)[1])
    return _decode(q, k, v, scale, causal, 0, S, S)


def decode_partials(q, k, v, scale: float, causal: bool, n_parts: int
                    ) -> List[Tuple[np.ndarray, np.ndarray]]:
    """Partials of n_parts equal contiguous key pieces, in key order."""
    S = int(np.asarray(k.shape)[1])
    assert S % n_parts == 0
    L = S // n_parts
    return [_decode(q, k, v, scale, causal, p * L, (p + 1) * L, S)
            for p in range(n_parts)]
