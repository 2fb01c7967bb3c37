"""Sequence layouts and the Ulysses all-to-all as index maps (oracle).

Test infrastructure only. These maps are written from the pages' own
descriptions, independently of the CUDA permute kernels:

* contiguous ("basic"): chunk i of cp equal chunks sits on rank i
  (ring-sliding-window README: q/k/v are split into cp_size chunks and chunk
  i goes to rank i).
* zigzag: the sequence is cut into 2*cp chunks and the causal mask is folded
  so rank i holds chunks i and 2*cp-1-i; every pair of chunks on two ranks is
  then a full square or empty, and the work per rank is even ("Long Context
  Attention" notes, "Zig-Zag Attention"; the YunChang README's
  zigzag_extract_local reorders inputs this way for load balance).
* stripe: token t goes to rank t mod cp, so with 16 tokens on 4 ranks rank 0
  holds tokens 0, 4, 8, 12 ("Long Context Attention" notes, "Solution").

The permuted ("rank-major") sequence is the concatenation of rank 0's shard,
rank 1's shard, ... each in increasing natural position.

USP (YunChang README, "2. Usage"): world = ulysses_degree * ring_degree. We
number global ranks w = rho * ud + u (Ulysses groups are runs of adjacent
ranks; the pages fix no order). Rank w holds the u-th 1/ud slice of ring rank
rho's shard, all heads. The Ulysses all-to-all then gives rank (rho, u) all
of rho's tokens for heads [u*H/ud, (u+1)*H/ud). On one device the post
all-to-all buffers are stored as Y[u][b][rho*S/cp + t][h'][d].
"""
from __future__ import annotations

import numpy as np


def shard_positions(layout: str, S: int, cp: int, rank: int) -> np.ndarray:
    """Natural positions held by ring rank `rank`, in increasing order."""
    if layout == "contiguous":
        n = S // cp
        return np.arange(rank * n, (rank + 1) * n)
    if layout == "zigzag":
        c = S // (2 * cp)
        first = np.arange(rank * c, (rank + 1) * c)
        j = 2 * cp - 1 - rank
        second = np.arange(j * c, (j + 1) * c)
        return np.concatenate([first, second])
    if layout == "stripe":
        return np.arange(rank, S, cp)
    raise ValueError(layout)


def permutation(layout: str, S: int, cp: int) -> np.ndarray:
    """perm[p] = natural position stored at permuted index p."""
    return np.concatenate([shard_positions(layout, S, cp, r)
                           for r in range(cp)])


def extract(x: np.ndarray, layout: str, cp: int, axis: int = 1) -> np.ndarray:
    """Natural order -> rank-major permuted order along `axis`."""
    perm = permutation(layout, x.shape[axis], cp)
    return np.take(x, perm, axis=axis)


def restore(x: np.ndarray, layout: str, cp: int, axis: int = 1) -> np.ndarray:
    """Rank-major permuted order -> natural order along `axis`."""
    perm = permutation(layout, x.shape[axis], cp)
    out = np.empty_like(x)
    idx = [slice(None)] * x.ndim
    idx[axis] = perm
    out[tuple(idx)] = x
    return out


def ulysses_seq2head(x: np.ndarray, cp: int, ud: int) -> np.ndarray:
    """All-to-all of a permuted [B, S, H, D] tensor, simulated rank by rank.

    Returns Y [ud, B, S, H/ud, D] as defined in the module docstring.
    """
    B, S, H, D = x.shape
    W = cp * ud
    n = S // W
    hq = H // ud
    # What each global rank holds before the exchange: its sequence slice.
    held = {w: x[:, w * n:(w + 1) * n] for w in range(W)}
    Y = np.empty((ud, B, S, hq, D), dtype=x.dtype)
    for rho in range(cp):
        for u_dst in range(ud):
            # rank (rho, u_dst) receives head slice u_dst from every peer u in
            # its Ulysses group and stacks them along the sequence in u order.
            recv = [held[rho * ud + u][:, :, u_dst * hq:(u_dst + 1) * hq]
                    for u in range(ud)]
            Y[u_dst, :, rho * (S // cp):(rho + 1) * (S // cp)] = \
                np.concatenate(recv, axis=1)
    return Y


def ulysses_head2seq(y: np.ndarray, cp: int, ud: int) -> np.ndarray:
    """Inverse all-to-all: Y [ud, B, S, H/ud, D] -> permuted [B, S, H, D]."""
    _, B, S, hq, D = y.shape
    W = cp * ud
    n = S // W
    x = np.empty((B, S, hq * ud, D), dtype=y.dtype)
    for rho in range(cp):
        for u_src in range(ud):
            # rank (rho, u_src) owns heads u_src*hq.. for all of rho's tokens
            # and returns to peer u the u-th sequence slice.
            block = y[u_src, :, rho * (S // cp):(rho + 1) * (S // cp)]
            for u in range(ud):
                w = rho * ud + u
                x[:, w * n:(w + 1) * n, u_src * hq:(u_src + 1) * hq] = \
                    block[:, u * n:(u + 1) * n]
    return x
