"""Per-step plan of a ring spread over real devices (host logic only).

"Long Context Attention" notes, "Ring Attention": the KV shards of the cp
ring ranks travel round the ring; at step s, ring rank rho holds the shard
that started on rank (rho - s) mod cp, passes it on to rank rho + 1 and
receives the next one from rank rho - 1 while it computes, until every rank
has seen every shard. The backward pass sends each shard's dK/dV along with
it and, after the last step, one hop further, home to the shard's owner (the
notes' "Motivation": dK/dV of a shard collect every query rank's share).
With Ulysses (YunChang README, "2. Usage") global rank w = rho * ud + u and
the all-to-all runs inside each group of ud adjacent ranks.

On one device the library folds all of this into its kernels (a ring hop is
an address offset). This module states the schedule that a multi-device run
follows: which shard each rank computes against at each step, whom it sends
to and receives from, which of two receive buffers the shard occupies (the
next shard lands in the other one while the current one is used), and which
chunk pairs of the step hold visible (query, key) pairs. It holds none of the
attention arithmetic and issues no communication itself.
"""
from __future__ import annotations

import dataclasses
from typing import List, Optional, Tuple

LAYOUTS = ("contiguous", "zigzag", "stripe")

# chunk-pair classes of a step (causal masks; without causality all are full)
FULL, DIAGONAL, STRICT, EMPTY = "full", "diagonal", "strict", "empty"


@dataclasses.dataclass(frozen=True)
class RingStep:
    step: int
    kv_owner: int                  # ring rank whose KV shard is used this step
    buf: int                       # receive buffer holding that shard (0 or 1)
    send_to: Optional[int]         # rank the shard goes to next (None: last step)
    recv_from: Optional[int]       # rank the next shard comes from (None: last step)
    # (query chunk, key chunk, class) of the rank's chunks against the shard's;
    # chunk indices are natural-order chunks (zigzag: 2 cp chunks; contiguous:
    # cp chunks; stripe: the rank's own residue class, one "chunk" per rank)
    pairs: Tuple[Tuple[int, int, str], ...]

    @property
    def has_work(self) -> bool:
        return any(c != EMPTY for _, _, c in self.pairs)


def rank_chunks(rank: int, cp: int, layout: str) -> Tuple[int, ...]:
    """Natural-order chunks a ring rank holds (zigzag: chunks rank and
    2 cp - 1 - rank of 2 cp; contiguous: chunk rank of cp; stripe: its residue
    class, written as the rank itself)."""
    if layout == "zigzag":
        return (rank, 2 * cp - 1 - rank)
    if layout in ("contiguous", "stripe"):
        return (rank,)
    raise ValueError(layout)


def pair_class(qc: int, kc: int, layout: str, causal: bool) -> str:
    """Class of a (query chunk, key chunk) pair under a causal mask.

    Contiguous and zigzag chunks are ranges of natural positions, so an
    earlier key chunk is fully visible, the same chunk is its causal
    diagonal and a later one is empty ("Zig-Zag Attention": every cross-chunk
    pair is full or empty). Stripe "chunks" are residue classes: query
    r + cp i sees key k + cp j iff j <= i when k <= r (a triangle with its
    diagonal) and iff j < i when k > r (without it) -- the notes' "Solution"
    rule of dropping the first query and the last key when the host id is
    below the round.
    """
    if not causal:
        return FULL
    if layout == "stripe":
        return DIAGONAL if kc <= qc else STRICT
    if kc < qc:
        return FULL
    return DIAGONAL if kc == qc else EMPTY


def forward_plan(rank: int, cp: int, layout: str, causal: bool = True) -> List[RingStep]:
    """The cp steps of ring rank `rank` in the forward pass."""
    if not 0 <= rank < cp:
        raise ValueError("rank out of range")
    steps = []
    for s in range(cp):
        owner = (rank - s) % cp
        last = s == cp - 1
        pairs = tuple((qc, kc, pair_class(qc, kc, layout, causal))
                      for qc in rank_chunks(rank, cp, layout)
                      for kc in rank_chunks(owner, cp, layout))
        steps.append(RingStep(step=s, kv_owner=owner, buf=s % 2,
                              send_to=None if last else (rank + 1) % cp,
                              recv_from=None if last else (rank - 1) % cp,
                              pairs=pairs))
    return steps


def backward_plan(rank: int, cp: int, layout: str, causal: bool = True
                  ) -> Tuple[List[RingStep], Tuple[int, int]]:
    """The backward's steps (the forward's, with each shard's dK/dV partial
    travelling beside it) and the final return hop: (destination, source) of
    the dK/dV that this rank sends home and receives home after the last
    step. At the last step rank rho holds shard rho + 1's dK/dV, which goes to
    rank rho + 1; its own comes from rank rho - 1."""
    return forward_plan(rank, cp, layout, causal), ((rank + 1) % cp, (rank - 1) % cp)


def global_rank(rho: int, u: int, ud: int) -> int:
    """Global rank of ring rank rho, Ulysses rank u (Ulysses innermost)."""
    return rho * ud + u


def ulysses_group(w: int, ud: int) -> List[int]:
    """The ud global ranks that exchange heads with global rank w."""
    rho = w // ud
    return [global_rank(rho, u, ud) for u in range(ud)]


def ring_peers(w: int, cp: int, ud: int) -> Tuple[int, int]:
    """(send_to, recv_from) global ranks of w's ring (the ranks with w's
    Ulysses rank, one per ring rank)."""
    rho, u = divmod(w, ud)
    return global_rank((rho + 1) % cp, u, ud), global_rank((rho - 1) % cp, u, ud)
