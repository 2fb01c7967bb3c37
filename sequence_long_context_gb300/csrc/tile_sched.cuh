// Tile-level view of the ring schedule shared by the tensor-core kernels.
//
// The tensor-core kernels work on 128-token tiles of the rank-major
// sequence. They require every tile to lie inside one zigzag chunk (or one
// rank's shard), so the natural positions of a tile's tokens increase with a
// fixed step: 1 for contiguous and zigzag, cp for stripe ("Long Context
// Attention" notes: the stripe permutation deals token t to rank t mod cp).
// A (query tile, key tile) pair is then classified from its extreme
// positions alone: empty (skipped, never loaded), full (no mask arithmetic)
// or masked (each element tested against the row's visible interval).
#pragma once

#include "common.cuh"

namespace usp {

constexpr int kTile = 128;
constexpr int kClsEmpty = 0, kClsFull = 1, kClsMasked = 2;

struct TileSpan {
  int lo, hi, step;  // natural positions lo, lo + step, ..., hi
};

__device__ __forceinline__ TileSpan tile_span(const AttnParams& P, int base) {
  TileSpan t;
  t.lo = nat_pos(P, base);
  t.step = (P.layout == kStripe) ? P.cp : 1;
  t.hi = t.lo + (kTile - 1) * t.step;
  return t;
}

// empty / full / masked for query tile q against key tile k.
__device__ __forceinline__ int classify(const AttnParams& P, const TileSpan& q,
                                        const TileSpan& k) {
  int qlo = q.lo, qhi = q.hi, klo = k.lo, khi = k.hi;
  if (P.cu != nullptr) {
    int sq0 = seg_of(P.cu, P.nseq, qlo), sq1 = seg_of(P.cu, P.nseq, qhi);
    int sk0 = seg_of(P.cu, P.nseq, klo), sk1 = seg_of(P.cu, P.nseq, khi);
    if (sk1 < sq0 || sk0 > sq1) return kClsEmpty;
    if (!(sq0 == sq1 && sk0 == sk1 && sq0 == sk0)) return kClsMasked;
    int st = __ldg(P.cu + sq0);
    qlo -= st; qhi -= st; klo -= st; khi -= st;
  }
  if (P.causal && klo > qhi) return kClsEmpty;
  bool full = !P.causal || khi <= qlo;
  if (P.window > 0) {
    bool any_window = qlo - khi < P.window || (!P.causal && khi > qlo);
    bool any_sink = klo < P.sink;
    if (!any_window && !any_sink) return kClsEmpty;
    bool all_window = qhi - klo < P.window || khi < P.sink;
    full = full && all_window;
  }
  return full ? kClsFull : kClsMasked;
}

// Permuted index of the first token of a natural-order run of `len` tokens
// starting at natural position `pos` (contiguous/zigzag; len divides chunk).
__device__ __forceinline__ int permuted_of(const AttnParams& P, int pos) {
  if (P.layout == kContiguous) return pos;
  int C = P.chunk, c = pos / C, off = pos - c * C;
  if (c < P.cp) return c * P.shard + off;
  return (2 * P.cp - 1 - c) * P.shard + C + off;
}

// Query-tile pairs (256 rows), heaviest first for causal dense problems:
// later natural positions see more keys.
__device__ __forceinline__ int qpair_for_rank(const AttnParams& P, int r, int npairs) {
  if (!P.causal || P.cu != nullptr) return r;
  if (P.layout == kStripe) {
    int ppr = P.shard / (2 * kTile);
    return (r % P.cp) * ppr + (ppr - 1 - r / P.cp);
  }
  return permuted_of(P, (npairs - 1 - r) * 2 * kTile) / (2 * kTile);
}

// Key tiles (128 rows), heaviest first for causal dense problems: earlier
// natural positions are seen by more queries.
__device__ __forceinline__ int ktile_for_rank(const AttnParams& P, int r, int ntiles) {
  if (!P.causal || P.cu != nullptr) return r;
  if (P.layout == kStripe) {
    int tpr = P.shard / kTile;
    return (r % P.cp) * tpr + r / P.cp;
  }
  (void)ntiles;
  return permuted_of(P, r * kTile) / kTile;
}

}  // namespace usp
