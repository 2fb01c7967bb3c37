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

// Packed sequences met by a tile: the indices of the sequences holding its
// first and last positions, and the first one's start (all 0 when dense).
struct SegInfo {
  int first, last, start;
};
// `hint` is a sequence index to try first (the previous tile's, since tiles
// are mostly visited in increasing position); the binary search runs only
// when the hint misses.
__device__ __forceinline__ SegInfo seg_info(const AttnParams& P, const TileSpan& t,
                                            int hint = -1) {
  SegInfo r{0, 0, 0};
  if (P.cu == nullptr) return r;
  if (hint >= 0 && hint < P.nseq && __ldg(P.cu + hint) <= t.lo && t.lo < __ldg(P.cu + hint + 1))
    r.first = hint;
  else
    r.first = seg_of(P.cu, P.nseq, t.lo);
  r.start = __ldg(P.cu + r.first);
  r.last = t.hi < __ldg(P.cu + r.first + 1) ? r.first : seg_of(P.cu, P.nseq, t.hi);
  return r;
}

// empty / full / masked for query tile q against key tile k, given the
// sequences each meets (seg_info).
__device__ __forceinline__ int classify(const AttnParams& P, const TileSpan& q,
                                        const SegInfo& qs, const TileSpan& k,
                                        const SegInfo& ks) {
  int qlo = q.lo, qhi = q.hi, klo = k.lo, khi = k.hi;
  if (P.cu != nullptr) {
    if (ks.last < qs.first || ks.first > qs.last) return kClsEmpty;
    if (!(qs.first == qs.last && ks.first == ks.last && qs.first == ks.first))
      return kClsMasked;
    const int st = qs.start;
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

// The same, looking the sequences up.
__device__ __forceinline__ int classify(const AttnParams& P, const TileSpan& q,
                                        const TileSpan& k) {
  return classify(P, q, seg_info(P, q), k, seg_info(P, k));
}

struct PosRange {
  int lo, hi;  // natural positions lo .. hi; empty when lo > hi
};

// Natural positions that can hold keys visible to some query of tile q (a
// superset), in two ranges: the band, from the start of q's first sequence
// (with a window: from q.lo - window + 1) to q.hi (causal) or the end of q's
// last sequence; and, with a window and attention sinks, the sink tokens of
// q's sequences (else empty). Key tiles outside both are empty and are
// rejected with a few comparisons instead of a full classification.
struct KeyWindows {
  PosRange band, sink;
};
__device__ __forceinline__ KeyWindows key_windows(const AttnParams& P, const TileSpan& q) {
  int s0 = 0, s1 = 0, e1 = P.S;
  if (P.cu != nullptr) {
    const int n1 = seg_of(P.cu, P.nseq, q.hi);
    s0 = __ldg(P.cu + seg_of(P.cu, P.nseq, q.lo));
    s1 = __ldg(P.cu + n1);
    e1 = __ldg(P.cu + n1 + 1);
  }
  KeyWindows w;
  w.band.lo = P.window > 0 ? max(s0, q.lo - P.window + 1) : s0;
  w.band.hi = P.causal ? q.hi : e1 - 1;
  if (P.window > 0 && P.sink > 0) {
    w.sink.lo = s0;
    w.sink.hi = s1 + P.sink - 1;
  } else {
    w.sink.lo = 1;
    w.sink.hi = 0;
  }
  return w;
}
// Natural positions [lo, hi] that can hold queries seeing some key of tile k
// (a superset): from k.lo (causal) or the start of k's first sequence to the
// end of k's last sequence, or, with a window, to k.hi + window - 1 unless
// the tile may hold sink tokens (seen by every later query of their
// sequence).
__device__ __forceinline__ PosRange query_window(const AttnParams& P, const TileSpan& k) {
  int s0 = 0, e1 = P.S;
  bool multi = false;
  if (P.cu != nullptr) {
    const int n0 = seg_of(P.cu, P.nseq, k.lo), n1 = seg_of(P.cu, P.nseq, k.hi);
    s0 = __ldg(P.cu + n0);
    e1 = __ldg(P.cu + n1 + 1);
    multi = n0 != n1;
  }
  const bool sinks = P.sink > 0 && (multi || k.lo < s0 + P.sink);
  PosRange r;
  r.lo = P.causal ? k.lo : s0;
  r.hi = (P.window > 0 && !sinks) ? min(e1 - 1, k.hi + P.window - 1) : e1 - 1;
  return r;
}
__device__ __forceinline__ bool disjoint(const TileSpan& t, const PosRange& r) {
  return r.lo > r.hi || t.hi < r.lo || t.lo > r.hi;
}

__device__ __forceinline__ int floor_div(int a, int b) {  // b > 0
  return a >= 0 ? a / b : -((-a + b - 1) / b);
}

// Columns j of tile t (natural position t.lo + j t.step) whose position lies
// in [lo, hi], as the range [a, b) (a == b: none).
struct ColRange {
  int a, b;
};
__device__ __forceinline__ ColRange tile_cols(const TileSpan& t, int lo, int hi) {
  ColRange r;
  r.a = min(kTile, max(0, -floor_div(t.lo - lo, t.step)));  // ceil((lo - t.lo) / step)
  r.b = min(kTile, max(r.a, floor_div(hi - t.lo, t.step) + 1));
  return r;
}
// Bit j (0..31) set when column base + j is in r.
__device__ __forceinline__ uint32_t col_bits(const ColRange& r, int base) {
  const int lo = max(r.a - base, 0), hi = min(r.b - base, 32);
  if (hi <= lo) return 0u;
  const uint32_t below_hi = hi >= 32 ? 0xffffffffu : ((1u << hi) - 1u);
  return below_hi & ~((1u << lo) - 1u);
}

// Permuted tile indices [begin, end) of ring rank `rank`'s shard whose
// natural positions can intersect w. A contiguous or stripe shard is one
// run; a zigzag shard is two chunks, so up to two runs. Returns the count.
struct TileRun {
  int begin, end;
};
__device__ __forceinline__ int shard_runs(const AttnParams& P, int rank, const PosRange& w,
                                          TileRun (&runs)[2]) {
  const int tps = P.shard / kTile;  // tiles per shard
  const int base = rank * tps;
  auto clip = [&](int nat0, int ntiles, int tile0, TileRun& r) {
    // tiles tile0 + t, t in [0, ntiles), hold natural [nat0 + 128 t, +127]
    int a = max(0, floor_div(w.lo - nat0, kTile));
    int b = min(ntiles - 1, floor_div(w.hi - nat0, kTile));
    r.begin = tile0 + a;
    r.end = tile0 + max(a, b + 1);
  };
  if (P.layout == kContiguous) {
    clip(rank * P.shard, tps, base, runs[0]);
    return 1;
  }
  if (P.layout == kZigzag) {
    const int cpt = P.chunk / kTile;  // tiles per chunk
    clip(rank * P.chunk, cpt, base, runs[0]);
    clip((2 * P.cp - 1 - rank) * P.chunk, cpt, base + cpt, runs[1]);
    return 2;
  }
  // stripe: local tile t holds natural (128 t + i) cp + rank, i in [0, 128)
  const int span = kTile * P.cp;
  int a = max(0, -floor_div(-(w.lo - rank - (kTile - 1) * P.cp), span));  // ceil
  int b = min(tps - 1, floor_div(w.hi - rank, span));
  runs[0].begin = base + a;
  runs[0].end = base + max(a, b + 1);
  return 1;
}

// Permuted index of the first token of a natural-order run of `len` tokens
// starting at natural position `pos` (contiguous/zigzag; len divides chunk).
__device__ __forceinline__ int permuted_of(const AttnParams& P, int pos) {
  if (P.layout == kContiguous) return pos;
  int C = P.chunk, c = pos / C, off = pos - c * C;
  if (c < P.cp) return c * P.shard + off;
  return (2 * P.cp - 1 - c) * P.shard + C + off;
}

// Order of the CTAs. The work units (a (batch, head) pair and the tiles of
// its sequence) are taken in batches of `per` units, sized on the host so a
// batch has enough CTAs to fill the GPU but keeps few enough heads in flight
// for their operands (K/V, and in the backward Q/dO and the dQ accumulator)
// to stay in L2. Inside a batch the CTAs go rank-major (heaviest tiles
// first, see below), units minor. Returns the unit and the rank of CTA idx.
struct CtaOrder {
  int unit, rank;
};
__device__ __forceinline__ CtaOrder batched_order(int idx, int nunits, int nranks, int per) {
  const int batch = idx / (per * nranks);
  const int u0 = batch * per;
  const int cnt = min(per, nunits - u0);
  const int r = idx - batch * per * nranks;
  CtaOrder o;
  o.rank = r / cnt;
  o.unit = u0 + r % cnt;
  return o;
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
