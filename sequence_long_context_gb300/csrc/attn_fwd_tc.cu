// Ring attention forward on the 5th-generation tensor cores (tcgen05), bf16
// inputs with fp32 accumulation in tensor memory.
//
// What it computes is the per-rank ring schedule of "Long Context
// Attention" ("Ring Attention": KV shards travel the ring until every host
// has seen all of them; "Tree Attention": partials merge with the
// associative log-sum-exp rule): for virtual ring rank rho the KV shards are
// visited in the order kappa = rho, rho-1, ..., and every visited key tile
// is folded into the running partial (row max m, row sum l, O accumulator),
// which is the unnormalised form of a merged (O, LSE) partial.
//
// One CTA owns one 128-row query tile of one (batch, head); two CTAs share
// an SM. Roles (192 threads):
//   warps 0-3   softmax: one query row per thread
//   warp  4     producer: classifies key tiles (empty / full / masked) and
//               streams K and V tiles with TMA, one slot each
//   warp  5     MMA issuer (one thread) and owner of the CTA's tensor memory
// Tensor memory (256 columns per CTA): S = Q K^T at [0, 128), overwritten in
// place by P (bf16 pairs) which feeds O += P V as the A operand from tensor
// memory; O at [128, 128 + D). P goes to the MMA warp in two halves of 64
// keys, so the first half's P V runs while the second half's exponentials
// are computed, and the two CTAs of an SM interleave their products on the
// tensor core.
// Masks are resolved per 128x128 tile: empty tiles are never loaded, full
// tiles run without any mask arithmetic, masked tiles test each element
// against the row's visible interval. The running max is only moved (and O
// rescaled) when it grows by more than 2^8, which keeps the result exact
// while skipping most rescales.
#include <cudaTypedefs.h>

#include <cstdio>

#include "internal.h"
#include "tc_ptx.cuh"
#include "tile_sched.cuh"

namespace usp {
namespace {

using namespace tc;

// Device status word of this kernel family (USP_ERR_TIMEOUT after a wait
// gave up); read and cleared by usp_device_status().
__device__ int g_fwd_tc_status = 0;

constexpr int kBM = 128;          // query rows per tile
constexpr int kBN = 128;          // keys per tile
constexpr int kEmpty = kClsEmpty, kMasked = kClsMasked;
constexpr int kEnd = -1;
constexpr float kRescaleThreshold = 8.0f;  // log2 units
constexpr float kLn2 = 0.6931471805599453f;

// Named CTA barrier 1, the set-up barrier: the producer warp only arrives
// (the barriers it initialised are ready), the other warps wait for all
// threads (and for the tensor-memory base the MMA warp allocated).
__device__ __forceinline__ void setup_arrive(int threads) {
  asm volatile("bar.arrive 1, %0;" ::"r"(threads) : "memory");
}
__device__ __forceinline__ void setup_sync(int threads) {
  asm volatile("bar.sync 1, %0;" ::"r"(threads) : "memory");
}

// CTA order: units are query heads ordered (kv head, batch, query head of
// the group), so a batch of consecutive units shares K/V.
__device__ __forceinline__ int fwd_head(const AttnParams& P, int unit) {
  return unit / (P.G * P.Bt) * P.G + unit % P.G;
}
__device__ __forceinline__ int fwd_batch(const AttnParams& P, int unit) {
  return (unit / P.G) % P.Bt;
}

// The softmax and epilogue of one query tile, one row per thread of four
// warps (the row's TMEM lane quarter = warp % 4). Per key tile: P =
// 2^(S scale log2e - m) written over S as bf16 pairs (the A operand of P V),
// the running max m moved only when it grows by more than 2^8 (and O
// rescaled then; exact, since O / l and m + log l do not depend on which m
// was used), the row sum accumulated on packed pairs; P is handed over in
// two halves (b_ph, then b_p). Epilogue: O / l as bf16 rows staged in
// `stage` (128-byte swizzle), each warp's 32 rows stored with TMA by its
// first thread, LSE =
// (m + log2 l) ln 2. b_* are the tile's barriers; nranks is the CTA order's
// ranks per unit (to recompute the head late).
template <int D, int kHalfBytes, int kHalves>
__device__ __forceinline__ void softmax_tile(const AttnParams& P, const int2* info,
                                             uint32_t b_info, uint32_t b_s, uint32_t b_ph,
                                             uint32_t b_p, uint32_t b_o,
                                             uint32_t s_tm,
                                             uint32_t o_tm, uint8_t* stage,
                                             const CUtensorMap* tm_o, int qrow0, int quarter,
                                             int lane, int nranks, volatile int* abort_flag) {
  const int r = quarter * 32 + lane;       // row within the tile = TMEM lane
  const int prow = qrow0 + r;              // permuted query row
  const RowMask rm = row_mask(P, nat_pos(P, prow));
  float m_run = -INFINITY, l_run = 0.f;
  int c = 0;
  bool ok = true;
  while (true) {
    ok = mbar_wait(b_info, c & 1, abort_flag, P.status);
    if (!(ok = __all_sync(0xffffffffu, ok))) break;
    const int2 inf = *info;
    if (inf.x == kEnd) break;
    // a masked tile: this row's visible keys in the tile (the main
    // interval and the sink interval of row_visible) as one bit per column
    uint32_t vis[4] = {~0u, ~0u, ~0u, ~0u};
    if (inf.y == kMasked) {
      const TileSpan ks = tile_span(P, inf.x * kBN);
      const ColRange c0 = tile_cols(ks, rm.lo, rm.hi);
      const ColRange c1 = tile_cols(ks, rm.qs, min(rm.sink_end - 1, rm.causal_hi));
#pragma unroll
      for (int ch = 0; ch < 4; ++ch) vis[ch] = col_bits(c0, 32 * ch) | col_bits(c1, 32 * ch);
    }
    ok = mbar_wait(b_s, c & 1, abort_flag, P.status);
    if (!(ok = __all_sync(0xffffffffu, ok))) break;
    tc_fence_after();
    uint32_t sr[4][32];
#pragma unroll
    for (int ch = 0; ch < 4; ++ch) tmem_ld32(s_tm + 32 * ch, sr[ch]);
    tmem_wait_ld();
    if (inf.y == kMasked) {
#pragma unroll
      for (int ch = 0; ch < 4; ++ch)
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if (!((vis[ch] >> j) & 1u)) sr[ch][j] = __float_as_uint(-INFINITY);
    }
    // row max as 8 independent chains (a single chain is latency-bound)
    float m8[8];
#pragma unroll
    for (int t = 0; t < 8; ++t) m8[t] = __uint_as_float(sr[t >> 5][t & 31]);
#pragma unroll
    for (int j = 8; j < 128; ++j)
      m8[j & 7] = fmaxf(m8[j & 7], __uint_as_float(sr[j >> 5][j & 31]));
    float mx = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])),
                     fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7])));
    mx *= P.scale_log2;
    // lazy rescale: move the running max only when it grows by > 2^8
    const bool need = mx > m_run + kRescaleThreshold;
    float alpha = 1.f;
    if (need) {
      alpha = (m_run == -INFINITY) ? 0.f : ex2(m_run - mx);
      m_run = mx;
    }
    l_run *= alpha;
    const float msub = (m_run == -INFINITY) ? 0.f : m_run;
    // p = exp2(s * scale_log2 - m): scale-and-subtract and the row sum run
    // on packed fp32 pairs (one FMA-pipe instruction per two elements). P
    // goes over S as bf16 pairs in two halves of 64 keys, each handed to the
    // MMA warp as soon as it is written (b_ph, then b_p), so the first
    // half's P V overlaps the second half's exponentials.
    const uint64_t sc2 = f2_pack(P.scale_log2, P.scale_log2);
    const uint64_t nm2 = f2_pack(-msub, -msub);
    uint64_t ls2[4] = {0, 0, 0, 0};
    // O_i holds PV of the previous tiles (complete: the commit that
    // signalled S_i tracks every earlier MMA); it is rescaled to the new max
    // before P_i V is accumulated onto it
    auto rescale_o = [&]() {
      if (__any_sync(0xffffffffu, need && c > 0)) {
#pragma unroll
        for (int oc = 0; oc < D / 32; ++oc) {
          uint32_t o[32];
          tmem_ld32(o_tm + 32 * oc, o);
          tmem_wait_ld();
#pragma unroll
          for (int jj = 0; jj < 32; ++jj)
            o[jj] = __float_as_uint(__uint_as_float(o[jj]) * alpha);
          tmem_st32(o_tm + 32 * oc, o);
        }
      }
    };
#pragma unroll
    for (int ch = 0; ch < 2; ++ch) {
      uint32_t pk[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const int j0 = 64 * ch + 2 * j;
        const uint64_t x = f2_fma(
            f2_pack(__uint_as_float(sr[j0 >> 5][j0 & 31]),
                    __uint_as_float(sr[(j0 + 1) >> 5][(j0 + 1) & 31])),
            sc2, nm2);
        float x0, x1;
        f2_unpack(x, x0, x1);
        const float p0 = ex2(x0), p1 = ex2(x1);
        ls2[j & 3] = f2_add(ls2[j & 3], f2_pack(p0, p1));
        pk[j] = pack_bf16(p0, p1);
      }
      tmem_st32(s_tm + 32 * ch, pk);
      if (ch == 0) rescale_o();  // before the first half goes
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(ch == 0 ? b_ph : b_p);  // one arrival per warp
    }
    {
      float a0, a1, b0, b1, c0, c1, d0, d1;
      f2_unpack(ls2[0], a0, a1);
      f2_unpack(ls2[1], b0, b1);
      f2_unpack(ls2[2], c0, c1);
      f2_unpack(ls2[3], d0, d1);
      l_run += ((a0 + a1) + (b0 + b1)) + ((c0 + c1) + (d0 + d1));
    }
    ++c;
  }
  // epilogue: O / l -> bf16 rows, LSE = (m + log2 l) ln 2. The rows are
  // staged in the 128-byte swizzle in this query tile's shared-memory slot
  // (free: every Q K^T has completed when O is) and each warp stores its
  // own 32 rows with TMA.
  if (ok) ok = mbar_wait(b_o, 0, abort_flag, P.status);
  ok = __all_sync(0xffffffffu, ok);
  tc_fence_after();
  // the CTA's head and batch, recomputed (not kept live through the loop)
  const int unit = batched_order(blockIdx.x, P.Hq * P.Bt, nranks, P.unit_batch).unit;
  const int h = fwd_head(P, unit), bt = fwd_batch(P, unit);
  if (ok) {
    const float inv = (l_run > 0.f) ? 1.f / l_run : 0.f;
    // all of O's columns in one round trip to tensor memory
    uint32_t ov[D / 32][32];
#pragma unroll
    for (int ch = 0; ch < D / 32; ++ch) tmem_ld32(o_tm + 32 * ch, ov[ch]);
    tmem_wait_ld();
#pragma unroll
    for (int ch = 0; ch < D / 32; ++ch) {
      const uint32_t* o = ov[ch];
      uint32_t wp[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const float a = (c > 0) ? __uint_as_float(o[2 * j]) * inv : 0.f;
        const float b = (c > 0) ? __uint_as_float(o[2 * j + 1]) * inv : 0.f;
        wp[j] = pack_bf16(a, b);
      }
      // columns 32 ch .. 32 ch + 31 = 16-byte chunks 4 ch .. 4 ch + 3 of
      // the row, in 64-column halves
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int c8 = 4 * ch + q, hf = c8 >> 3, chunk = c8 & 7;
        *reinterpret_cast<uint4*>(stage + hf * kHalfBytes + r * 128 +
                                  ((chunk ^ (r & 7)) << 4)) =
            make_uint4(wp[4 * q], wp[4 * q + 1], wp[4 * q + 2], wp[4 * q + 3]);
      }
    }
    fence_proxy_async_smem();  // the staged rows are read next by the TMA unit
    __syncwarp();
    if (lane == 0) {
      // this warp's 32 rows (1024-byte aligned in the staging, so the
      // swizzle phase is the tile's), no wait for the other warps
      const TensorPos t = tensor_pos(P, h, qrow0, bt, P.Hq);
      for (int hf = 0; hf < kHalves; ++hf)
        tma_store_4d(tm_o, smem_u32(stage + hf * kHalfBytes + quarter * 32 * 128), hf * 64,
                     t.h, t.row + 32 * quarter, t.b);
      bulk_commit_group();
      // the rows have been read out of shared memory before the CTA exits
      // (the global writes complete on their own)
      bulk_wait_group_read0();
    }
    P.lse[lse_index(P, bt, h, prow)] =
        (l_run > 0.f) ? (m_run + log2f(l_run)) * kLn2 : -INFINITY;
  }
}

// ---------------------------------------------------------------------------
// The kernel. One query tile per CTA (S at [0,128) of the CTA's 256 tensor
// memory columns, overwritten by P, O at [128, 128+D); one Q tile, one K and
// one V slot of shared memory), so the SM runs two CTAs: one's start and end
// overlap the other's loop, and their Q K^T and P V products interleave on
// the tensor core.
constexpr int kThreads = 192;      // softmax warps 0-3, producer 4, MMA 5
constexpr int kProducerWarp = 4;
constexpr int kMmaWarp = 5;

template <int D>
struct Smem {
  static constexpr int kHalves = D / 64;
  static constexpr int kTileBytes = kBM * D * 2;
  static constexpr int kHalfBytes = kBM * 128;
  static constexpr int kQ = 0;
  static constexpr int kK = kQ + kTileBytes;
  static constexpr int kV = kK + kTileBytes;
  static constexpr int kBar = kV + kTileBytes;
  static constexpr int kQFull = 0, kKFull = 1, kKEmpty = 2, kVFull = 3, kVEmpty = 4,
                       kSFull = 5, kPFull = 6, kOFull = 7, kInfoFull = 8, kMmaDone = 9,
                       kPHalf = 10, kNumBars = 11;
  static constexpr int kSched = (kBar + 8 * kNumBars + 15) / 16 * 16;  // int4
  static constexpr int kInfo = kSched + 16;                           // int2
  static constexpr int kMisc = kInfo + 16;                            // tmem base, abort
  static constexpr int kBytes = kMisc + 16;
  static constexpr int kAlloc = kBytes + 1024;
  static_assert(kK % 1024 == 0 && kV % 1024 == 0, "swizzled tiles need 1024-byte alignment");
  static_assert(2 * kAlloc <= 232448, "two CTAs must fit one SM's shared memory");
};

// Query tiles (128 rows), heaviest first for causal dense problems.
__device__ __forceinline__ int qtile_for_rank(const AttnParams& P, int r, int ntiles) {
  if (!P.causal || P.cu != nullptr) return r;
  if (P.layout == kStripe) {
    const int tpr = P.shard / kBM;
    return (r % P.cp) * tpr + (tpr - 1 - r / P.cp);
  }
  return permuted_of(P, (ntiles - 1 - r) * kBM) / kBM;
}

template <int D>
__global__ void __launch_bounds__(kThreads, 2)
attn_fwd_tc_kernel(const AttnParams P, const __grid_constant__ CUtensorMap tm_q,
                    const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v,
                    const __grid_constant__ CUtensorMap tm_o) {
  using L = Smem<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(sm);
  auto bar = [&](int i) { return sbase + L::kBar + 8 * i; };
  int4* sched = reinterpret_cast<int4*>(sm + L::kSched);
  int2* info = reinterpret_cast<int2*>(sm + L::kInfo);
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(sm + L::kMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + L::kMisc + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ntiles = P.S / kBM;
  const CtaOrder ord = batched_order(blockIdx.x, P.Hq * P.Bt, ntiles, P.unit_batch);
  const int qt = qtile_for_rank(P, ord.rank, ntiles);
  const int h = fwd_head(P, ord.unit), bt = fwd_batch(P, ord.unit);
  const int g = h / P.G;
  const int qbase = qt * kBM;            // permuted row of the tile
  const int rho = qbase / P.shard;       // its ring rank

  // the producer thread sets up the barriers and starts the Q load
  if (warp == kProducerWarp && lane == 0) {
    mbar_init(bar(L::kQFull), 1);
    mbar_init(bar(L::kKFull), 1);
    mbar_init(bar(L::kKEmpty), 1);
    mbar_init(bar(L::kVFull), 1);
    mbar_init(bar(L::kVEmpty), 1);
    mbar_init(bar(L::kSFull), 1);
    mbar_init(bar(L::kPFull), kBM / 32);    // one arrival per softmax warp
    mbar_init(bar(L::kPHalf), kBM / 32);
    mbar_init(bar(L::kOFull), 1);
    mbar_init(bar(L::kInfoFull), 1);
    mbar_init(bar(L::kMmaDone), 1);
    *abort_flag = 0;
    fence_barrier_init();
    tma_prefetch(&tm_q);
    tma_prefetch(&tm_k);
    tma_prefetch(&tm_v);
    mbar_expect_tx(bar(L::kQFull), L::kTileBytes);
    const TensorPos t = tensor_pos(P, h, qbase, bt, P.Hq);
    for (int hf = 0; hf < L::kHalves; ++hf)
      tma_load_4d(sbase + L::kQ + hf * L::kHalfBytes, &tm_q, bar(L::kQFull), hf * 64, t.h,
                  t.row, t.b);
  }
  if (warp == kMmaWarp) {
    tmem_alloc(sbase + L::kMisc, 256);
    tmem_relinquish();
  }
  // The producer needs nothing from the other warps' set-up: it signals that
  // the barriers exist and goes straight on to classify and load the key
  // tiles, so that the first K/V loads overlap the tensor-memory allocation.
  uint32_t tmem = 0;  // the producer never uses it
  if (warp == kProducerWarp) {
    __syncwarp();
    setup_arrive(kThreads);
  } else {
    tc_fence_before();
    setup_sync(kThreads);
    tc_fence_after();
    tmem = *tmem_holder;
  }

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const TileSpan q0 = tile_span(P, qbase);
      const KeyWindows w0 = key_windows(P, q0);
      int n = 0;   // key tiles with K and V issued
      int nk = 0;  // key tiles with K issued
      bool ok = true;
      const SegInfo sq0 = seg_info(P, q0);
      int khint = sq0.first;
      // one key tile: classified for the query tile, loaded unless empty;
      // K and V have one slot each, freed by the tile's Q K^T and P V
      auto visit = [&](int kt) {
        const TileSpan ks = tile_span(P, kt * kBN);
        if (disjoint(ks, w0.band) && disjoint(ks, w0.sink)) return;
        const SegInfo sk = seg_info(P, ks, khint);
        khint = sk.last;
        const int c0 = classify(P, q0, sq0, ks, sk);
        if (c0 == kEmpty) return;
        if (n >= 1 && !(ok = mbar_wait(bar(L::kKEmpty), (n - 1) & 1, abort_flag, P.status)))
          return;
        *sched = make_int4(kt, c0, 0, 0);
        const TensorPos kv = tensor_pos(P, g, kt * kBN, bt, P.Hkv);
        mbar_expect_tx(bar(L::kKFull), L::kTileBytes);
        for (int hf = 0; hf < L::kHalves; ++hf)
          tma_load_4d(sbase + L::kK + hf * L::kHalfBytes, &tm_k, bar(L::kKFull), hf * 64, kv.h,
                      kv.row, kv.b);
        ++nk;
        if (n >= 1 && !(ok = mbar_wait(bar(L::kVEmpty), (n - 1) & 1, abort_flag, P.status)))
          return;
        mbar_expect_tx(bar(L::kVFull), L::kTileBytes);
        for (int hf = 0; hf < L::kHalves; ++hf)
          tma_load_4d(sbase + L::kV + hf * L::kHalfBytes, &tm_v, bar(L::kVFull), hf * 64, kv.h,
                      kv.row, kv.b);
        ++n;
      };
      for (int s = 0; s < P.cp && ok; ++s) {
        const int kap = (rho - s + P.cp) % P.cp;
        TileRun sr[2], br[2];
        const int nsr = w0.sink.lo <= w0.sink.hi ? shard_runs(P, kap, w0.sink, sr) : 0;
        const int nbr = shard_runs(P, kap, w0.band, br);
        for (int ri = 0; ri < nsr && ok; ++ri)
          for (int kt = sr[ri].begin; kt < sr[ri].end && ok; ++kt) visit(kt);
        for (int ri = 0; ri < nbr && ok; ++ri)
          for (int kt = br[ri].begin; kt < br[ri].end && ok; ++kt) {
            bool seen = false;
            for (int rj = 0; rj < nsr; ++rj) seen |= kt >= sr[rj].begin && kt < sr[rj].end;
            if (!seen) visit(kt);
          }
      }
      if (ok) {
        if (n < 1 || mbar_wait(bar(L::kKEmpty), (n - 1) & 1, abort_flag, P.status)) {
          *sched = make_int4(kEnd, 0, 0, 0);
          mbar_arrive(bar(L::kKFull));
        }
        // the last V has been consumed before the CTA may exit
        if (n >= 1) mbar_wait(bar(L::kVEmpty), (n - 1) & 1, abort_flag, P.status);
      }
      if (*abort_flag) {
        // aborted: let the copies already issued land before the CTA exits
        mbar_wait_drain(bar(L::kQFull), 0);
        if (nk >= 1) mbar_wait_drain(bar(L::kKFull), (nk - 1) & 1);
        if (n >= 1) mbar_wait_drain(bar(L::kVFull), (n - 1) & 1);
      }
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    // Per key tile n: S = Q K^T (then the K slot is free), P V once the
    // softmax has written P over S (then the V slot is free). The next
    // Q K^T follows this P V in issue order, so S may overwrite P in place.
    if (lane == 0) {
      constexpr uint32_t kIdQK = idesc_bf16_f32(kBM, kBN, 0, 0);
      constexpr uint32_t kIdPV = idesc_bf16_f32(kBM, D, 0, 1);
      const uint32_t s_tm = tmem, o_tm = tmem + 128;
      const uint64_t dq0 = sdesc_sw128(sbase + L::kQ, 16, 1024);
      const uint64_t dk0 = sdesc_sw128(sbase + L::kK, 16, 1024);
      const uint64_t dv0 = sdesc_sw128(sbase + L::kV, L::kHalfBytes, 1024);
      bool ok = mbar_wait(bar(L::kQFull), 0, abort_flag, P.status);
      int n = 0;
      while (ok) {
        if (!(ok = mbar_wait(bar(L::kKFull), n & 1, abort_flag, P.status))) break;
        const int4 e = *sched;
        if (e.x == kEnd) break;
        tc_fence_after();
        *info = make_int2(e.x, e.y);
        mbar_arrive(bar(L::kInfoFull));
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * L::kHalfBytes + (kk & 3) * 32;
          mma_ss(s_tm, sdesc_add(dq0, off), sdesc_add(dk0, off), kIdQK, kk > 0 ? 1u : 0u);
        }
        mma_commit(bar(L::kSFull));
        mma_commit(bar(L::kKEmpty));
        // the first 64 keys' P as soon as the softmax has written them
        if (!(ok = mbar_wait(bar(L::kPHalf), n & 1, abort_flag, P.status))) break;
        if (!(ok = mbar_wait(bar(L::kVFull), n & 1, abort_flag, P.status))) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < kBN / 32; ++kk)
          mma_ts(o_tm, s_tm + kk * 8, sdesc_add(dv0, kk * 2048), kIdPV,
                 (n > 0 || kk > 0) ? 1u : 0u);
        if (!(ok = mbar_wait(bar(L::kPFull), n & 1, abort_flag, P.status))) break;
        tc_fence_after();
#pragma unroll
        for (int kk = kBN / 32; kk < kBN / 16; ++kk)
          mma_ts(o_tm, s_tm + kk * 8, sdesc_add(dv0, kk * 2048), kIdPV, 1u);
        mma_commit(bar(L::kVEmpty));
        ++n;
      }
      mma_commit(bar(L::kOFull));
      *info = make_int2(kEnd, 0);
      mbar_arrive(bar(L::kInfoFull));
      // nothing of ours may still run on the tensor core when TMEM is freed
      mma_commit(bar(L::kMmaDone));
      mbar_wait_drain(bar(L::kMmaDone), 0);
    }
  } else {
    // ------------------------------------------------------------ softmax
    // one query row per thread
    const int quarter = warp & 3;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    softmax_tile<D, L::kHalfBytes, L::kHalves>(
        P, info, bar(L::kInfoFull), bar(L::kSFull), bar(L::kPHalf), bar(L::kPFull),
        bar(L::kOFull),
        tmem + lane_off, tmem + lane_off + 128, sm + L::kQ, &tm_o, qbase,
        quarter, lane, ntiles, abort_flag);
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp) tmem_dealloc(tmem, 256);
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (fn == nullptr) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// [Bt][S][H][D] bf16 -> 4-D map (D, H, S, Bt), box (64, 1, rows, 1), 128B swizzle.
// tok: elements between tokens (0: dense H*D; 3*H*D in a packed q/k/v tensor)
bool make_map(CUtensorMap* m, const void* base, int Bt, int S, int H, int D,
              long long tok = 0, int rows = kBM) {
  if (tok == 0) tok = (long long)H * D;
  auto fn = encode_fn();
  if (!fn) {
    fail_cuda_msg("cuTensorMapEncodeTiled", "driver entry point not found");
    return false;
  }
  cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)S, (cuuint64_t)Bt};
  cuuint64_t strides[3] = {(cuuint64_t)D * 2, (cuuint64_t)tok * 2,
                           (cuuint64_t)S * tok * 2};
  cuuint32_t box[4] = {64, 1, (cuuint32_t)rows, 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims,
                  strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    char msg[64];
    std::snprintf(msg, sizeof(msg), "CUresult %d", (int)r);
    fail_cuda_msg("cuTensorMapEncodeTiled", msg);
    return false;
  }
  return true;
}

template <int D>
usp_status_t launch_d(const AttnParams& P, cudaStream_t st) {
  CUtensorMap mq, mk, mv, mo;
  // natural-order tensors in place: all heads of every token, B batch rows
  const int Bm = P.nat ? P.B : P.Bt, hm = P.nat ? P.ud : 1;
  if (!make_map(&mq, P.q, Bm, P.S, P.Hq * hm, D, P.qkv_tok) ||
      !make_map(&mk, P.k, Bm, P.S, P.Hkv * hm, D, P.qkv_tok) ||
      !make_map(&mv, P.v, Bm, P.S, P.Hkv * hm, D, P.qkv_tok) ||
      !make_map(&mo, P.o, Bm, P.S, P.Hq * hm, D, 0, 32))  // O: one warp's rows
    return USP_ERR_CUDA;  // detail recorded by make_map
  static int* status = nullptr;
  if (status == nullptr) {
    cudaError_t e = cudaGetSymbolAddress(reinterpret_cast<void**>(&status), g_fwd_tc_status);
    if (e != cudaSuccess) return fail_cuda("cudaGetSymbolAddress(status)", e);
  }
  AttnParams Pk = P;
  Pk.status = status;
  // L2 batches of about eight waves of CTAs (two per SM), in whole GQA
  // groups. One query tile per CTA on every problem: on dense rings this ran
  // 8-11 % faster than a kernel with two query tiles per CTA ping-ponging on
  // one tensor core (S=32K 6.57 -> 5.93 ms), and more on windowed problems and
  // packed sequences (short key ranges per query tile).
  const int ntiles = P.S / kBM;
  int per = (16 * sm_count() + ntiles - 1) / ntiles;
  per = (per + P.G - 1) / P.G * P.G;
  // packed sequences: one batch (a query tile only meets the keys of its own
  // sequence; measured 4 % faster on the 128K packed batch than 8 waves)
  if (P.cu != nullptr) per = P.Hq * P.Bt;
  Pk.unit_batch = per < P.Hq * P.Bt ? per : P.Hq * P.Bt;
  const int smem = Smem<D>::kAlloc;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(attn_fwd_tc_kernel<D>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return fail_cuda("cudaFuncSetAttribute(smem)", e);
    attr_set = true;
  }
  const long long blocks = (long long)ntiles * P.Hq * P.Bt;
  {
    ProfScope ps(st, "attn_fwd_tc");
    attn_fwd_tc_kernel<D><<<(unsigned)blocks, kThreads, smem, st>>>(Pk, mq, mk, mv, mo);
  }
  note_launch();
  return check_launch();
}

}  // namespace

int read_clear_fwd_tc_status() {
  int v = 0, z = 0;
  if (cudaMemcpyFromSymbol(&v, g_fwd_tc_status, sizeof(int)) != cudaSuccess) return -1;
  if (v != 0) cudaMemcpyToSymbol(g_fwd_tc_status, &z, sizeof(int));
  return v;
}

bool fwd_tc_supported(const AttnParams& P) {
  if (P.D != 128 && P.D != 64) return false;
  if (P.shard % kBM != 0) return false;
  if (P.layout == kZigzag && P.chunk % kBM != 0) return false;
  return true;
}

usp_status_t launch_fwd_tc(const AttnParams& P, cudaStream_t st) {
  return P.D == 128 ? launch_d<128>(P, st) : launch_d<64>(P, st);
}

}  // namespace usp
