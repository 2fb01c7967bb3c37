// Ring attention backward on the tcgen05 tensor cores (bf16 in, fp32 acc).
//
// Gradient of the ring forward from its saved LSE ("Long Context Attention"
// notes, "Motivation": QKV, output, LSE and dout are what the backward
// needs). With P = exp(scale q.k - LSE) and Delta_i = <dO_i, O_i>:
//   dV = P^T dO,  dS = P * (dO V^T - Delta),  dK = scale dS^T Q,
//   dQ = scale dS K.
// One CTA owns one 128-key tile of one KV head. The shard the tile belongs
// to visits the query ranks in ring order (kappa, kappa+1, ...), and for each
// query tile every query head of the GQA group is taken in turn, so dK and
// dV accumulate in tensor memory over the whole ring and the group and are
// written once (the shard's ring return). dQ contributions are added into an
// fp32 accumulator in global memory by TMA reduce-add operations.
//
// Roles (608 threads):
//   warps 0-15  softmax, four threads per key row (warp w owns query columns
//              [32 (w/4), 32 (w/4) + 32)): P^T = exp2(S^T - LSE),
//              dS^T = P^T (dP^T - Delta); P^T and dS^T go back to tensor
//              memory as bf16 (A operands of dV and dK) and dS to shared
//              memory (A operand of dQ). No row reductions are needed (P
//              comes from the saved LSE), so the columns split freely; four
//              warps per TMEM lane quarter hide the latency of each phase.
//              Then, while the next tile's S^T is computed, the same warps
//              take the tile's dQ out of tensor memory (warp w: query rows
//              [32 (w%4), +32), dQ columns [32 (w/4), +32); one load each,
//              freeing the columns for the next dP^T) and stage it, scaled,
//              in the Q and dO tiles of the tile's ring slot (dead once the
//              tile's dK and dQ MMAs are done)
//   warp 16    dQ reduction: has the TMA unit add the staged dQ into the
//              global fp32 accumulator, and hands the Q and dO halves of the
//              slot back once the TMA has read them
//   warp 17    producer: K, V once; then Q, dO tiles through a 2-slot ring;
//              each half of a slot (the Q half also holds the LSE and Delta
//              rows) is refilled once the dQ reduction hands it back
//   warp 18    MMA issuer and tensor-memory owner
// Tensor memory (512 columns): S^T [0,128); the 32 queries of column chunk
// c live in columns [32c, 32c+32) and are overwritten in place by their P^T
// (bf16 pairs, first 16 columns) and dS^T (last 16); dP^T [128,256),
// overwritten by dQ (fp32, D columns); dV [256, 256+D); dK [256+D, 256+2D).
#include <cudaTypedefs.h>

#include <cstdio>

#include "internal.h"
#include "tc_ptx.cuh"
#include "tile_sched.cuh"

namespace usp {
namespace {

using namespace tc;

__device__ int g_bwd_tc_status = 0;

// Packed product of two fp32 pairs (one FMA-pipe instruction).
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

constexpr int kSoftWarps = 16;  // four per TMEM lane quarter, one per 32 queries
constexpr int kReduceWarp = kSoftWarps;
constexpr int kProducerWarp = kReduceWarp + 1;
constexpr int kMmaWarp = kProducerWarp + 1;
constexpr int kThreads = 32 * (kMmaWarp + 1);  // 608
constexpr int kEnd = -1;

template <int D>
struct BSmem {
  static constexpr int kHalves = D / 64;
  static constexpr int kTileBytes = kTile * D * 2;
  static constexpr int kHalfBytes = kTile * 128;
  static constexpr int kK = 0;
  static constexpr int kV = kK + kTileBytes;
  static constexpr int kQ = kV + kTileBytes;        // 2 slots
  static constexpr int kDO = kQ + 2 * kTileBytes;   // 2 slots
  static constexpr int kDS = kDO + 2 * kTileBytes;  // 128 x 128 bf16
  // per Q/dO slot: the query tile's LSE*log2e then Delta, 128 fp32 each,
  // copied in by the producer with the tile
  static constexpr int kStatBytes = 2 * kTile * 4;
  static constexpr int kStats = kDS + kTile * kTile * 2;
  static constexpr int kBar = kStats + 2 * kStatBytes;
  static constexpr int kKVFull = 0, kQFull = 1, kQEmpty = 3, kSFull = 5, kDPFull = 6,
                       kDSFull = 7, kDQFull = 8, kDQEmpty = 9, kInfoS = 10, kInfoQ = 11,
                       kDKVFull = 12, kMmaDone = 13, kPReady = 14, kDQStaged = 15,
                       kDOFull = 16, kStageFreeDO = 18, kStageFreeQ = 20, kKVStaged = 22,
                       kNumBars = 24;
  // Each Q/dO slot has two halves with their own full/free barriers: the Q
  // half (Q tile, LSE and Delta rows; kQFull / kStageFreeQ) and the dO half
  // (kDOFull / kStageFreeDO). Once the tile's dQ MMA is done (the dO half)
  // and its dK MMA too (kQEmpty, the commit of the tile's last MMA: the Q
  // tile), the tile's dQ is staged through both, and the dQ reduction hands
  // each back when the TMA unit has read it. kDQEmpty: the dQ columns have
  // been read (and the reduction warp has read the tile's entry);
  // kDQStaged: every dQ row is staged.
  // 16-byte aligned: int4 / float4 accesses below
  static constexpr int kSched = (kBar + 8 * kNumBars + 15) / 16 * 16;  // int4 x 2
  static constexpr int kInfo = kSched + 32;           // int4 x 2 (softmax, dQ)
  static constexpr int kMisc = kInfo + 32;            // tmem base, abort
  static constexpr int kBytes = kMisc + 16;
  // No alignment slack: the dynamic shared window starts 1024-byte aligned
  // (checked at kernel entry).
  static constexpr int kAlloc = kBytes;
  static_assert(kSched % 16 == 0 && kInfo % 16 == 0 && kStats % 16 == 0,
                "vector accesses need 16-byte alignment");
  static_assert(kDS % 1024 == 0 && kQ % 1024 == 0 && kDO % 1024 == 0,
                "128-byte swizzled tiles need 1024-byte alignment");
  static_assert(kAlloc <= 232448, "exceeds the per-CTA shared memory limit");
};

// Visible query interval of one key (natural positions): a key at position j
// of a sequence [s, e) is seen by queries i in [j (causal) or s,
// j + window - 1 (window, unless j is one of the first sink_tokens) or e-1].
struct ColMask {
  int lo, hi;
};

__device__ __forceinline__ ColMask col_mask(const AttnParams& P, int j) {
  int ks = 0, ke = P.S;
  if (P.cu != nullptr) {
    int n = seg_of(P.cu, P.nseq, j);
    ks = __ldg(P.cu + n);
    ke = __ldg(P.cu + n + 1);
  }
  ColMask m;
  m.lo = P.causal ? j : ks;
  m.hi = ke - 1;
  if (P.window > 0 && j - ks >= P.sink) m.hi = min(m.hi, j + P.window - 1);
  return m;
}

// 19 warps: five share a 16K-register sub-partition, so <= 102 each (96 in
// the allocation's steps of 8).
template <int D>
__global__ void __maxnreg__(96)
attn_bwd_tc_kernel(const AttnParams P, const __grid_constant__ CUtensorMap tm_q,
                   const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v,
                   const __grid_constant__ CUtensorMap tm_do,
                   const __grid_constant__ CUtensorMap tm_dq,
                   const __grid_constant__ CUtensorMap tm_dk,
                   const __grid_constant__ CUtensorMap tm_dv) {
  using L = BSmem<D>;
  // dQ staging: D/32 boxes of 32 fp32 columns x 128 rows (16 KB each) in the
  // 128-byte swizzle; the first half fill the Q tile of the tile's slot, the
  // rest its dO tile. The softmax warps of column chunks ch < D/32 read and
  // stage box ch.
  constexpr int kBoxBytes = kTile * 128;
  constexpr int kBoxes = D / 32;
  constexpr int kBoxesInQ = L::kTileBytes / kBoxBytes;
  constexpr int kDQWarps = 4 * kBoxes;
  static_assert(kBoxesInQ >= 1 && kBoxesInQ < kBoxes, "staging needs both halves");
  static_assert((kBoxes - kBoxesInQ) * kBoxBytes <= L::kTileBytes,
                "staging exceeds the dO half");
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // the swizzled tiles need a 1024-byte aligned window; there is no slack to
  // realign into, so a misaligned window is reported and the CTA does nothing
  if (smem_u32(smem_raw) & 1023u) {
    if (threadIdx.x == 0) atomicExch(P.status, kStatusCudaError);
    return;
  }
  uint8_t* sm = smem_raw;
  const uint32_t sbase = smem_u32(sm);
  auto bar = [&](int i) { return sbase + L::kBar + 8 * i; };
  auto stage_box = [&](int slot, int cg) -> uint8_t* {
    return cg < kBoxesInQ ? sm + L::kQ + slot * L::kTileBytes + cg * kBoxBytes
                          : sm + L::kDO + slot * L::kTileBytes + (cg - kBoxesInQ) * kBoxBytes;
  };
  int4* sched = reinterpret_cast<int4*>(sm + L::kSched);
  int4* info = reinterpret_cast<int4*>(sm + L::kInfo);
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(sm + L::kMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + L::kMisc + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ntiles = P.S / kTile;
  const CtaOrder ord = batched_order(blockIdx.x, P.Hkv * P.Bt, ntiles, P.unit_batch);
  const int kt = ktile_for_rank(P, ord.rank, ntiles);
  const int g = ord.unit / P.Bt, bt = ord.unit % P.Bt;
  const int kappa = (kt * kTile) / P.shard;  // ring rank owning the key tile

  // The producer thread sets up the barriers and starts the K and V tiles'
  // load before the CTA-wide barrier, so the load overlaps the set-up.
  if (warp == kProducerWarp && lane == 0) {
    mbar_init(bar(L::kKVFull), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(L::kQFull + s), 1);
      mbar_init(bar(L::kQEmpty + s), 1);
    }
    mbar_init(bar(L::kSFull), 1);
    mbar_init(bar(L::kDPFull), 1);
    mbar_init(bar(L::kDSFull), kSoftWarps);  // one arrival per softmax warp
    mbar_init(bar(L::kDQFull), 1);
    // one arrival per softmax warp that reads dQ columns, and one by the
    // reduction warp once it has read the tile's entry
    mbar_init(bar(L::kDQEmpty), kDQWarps + 1);
    mbar_init(bar(L::kDQStaged), kDQWarps);   // one arrival per such warp
    for (int s = 0; s < 2; ++s) {  // dO halves, handed back by the dQ reduction
      mbar_init(bar(L::kStageFreeDO + s), 1);
      mbar_init(bar(L::kStageFreeQ + s), 1);
      mbar_init(bar(L::kDOFull + s), 1);
    }
    mbar_init(bar(L::kInfoS), 1);
    mbar_init(bar(L::kInfoQ), 1);
    mbar_init(bar(L::kDKVFull), 1);
    mbar_init(bar(L::kMmaDone), 1);
    mbar_init(bar(L::kPReady), kSoftWarps);  // one arrival per softmax warp
    for (int s = 0; s < 2; ++s) mbar_init(bar(L::kKVStaged + s), kTile / 32);
    *abort_flag = 0;
    fence_barrier_init();
    tma_prefetch(&tm_q);
    tma_prefetch(&tm_k);
    tma_prefetch(&tm_v);
    tma_prefetch(&tm_do);
    mbar_expect_tx(bar(L::kKVFull), 2 * L::kTileBytes);
    const TensorPos kv = tensor_pos(P, g, kt * kTile, bt, P.Hkv);
    for (int hf = 0; hf < L::kHalves; ++hf) {
      tma_load_4d(sbase + L::kK + hf * L::kHalfBytes, &tm_k, bar(L::kKVFull), hf * 64, kv.h,
                  kv.row, kv.b);
      tma_load_4d(sbase + L::kV + hf * L::kHalfBytes, &tm_v, bar(L::kKVFull), hf * 64, kv.h,
                  kv.row, kv.b);
    }
  }
  if (warp == kMmaWarp) {
    tmem_alloc(sbase + L::kMisc, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const TileSpan ks = tile_span(P, kt * kTile);
      const PosRange wq = query_window(P, ks);
      int n = 0;    // tiles with Q and dO issued
      int nq = 0;   // tiles with Q issued (n or n + 1)
      bool ok = true;
      // packed sequences of the key tile (fixed) and of the last query tile
      // (the next one's first guess)
      const SegInfo sk = seg_info(P, ks);
      int qhint = sk.first;
      // the key shard travels the ring: step s finds it on rank kappa + s
      for (int s = 0; s < P.cp && ok; ++s) {
        const int rho = (kappa + s) % P.cp;
        // only the runs of the shard that can hold queries seeing the keys
        TileRun runs[2];
        const int nr = shard_runs(P, rho, wq, runs);
        for (int ri = 0; ri < nr && ok; ++ri)
        for (int qt = runs[ri].begin; qt < runs[ri].end && ok; ++qt) {
          const TileSpan qsp = tile_span(P, qt * kTile);
          const SegInfo sq = seg_info(P, qsp, qhint);
          qhint = sq.last;
          const int cls = classify(P, qsp, sq, ks, sk);
          if (cls == kClsEmpty) continue;
          for (int hh = 0; hh < P.G && ok; ++hh) {
            const int h = g * P.G + hh;
            const int slot = n & 1, use = n >> 1;
            // each half is free once the dQ reduction has used it as staging
            if (use >= 1 && !(ok = mbar_wait(bar(L::kStageFreeQ + slot), (use - 1) & 1,
                                             abort_flag, P.status)))
              break;
            sched[slot] = make_int4(qt, h, cls, 0);
            mbar_expect_tx(bar(L::kQFull + slot), L::kTileBytes + L::kStatBytes);
            {
              const long long row_off = ((long long)bt * P.Hq + h) * P.S + (long long)qt * kTile;
              const uint32_t st = sbase + L::kStats + slot * L::kStatBytes;
              bulk_load(st, P.lse2 + row_off, kTile * 4, bar(L::kQFull + slot));
              bulk_load(st + kTile * 4, P.delta + row_off, kTile * 4, bar(L::kQFull + slot));
            }
            const TensorPos qp = tensor_pos(P, h, qt * kTile, bt, P.Hq);
            for (int hf = 0; hf < L::kHalves; ++hf)
              tma_load_4d(sbase + L::kQ + slot * L::kTileBytes + hf * L::kHalfBytes, &tm_q,
                          bar(L::kQFull + slot), hf * 64, qp.h, qp.row, qp.b);
            ++nq;
            if (use >= 1 && !(ok = mbar_wait(bar(L::kStageFreeDO + slot), (use - 1) & 1,
                                             abort_flag, P.status)))
              break;
            mbar_expect_tx(bar(L::kDOFull + slot), L::kTileBytes);
            for (int hf = 0; hf < L::kHalves; ++hf)
              tma_load_4d(sbase + L::kDO + slot * L::kTileBytes + hf * L::kHalfBytes, &tm_do,
                          bar(L::kDOFull + slot), hf * 64, qp.h, qp.row, qp.b);
            ++n;
          }
        }
      }
      if (ok) {
        const int slot = n & 1, use = n >> 1;
        if (use < 1 || mbar_wait(bar(L::kStageFreeQ + slot), (use - 1) & 1, abort_flag,
                                 P.status)) {
          sched[slot] = make_int4(kEnd, 0, 0, 0);
          mbar_arrive(bar(L::kQFull + slot));
        }
        for (int m = (n >= 2 ? n - 2 : 0); m < n; ++m)
          if (!mbar_wait(bar(L::kStageFreeQ + (m & 1)), (m >> 1) & 1, abort_flag, P.status) ||
              !mbar_wait(bar(L::kStageFreeDO + (m & 1)), (m >> 1) & 1, abort_flag, P.status))
            break;
      }
      if (*abort_flag) {
        // aborted: let the copies already issued land before the CTA exits
        mbar_wait_drain(bar(L::kKVFull), 0);
        for (int m = (nq >= 2 ? nq - 2 : 0); m < nq; ++m)
          mbar_wait_drain(bar(L::kQFull + (m & 1)), (m >> 1) & 1);
        for (int m = (n >= 2 ? n - 2 : 0); m < n; ++m)
          mbar_wait_drain(bar(L::kDOFull + (m & 1)), (m >> 1) & 1);
      }
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    // Per query tile n: S^T = K Q^T into [0,128); dP^T = V dO^T into
    // [128,256) once the previous tile's dQ has been taken out of those
    // columns; when P^T is ready: dV += P^T dO (P^T read as bf16 from the
    // S^T columns, 16 queries per MMA), overlapping the softmax's dS; when dS
    // is ready: dQ = dS K into [128,256) as one N=D block, then
    // dK += dS^T Q. The next S^T only has to follow this tile's dV/dK in
    // issue order, never the dQ reduction.
    if (lane == 0) {
      constexpr uint32_t kIdS = idesc_bf16_f32(kTile, kTile, 0, 0);
      constexpr uint32_t kIdDQ = idesc_bf16_f32(kTile, D, 1, 1);
      constexpr uint32_t kIdKV = idesc_bf16_f32(kTile, D, 0, 1);
      const uint32_t t_s = tmem, t_dp = tmem + 128;
      const uint32_t t_dv = tmem + 256, t_dk = tmem + 256 + D;
      // operand descriptors, built once and stepped by constants: K and V
      // as K-major (S^T, dP^T) and MN-major (dQ) operands, the first Q and
      // dO slots both ways, and the dS tile
      const uint64_t dk_k = sdesc_sw128(sbase + L::kK, 16, 1024);
      const uint64_t dv_k = sdesc_sw128(sbase + L::kV, 16, 1024);
      const uint64_t dk_mn = sdesc_sw128(sbase + L::kK, L::kHalfBytes, 1024);
      const uint64_t dq_k = sdesc_sw128(sbase + L::kQ, 16, 1024);
      const uint64_t dq_mn = sdesc_sw128(sbase + L::kQ, L::kHalfBytes, 1024);
      const uint64_t ddo_k = sdesc_sw128(sbase + L::kDO, 16, 1024);
      const uint64_t ddo_mn = sdesc_sw128(sbase + L::kDO, L::kHalfBytes, 1024);
      const uint64_t dds_mn = sdesc_sw128(sbase + L::kDS, L::kHalfBytes, 1024);
      bool ok = mbar_wait(bar(L::kKVFull), 0, abort_flag, P.status);
      int n = 0;
      while (ok) {
        const int slot = n & 1, use = n >> 1;
        if (!(ok = mbar_wait(bar(L::kQFull + slot), use & 1, abort_flag, P.status))) break;
        const int4 e = sched[slot];
        if (e.x == kEnd) break;
        tc_fence_after();
        info[0] = e;
        mbar_arrive(bar(L::kInfoS));
        const uint32_t slot_off = slot * L::kTileBytes;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * L::kHalfBytes + (kk & 3) * 32;
          mma_ss(t_s, sdesc_add(dk_k, off), sdesc_add(dq_k, slot_off + off), kIdS,
                 kk > 0 ? 1u : 0u);
        }
        mma_commit(bar(L::kSFull));
        // the dO tile (its load does not depend on this tile's progress)
        // is checked first, so that its check is not added to the wait for
        // the previous dQ, which must have left [128,256) (and the
        // reduction warp must have read its entry) before dP^T and the
        // next entry
        if (!(ok = mbar_wait(bar(L::kDOFull + slot), use & 1, abort_flag, P.status))) break;
        if (n > 0 && !(ok = mbar_wait(bar(L::kDQEmpty), (n - 1) & 1, abort_flag, P.status)))
          break;
        tc_fence_after();
        info[1] = e;
        mbar_arrive(bar(L::kInfoQ));
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * L::kHalfBytes + (kk & 3) * 32;
          mma_ss(t_dp, sdesc_add(dv_k, off), sdesc_add(ddo_k, slot_off + off), kIdS,
                 kk > 0 ? 1u : 0u);
        }
        mma_commit(bar(L::kDPFull));
        // dV += P^T dO as soon as P^T is in tensor memory: it runs while the
        // softmax warps compute dS (K dim = queries; A from tensor memory:
        // queries 32c .. 32c+31 as bf16 pairs in columns 32c .. 32c+15)
        if (!(ok = mbar_wait(bar(L::kPReady), n & 1, abort_flag, P.status))) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk)
          mma_ts(t_dv, t_s + 32 * (kk >> 1) + 8 * (kk & 1), sdesc_add(ddo_mn, slot_off + kk * 2048),
                 kIdKV, (n > 0 || kk > 0) ? 1u : 0u);
        if (!(ok = mbar_wait(bar(L::kDSFull), n & 1, abort_flag, P.status))) break;
        tc_fence_after();
        // dQ = dS K (M = queries, K dim = keys; both operands MN-major)
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk)
          mma_ss(t_dp, sdesc_add(dds_mn, kk * 2048), sdesc_add(dk_mn, kk * 2048), kIdDQ,
                 kk > 0 ? 1u : 0u);
        mma_commit(bar(L::kDQFull));
        // dK += dS^T Q (dS^T of queries 32c .. 32c+31 in columns 32c+16 ..)
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk)
          mma_ts(t_dk, t_s + 32 * (kk >> 1) + 16 + 8 * (kk & 1),
                 sdesc_add(dq_mn, slot_off + kk * 2048), kIdKV, (n > 0 || kk > 0) ? 1u : 0u);
        mma_commit(bar(L::kQEmpty + slot));
        ++n;
      }
      mma_commit(bar(L::kDKVFull));
      info[0] = make_int4(kEnd, n, 0, 0);
      mbar_arrive(bar(L::kInfoS));
      // the reduction warp must have read the last real entry before the
      // end marker overwrites it
      if (ok && n > 0) mbar_wait(bar(L::kDQEmpty), (n - 1) & 1, abort_flag, P.status);
      info[1] = make_int4(kEnd, n, 0, 0);
      mbar_arrive(bar(L::kInfoQ));
      mma_commit(bar(L::kMmaDone));
      mbar_wait_drain(bar(L::kMmaDone), 0);
    }
  } else if (warp < kSoftWarps) {
    // ------------------------------------------------------------ softmax
    // Four warps share each key row: warp w owns query columns
    // [32 ch, 32 ch + 32), ch = w / 4, of S^T, dP^T and the dS tile, and
    // columns [32 ch, 32 ch + 16) (P^T) and [32 ch + 16, 32 ch + 32) (dS^T)
    // of the bf16 results over its dead S^T columns.
    const int ch = warp >> 2, quarter = warp & 3;
    const int half = ch;                // epilogue group (warps 0-7)
    const int j = quarter * 32 + lane;  // key row = TMEM lane
    const int kp = kt * kTile + j;      // permuted key row
    const ColMask cm = col_mask(P, nat_pos(P, kp));
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t t_s = tmem + lane_off + 32 * ch, t_dp = tmem + lane_off + 128 + 32 * ch;
    // this warp's 16-byte chunks of row j of the 128B-swizzled MN-major dS
    // tile: queries 32ch .. 32ch+31 are 8-query chunks 4ch .. 4ch+3
    uint8_t* ds_row = sm + L::kDS + (ch >> 1) * L::kHalfBytes + j * 128;
    const uint64_t sc2 = f2_pack(P.scale_log2, P.scale_log2);
    int c = 0;
    bool ok = true;
    while (true) {
      ok = mbar_wait(bar(L::kInfoS), c & 1, abort_flag, P.status);
      if (!(ok = __all_sync(0xffffffffu, ok))) break;
      const int4 e = info[0];
      if (e.x == kEnd) break;
      const int qt = e.x;
      const bool masked = e.z == kClsMasked;
      // natural position of this warp's first query and the step between
      const TileSpan qs = tile_span(P, qt * kTile);
      const int i_first = qs.lo + 32 * ch * qs.step;
      // this query tile's LSE (log2 units) and Delta, copied into the tile's
      // Q/dO slot by the producer with the tile itself
      const float* lse2 = reinterpret_cast<const float*>(sm + L::kStats + (c & 1) * L::kStatBytes) + 32 * ch;
      const float* delta = lse2 + kTile;
      ok = mbar_wait(bar(L::kQFull + (c & 1)), (c >> 1) & 1, abort_flag, P.status);
      if (ok) ok = mbar_wait(bar(L::kSFull), c & 1, abort_flag, P.status);
      if (!(ok = __all_sync(0xffffffffu, ok))) break;
      tc_fence_after();
      // P^T = exp2(S^T scale log2e - LSE log2e): kept in fp32 registers for
      // dS, and written over the S^T columns as bf16 pairs for dV
      float pf[32];
      {
        uint32_t sv[32];
        tmem_ld32(t_s, sv);
        tmem_wait_ld();
        uint32_t pk[16];
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          const float4 l4 = reinterpret_cast<const float4*>(lse2)[k >> 1];
          const float2 l = (k & 1) ? make_float2(l4.z, l4.w) : make_float2(l4.x, l4.y);
          const uint64_t x = f2_fma(f2_pack(__uint_as_float(sv[2 * k]), __uint_as_float(sv[2 * k + 1])),
                                    sc2, f2_pack(-l.x, -l.y));
          float x0, x1;
          f2_unpack(x, x0, x1);
          float p0 = ex2(x0), p1 = ex2(x1);
          if (masked) {
            const int i0 = i_first + 2 * k * qs.step;
            const int i1 = i0 + qs.step;
            if (i0 < cm.lo || i0 > cm.hi) p0 = 0.f;
            if (i1 < cm.lo || i1 > cm.hi) p1 = 0.f;
          }
          pf[2 * k] = p0;
          pf[2 * k + 1] = p1;
          pk[k] = pack_bf16(p0, p1);
        }
        tmem_st16(t_s, pk);  // own columns, already read
      }
      // P^T is in tensor memory: dV may start
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(L::kPReady));
      // (the dS tile is free: the previous tile's dQ MMA, its only reader,
      // completed before this tile's S^T)
      ok = mbar_wait(bar(L::kDPFull), c & 1, abort_flag, P.status);
      if (!(ok = __all_sync(0xffffffffu, ok))) break;
      tc_fence_after();
      {
        // dS^T = P^T (dP^T - Delta) on packed pairs, P from the P phase
        uint32_t dv[32], pv[16];
        tmem_ld32(t_dp, dv);
        tmem_wait_ld();
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          const float4 d4 = reinterpret_cast<const float4*>(delta)[k >> 1];
          const float2 dl = (k & 1) ? make_float2(d4.z, d4.w) : make_float2(d4.x, d4.y);
          const uint64_t d2 = f2_add(f2_pack(__uint_as_float(dv[2 * k]), __uint_as_float(dv[2 * k + 1])),
                                     f2_pack(-dl.x, -dl.y));
          const uint64_t ds2 = f2_mul(f2_pack(pf[2 * k], pf[2 * k + 1]), d2);
          float d0, d1;
          f2_unpack(ds2, d0, d1);
          pv[k] = pack_bf16(d0, d1);
        }
        tmem_st16(t_s + 16, pv);  // own dead S^T columns
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int chunk = (4 * ch + q) & 7;
          uint4 w = make_uint4(pv[4 * q], pv[4 * q + 1], pv[4 * q + 2], pv[4 * q + 3]);
          *reinterpret_cast<uint4*>(ds_row + ((chunk ^ (j & 7)) << 4)) = w;
        }
      }
      tmem_wait_st();
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(L::kDSFull));
      if (ch < kBoxes) {
        // this tile's dQ, rows [32 quarter, +32) x columns [32 ch, +32): out
        // of tensor memory as soon as the dQ MMA is done (the columns go back
        // for the next dP^T), then staged, scaled, for the reduction warp.
        // The next S^T is being computed meanwhile. Once the dQ MMA is done,
        // nothing reads the dO tile of the tile's slot any more (the dP^T and
        // dV MMAs that read it were issued before), and once the dK MMA is
        // done nothing reads its Q tile; neither is written again before the
        // reduction hands it back.
        ok = mbar_wait(bar(L::kDQFull), c & 1, abort_flag, P.status);
        if (!(ok = __all_sync(0xffffffffu, ok))) break;
        tc_fence_after();
        uint32_t v[32];
        tmem_ld32(t_dp, v);
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(L::kDQEmpty));
        if (ch < kBoxesInQ) {
          ok = mbar_wait(bar(L::kQEmpty + (c & 1)), (c >> 1) & 1, abort_flag, P.status);
          if (!(ok = __all_sync(0xffffffffu, ok))) break;
        }
        const int i = quarter * 32 + lane;  // query row = TMEM lane
        uint8_t* rowp = stage_box(c & 1, ch) + i * 128;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const float4 x = make_float4(__uint_as_float(v[4 * k]) * P.scale,
                                       __uint_as_float(v[4 * k + 1]) * P.scale,
                                       __uint_as_float(v[4 * k + 2]) * P.scale,
                                       __uint_as_float(v[4 * k + 3]) * P.scale);
          *reinterpret_cast<float4*>(rowp + ((k ^ (i & 7)) << 4)) = x;
        }
        // read next by the TMA unit (async proxy)
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(L::kDQStaged));
      }
      ++c;
    }
    // epilogue: warps 0-3 write dV, warps 4-7 scale * dK for their key
    // row, staged in the 128-byte swizzle in the V / K tile (free: every MMA
    // has completed) and stored with TMA by one thread of the group
    if (ok && half < 2) ok = mbar_wait(bar(L::kDKVFull), 0, abort_flag, P.status);
    ok = __all_sync(0xffffffffu, ok);
    tc_fence_after();
    if (ok && half < 2) {
      uint8_t* stage = sm + (half ? L::kK : L::kV);
      const uint32_t src = tmem + lane_off + 256 + half * D;
      const float mul = half ? P.scale : 1.f;
#pragma unroll
      for (int cq = 0; cq < D / 32; ++cq) {
        uint32_t o[32];
        tmem_ld32(src + 32 * cq, o);
        tmem_wait_ld();
        uint32_t wp[16];
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          const float a = c > 0 ? __uint_as_float(o[2 * k]) * mul : 0.f;
          const float b = c > 0 ? __uint_as_float(o[2 * k + 1]) * mul : 0.f;
          wp[k] = pack_bf16(a, b);
        }
        // columns 32 cq .. 32 cq + 31 = 16-byte chunks 4 cq .. 4 cq + 3
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int c8 = 4 * cq + q, hf = c8 >> 3, chunk = c8 & 7;
          *reinterpret_cast<uint4*>(stage + hf * L::kHalfBytes + j * 128 +
                                    ((chunk ^ (j & 7)) << 4)) =
              make_uint4(wp[4 * q], wp[4 * q + 1], wp[4 * q + 2], wp[4 * q + 3]);
        }
      }
      fence_proxy_async_smem();  // read next by the TMA unit
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(L::kKVStaged + half));
      if (quarter == 0 && lane == 0 &&
          mbar_wait(bar(L::kKVStaged + half), 0, abort_flag, P.status)) {
        const TensorPos kv = tensor_pos(P, g, kt * kTile, bt, P.Hkv);
        for (int hf = 0; hf < L::kHalves; ++hf)
          tma_store_4d(half ? &tm_dk : &tm_dv, smem_u32(stage + hf * L::kHalfBytes), hf * 64,
                       kv.h, kv.row, kv.b);
        bulk_commit_group();
        // the tile has been read out of shared memory before the CTA exits
        // (the global writes complete on their own)
        bulk_wait_group_read0();
      }
    }
  } else if (warp == kReduceWarp) {
    // ------------------------------------------------------------ dQ reduction
    // Per query tile: the staged dQ boxes are added into the global fp32
    // accumulator by the TMA unit, the Q tile's boxes first as their own bulk
    // group. Each space goes back to the producer as soon as the TMA has read
    // it; the additions complete asynchronously.
    int c = 0;
    while (true) {
      bool ok = mbar_wait(bar(L::kInfoQ), c & 1, abort_flag, P.status);
      if (!__all_sync(0xffffffffu, ok)) break;
      const int4 e = info[1];
      if (e.x == kEnd) break;
      const int qt = e.x, h = e.y;
      // the entry has been read: the MMA warp may post the next one
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(L::kDQEmpty));
      ok = mbar_wait(bar(L::kDQStaged), c & 1, abort_flag, P.status);
      if (!__all_sync(0xffffffffu, ok)) break;
      const int slot = c & 1;
      if (lane == 0) {
#pragma unroll
        for (int cg = 0; cg < kBoxes; ++cg) {
          tma_reduce_add_4d(&tm_dq, smem_u32(stage_box(slot, cg)), 32 * cg, h, qt * kTile, bt);
          if (cg + 1 == kBoxesInQ) bulk_commit_group();
        }
        bulk_commit_group();
        bulk_wait_group_read1();
        mbar_arrive(bar(L::kStageFreeQ + slot));
        bulk_wait_group_read0();
        mbar_arrive(bar(L::kStageFreeDO + slot));
      }
      __syncwarp();
      ++c;
    }
    // every reduction has landed before the CTA exits
    if (lane == 0) bulk_wait_group0();
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp) tmem_dealloc(tmem, 512);
}

// dq (bf16) <- dq_acc (fp32), 8 elements per thread-iteration. Token rows of
// row8 8-element groups; dst rows are tok8 groups apart (== row8 when dense,
// three times it in a packed q/k/v gradient). With P.nat the dst is the
// caller's natural-order dq: head group u of token row p goes to groups
// u*row8.. of natural row nat(p), rows tok8 = ud*row8 apart.
__global__ void __launch_bounds__(256) dq_convert_kernel(const float4* __restrict__ src,
                                                         uint4* __restrict__ dst,
                                                         long long n8, int row8,
                                                         long long tok8, const AttnParams P) {
  for (long long i = blockIdx.x * 256ll + threadIdx.x; i < n8; i += (long long)gridDim.x * 256) {
    const float4 a = __ldg(src + 2 * i), b = __ldg(src + 2 * i + 1);
    const long long row = i / row8;
    long long drow = row, doff = 0;
    if (P.nat) {
      const int bt = (int)(row / P.S), p = (int)(row - (long long)bt * P.S);
      const int u = bt / P.B;
      drow = (long long)(bt - u * P.B) * P.S + nat_pos(p, P.layout, P.cp, P.shard, P.chunk);
      doff = (long long)u * row8;
    }
    dst[drow * tok8 + doff + (i - row * row8)] =
        make_uint4(pack_bf16(a.x, a.y), pack_bf16(a.z, a.w), pack_bf16(b.x, b.y),
                   pack_bf16(b.z, b.w));
  }
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

// [Bt][S][H][D] -> 4-D map (D, H, S, Bt), box (box0, 1, 128, 1), 128B swizzle;
// bf16 operand tiles (box0 = 64) or the fp32 dQ accumulator (box0 = 32).
// tok: elements between tokens (0: dense H*D; 3*H*D in a packed q/k/v tensor)
bool make_map(CUtensorMap* m, const void* base, int Bt, int S, int H, int D,
              bool fp32 = false, long long tok = 0) {
  if (tok == 0) tok = (long long)H * D;
  auto fn = encode_fn();
  if (!fn) {
    fail_cuda_msg("cuTensorMapEncodeTiled", "driver entry point not found");
    return false;
  }
  cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)S, (cuuint64_t)Bt};
  const cuuint64_t es_b = fp32 ? 4 : 2;
  cuuint64_t strides[3] = {(cuuint64_t)D * es_b, (cuuint64_t)tok * es_b,
                           (cuuint64_t)S * tok * es_b};
  cuuint32_t box[4] = {fp32 ? 32u : 64u, 1, (cuuint32_t)kTile, 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  CUresult r = fn(m, fp32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4,
                  const_cast<void*>(base), dims,
                  strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
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
  CUtensorMap mq, mk, mv, mdo, mdq, mdk, mdv;
  const long long tok = P.qkv_tok;
  // natural-order tensors in place: all heads of every token, B batch rows
  // (the dQ accumulator stays in the kernels' own head groups)
  const int Bm = P.nat ? P.B : P.Bt, hm = P.nat ? P.ud : 1;
  if (!make_map(&mq, P.q, Bm, P.S, P.Hq * hm, D, false, tok) ||
      !make_map(&mk, P.k, Bm, P.S, P.Hkv * hm, D, false, tok) ||
      !make_map(&mv, P.v, Bm, P.S, P.Hkv * hm, D, false, tok) ||
      !make_map(&mdo, P.dout, Bm, P.S, P.Hq * hm, D) ||
      !make_map(&mdq, P.dq_acc, P.Bt, P.S, P.Hq, D, true) ||
      !make_map(&mdk, P.dk, Bm, P.S, P.Hkv * hm, D, false, tok) ||
      !make_map(&mdv, P.dv, Bm, P.S, P.Hkv * hm, D, false, tok))
    return USP_ERR_CUDA;
  static int* status = nullptr;
  if (status == nullptr) {
    cudaError_t e = cudaGetSymbolAddress(reinterpret_cast<void**>(&status), g_bwd_tc_status);
    if (e != cudaSuccess) return fail_cuda("cudaGetSymbolAddress(status)", e);
  }
  AttnParams Pk = P;
  Pk.status = status;
  // L2 batches of units (KV head, batch), heaviest CTAs first inside each.
  // Contiguous and zigzag: about 6.5 waves of CTAs per batch. Their CTAs walk
  // the query shards in ring order, so a batch touches a moving window of
  // query tiles, and wide batches spread the CTAs that reach the same
  // (popular, late) query tiles over more heads: at S=8K with 64 key tiles
  // per head, 16 heads per batch ran the backward 7 % faster than 4, and
  // the S=32K ring 5 % faster with 4 KV groups than with 1. Stripe: about
  // 1.5 waves, since every key tile visits nearly every query tile of its
  // head and wider batches overflow L2 (S=32K: 19.4 ms with 1 group, 25.2
  // with 8). Packed sequences: one batch, since a key tile only meets the
  // query tiles of its own sequence.
  {
    const int ntiles = P.S / kTile;
    const int units = P.Hkv * P.Bt;
    const int waves2 = P.layout == kStripe ? 3 : 13;  // twice the waves per batch
    int per = (waves2 * sm_count() / 2 + ntiles - 1) / ntiles;
    if (P.cu != nullptr) per = units;
    Pk.unit_batch = per < units ? per : units;
  }
  const int smem = BSmem<D>::kAlloc;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(attn_bwd_tc_kernel<D>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return fail_cuda("cudaFuncSetAttribute(smem)", e);
    attr_set = true;
  }
  const long long blocks = (long long)(P.S / kTile) * P.Hkv * P.Bt;
  {
    ProfScope ps(st, "attn_bwd_tc");
    attn_bwd_tc_kernel<D><<<(unsigned)blocks, kThreads, smem, st>>>(Pk, mq, mk, mv, mdo, mdq, mdk, mdv);
  }
  note_launch();
  usp_status_t r = check_launch();
  if (r != USP_OK) return r;
  const long long n8 = (long long)P.Bt * P.S * P.Hq * D / 8;
  {
    ProfScope ps(st, "attn_bwd_dq_convert");
    dq_convert_kernel<<<(unsigned)(n8 < 152LL * 32 * 4 ? (n8 + 255) / 256 : 152 * 16), 256, 0,
                        st>>>(reinterpret_cast<const float4*>(P.dq_acc),
                              reinterpret_cast<uint4*>(P.dq), n8, P.Hq * D / 8,
                              P.nat ? (long long)P.ud * P.Hq * D / 8 : qkv_stride(P, P.Hq) / 8, P);
  }
  note_launch();
  return check_launch();
}

}  // namespace

int read_clear_bwd_tc_status() {
  int v = 0, z = 0;
  if (cudaMemcpyFromSymbol(&v, g_bwd_tc_status, sizeof(int)) != cudaSuccess) return -1;
  if (v != 0) cudaMemcpyToSymbol(g_bwd_tc_status, &z, sizeof(int));
  return v;
}

bool bwd_tc_supported(const AttnParams& P) {
  if (P.D != 128 && P.D != 64) return false;
  if (P.shard % kTile != 0) return false;
  if (P.layout == kZigzag && P.chunk % kTile != 0) return false;
  return true;
}

usp_status_t launch_bwd_tc(const AttnParams& P, cudaStream_t st) {
  return P.D == 128 ? launch_d<128>(P, st) : launch_d<64>(P, st);
}

}  // namespace usp
