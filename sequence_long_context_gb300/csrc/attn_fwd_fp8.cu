// Ring attention forward with e4m3 q, k, v on the tcgen05 tensor cores
// (kind::f8f6f4, fp32 accumulation in tensor memory), and the two copy
// kernels it needs: bf16 -> e4m3 quantization and the V transpose.
//
// The USP README ("3. Test") runs a forward-only fp8 attention backend under
// the sequence-parallel wrappers; here the attention itself is the same ring
// schedule as the bf16 forward ("Long Context Attention" notes, "Ring
// Attention": KV shards visit every rank; "Tree Attention": partials merge
// with the log-sum-exp rule), computed on 8-bit operands. The real value of
// a code c of a tensor with descale d is e4m3(c) * d.
//
// One CTA owns one 128-row query tile of one (batch, head) of one ring rank
// and two CTAs share an SM; roles (192 threads):
//   warps 0-3  softmax, one query row per thread
//   warp  4    producer: classifies key tiles, streams K and V^T tiles
//   warp  5    MMA issuer and owner of the CTA's tensor memory
// What the 8-bit operands change:
//  * Q and K tiles are 128 tokens x 128 codes, one 128-byte swizzle row per
//    token. V is read transposed ([d][key], keys contiguous, written by the
//    transpose pre-pass), so both products take K-major operands:
//    S = Q K^T and O += P (V^T)^T, 32 K elements per instruction.
//  * P goes to shared memory as e4m3 codes of 16 p, a 128 x 128 K-major
//    tile. The running max moves whenever the row max grows by more than 2^4,
//    so p <= 2^4 and 16 p <= 256, below the largest code (448); the row sum
//    l accumulates 16 p in fp32 and the scale cancels in O = sum(16 p v) / l.
//  * Since P does not go back into tensor memory, S is free as soon as the
//    softmax has loaded it: the next key tile's Q K^T is issued then, and
//    runs while this tile's exponentials are computed.
//  * q_descale * k_descale is folded into the softmax scale; v_descale
//    multiplies O in the epilogue.
// Tensor memory (256 columns per CTA): S at [0, 128), O at [128, 256).
#include <cudaTypedefs.h>

#include <cstdio>

#include "internal.h"
#include "tc_ptx.cuh"
#include "tile_sched.cuh"

namespace usp {
namespace {

using namespace tc;

__device__ int g_fwd_fp8_status = 0;

constexpr int kBM = 128;  // query rows per tile
constexpr int kBN = 128;  // keys per tile
constexpr int kD = 128;   // head dim (one 128-byte swizzle row of codes)
constexpr int kThreads = 192;
constexpr int kProducerWarp = 4;
constexpr int kMmaWarp = 5;
constexpr int kEmpty = kClsEmpty, kMasked = kClsMasked;
constexpr int kEnd = -1;
constexpr float kRescaleThreshold = 4.0f;  // log2 units; bounds p by 2^4
constexpr float kPLog2 = 4.0f;             // P codes hold 2^4 p
constexpr float kLn2 = 0.6931471805599453f;

// Largest of three values in one instruction (three-input max.f32).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Four fp32 -> four e4m3 codes in one 32-bit word (a in the low byte):
// round to nearest even, finite values beyond the largest code saturate.
__device__ __forceinline__ uint32_t pack_e4m3x4(float a, float b, float c, float d) {
  uint32_t r;
  asm("{\n\t.reg .b16 lo, hi;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 lo, %2, %1;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 hi, %4, %3;\n\t"
      "mov.b32 %0, {lo, hi};\n\t}"
      : "=r"(r)
      : "f"(a), "f"(b), "f"(c), "f"(d));
  return r;
}

// Non-blocking test of one mbarrier phase (acquire semantics, like a wait).
__device__ __forceinline__ uint32_t mbar_test1(uint32_t a, uint32_t pa) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(r)
      : "r"(a), "r"(pa)
      : "memory");
  return r;
}
// Non-blocking tests of two mbarrier phases issued back to back: bit 0 set
// if the phase of a with parity pa has completed, bit 1 likewise for b.
__device__ __forceinline__ uint32_t mbar_test2(uint32_t a, uint32_t pa, uint32_t b,
                                               uint32_t pb) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 q, [%3], %4;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t"
      "@q or.b32 %0, %0, 2;\n\t}"
      : "=r"(r)
      : "r"(a), "r"(pa), "r"(b), "r"(pb)
      : "memory");
  return r;
}

struct Smem8 {
  static constexpr int kTileBytes = 128 * 128;  // 128 rows x 128 one-byte codes
  static constexpr int kQ = 0;
  static constexpr int kK = kQ + kTileBytes;       // 2 key slots
  static constexpr int kV = kK + 2 * kTileBytes;   // 2 V^T slots
  static constexpr int kP = kV + 2 * kTileBytes;   // the P tile
  static constexpr int kBar = kP + kTileBytes;
  // kSFree: the softmax has loaded S (the next Q K^T may overwrite it);
  // kPFree: the P V that read the P tile (and updated O) is done
  static constexpr int kQFull = 0, kKFull = 1, kKEmpty = 3, kVFull = 5, kVEmpty = 7,
                       kSFull = 9, kSFree = 10, kPFull = 11, kPFree = 12, kOFull = 13,
                       kInfoFull = 14, kMmaDone = 15, kOStaged = 16, kNumBars = 17;
  static constexpr int kSched = (kBar + 8 * kNumBars + 15) / 16 * 16;  // int4 x 2
  static constexpr int kInfo = kSched + 32;                            // int2
  static constexpr int kMisc = kInfo + 16;                             // tmem base, abort
  static constexpr int kBytes = kMisc + 16;
  static constexpr int kAlloc = kBytes + 1024;  // alignment slack
  static_assert(kK % 1024 == 0 && kV % 1024 == 0 && kP % 1024 == 0,
                "swizzled tiles need 1024-byte alignment");
  static_assert(2 * kAlloc <= 232448, "two CTAs must fit one SM's shared memory");
};

__device__ __forceinline__ int fwd_head(const AttnParams& P, int unit) {
  return unit / (P.G * P.Bt) * P.G + unit % P.G;
}
__device__ __forceinline__ int fwd_batch(const AttnParams& P, int unit) {
  return (unit / P.G) % P.Bt;
}
// Query tiles (128 rows), heaviest first for causal dense problems.
__device__ __forceinline__ int qtile_for_rank(const AttnParams& P, int r, int ntiles) {
  if (!P.causal || P.cu != nullptr) return r;
  if (P.layout == kStripe) {
    const int tpr = P.shard / kBM;
    return (r % P.cp) * tpr + (tpr - 1 - r / P.cp);
  }
  return permuted_of(P, (ntiles - 1 - r) * kBM) / kBM;
}

__global__ void __launch_bounds__(kThreads, 2)
attn_fwd_fp8_kernel(const AttnParams P, float o_mul,
                    const __grid_constant__ CUtensorMap tm_q,
                    const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_vt,
                    const __grid_constant__ CUtensorMap tm_o) {
  using L = Smem8;
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
  const int qbase = qt * kBM;        // permuted row of the tile
  const int rho = qbase / P.shard;   // its ring rank

  // the producer thread sets up the barriers and starts the Q load
  if (warp == kProducerWarp && lane == 0) {
    mbar_init(bar(L::kQFull), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(L::kKFull + s), 1);
      mbar_init(bar(L::kKEmpty + s), 1);
      mbar_init(bar(L::kVFull + s), 1);
      mbar_init(bar(L::kVEmpty + s), 1);
    }
    mbar_init(bar(L::kSFull), 1);
    mbar_init(bar(L::kSFree), kBM / 32);   // one arrival per softmax warp
    mbar_init(bar(L::kPFull), kBM / 32);   // one arrival per softmax warp
    mbar_init(bar(L::kPFree), 1);
    mbar_init(bar(L::kOFull), 1);
    mbar_init(bar(L::kInfoFull), 1);
    mbar_init(bar(L::kMmaDone), 1);
    mbar_init(bar(L::kOStaged), kBM / 32);  // one arrival per softmax warp
    *abort_flag = 0;
    fence_barrier_init();
    tma_prefetch(&tm_q);
    tma_prefetch(&tm_k);
    tma_prefetch(&tm_vt);
    mbar_expect_tx(bar(L::kQFull), L::kTileBytes);
    tma_load_4d(sbase + L::kQ, &tm_q, bar(L::kQFull), 0, h, qbase, bt);
  }
  if (warp == kMmaWarp) {
    tmem_alloc(sbase + L::kMisc, 256);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    // Key tiles in ring order, classified for the query tile and loaded
    // unless empty: K and V^T through two-slot rings, freed by the tile's
    // Q K^T and P V.
    if (lane == 0) {
      const TileSpan q0 = tile_span(P, qbase);
      const KeyWindows w0 = key_windows(P, q0);
      const SegInfo sq0 = seg_info(P, q0);
      int khint = sq0.first;
      int n = 0, nk = 0;
      bool ok = true;
      auto visit = [&](int kt) {
        const TileSpan ks = tile_span(P, kt * kBN);
        if (disjoint(ks, w0.band) && disjoint(ks, w0.sink)) return;
        const SegInfo sk = seg_info(P, ks, khint);
        khint = sk.last;
        const int c0 = classify(P, q0, sq0, ks, sk);
        if (c0 == kEmpty) return;
        const int slot = n & 1, use = n >> 1;
        if (use >= 1 && !(ok = mbar_wait(bar(L::kKEmpty + slot), (use - 1) & 1,
                                         abort_flag, P.status)))
          return;
        sched[slot] = make_int4(kt, c0, 0, 0);
        mbar_expect_tx(bar(L::kKFull + slot), L::kTileBytes);
        tma_load_4d(sbase + L::kK + slot * L::kTileBytes, &tm_k, bar(L::kKFull + slot), 0, g,
                    kt * kBN, bt);
        ++nk;
        if (use >= 1 && !(ok = mbar_wait(bar(L::kVEmpty + slot), (use - 1) & 1,
                                         abort_flag, P.status)))
          return;
        mbar_expect_tx(bar(L::kVFull + slot), L::kTileBytes);
        // V^T map (key, d, head, batch): 128 keys x 128 d rows
        tma_load_4d(sbase + L::kV + slot * L::kTileBytes, &tm_vt, bar(L::kVFull + slot),
                    kt * kBN, 0, g, bt);
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
        const int slot = n & 1, use = n >> 1;
        if (use < 1 || mbar_wait(bar(L::kKEmpty + slot), (use - 1) & 1, abort_flag,
                                 P.status)) {
          sched[slot] = make_int4(kEnd, 0, 0, 0);
          mbar_arrive(bar(L::kKFull + slot));
        }
        // the last V^T tiles have been consumed before the CTA may exit
        for (int m = (n >= 2 ? n - 2 : 0); m < n; ++m)
          if (!mbar_wait(bar(L::kVEmpty + (m & 1)), (m >> 1) & 1, abort_flag, P.status)) break;
      }
      if (*abort_flag) {
        // aborted: let the copies already issued land before the CTA exits
        mbar_wait_drain(bar(L::kQFull), 0);
        for (int m = (nk >= 2 ? nk - 2 : 0); m < nk; ++m)
          mbar_wait_drain(bar(L::kKFull + (m & 1)), (m >> 1) & 1);
        for (int m = (n >= 2 ? n - 2 : 0); m < n; ++m)
          mbar_wait_drain(bar(L::kVFull + (m & 1)), (m >> 1) & 1);
      }
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    // Per key tile c: S = Q K^T; once the softmax has loaded S(c) into
    // registers, the next key tile's Q K^T (its K slot loaded); then, once P(c)
    // is in shared memory, O (+)= P V(c), whose commit frees the P tile and
    // the V^T slot. The tensor core thus runs the next Q K^T while the
    // softmax computes this tile's P.
    if (lane == 0) {
      constexpr uint32_t kIdQK = idesc_e4m3_f32(kBM, kBN);
      constexpr uint32_t kIdPV = idesc_e4m3_f32(kBM, kD);
      const uint32_t s_tm = tmem, o_tm = tmem + 128;
      // operand descriptors, built once and stepped by constants
      const uint64_t dq0 = sdesc_sw128(sbase + L::kQ, 16, 1024);
      const uint64_t dk0 = sdesc_sw128(sbase + L::kK, 16, 1024);
      const uint64_t dp0 = sdesc_sw128(sbase + L::kP, 16, 1024);
      const uint64_t dv0 = sdesc_sw128(sbase + L::kV, 16, 1024);
      auto qk = [&](int slot) {
        const uint64_t kd = sdesc_add(dk0, slot * L::kTileBytes);
#pragma unroll
        for (int kk = 0; kk < kD / 32; ++kk)
          mma_ss_f8(s_tm, sdesc_add(dq0, 32 * kk), sdesc_add(kd, 32 * kk), kIdQK,
                    kk > 0 ? 1u : 0u);
        mma_commit(bar(L::kSFull));
        mma_commit(bar(L::kKEmpty + slot));
      };
      bool ok = mbar_wait(bar(L::kQFull), 0, abort_flag, P.status);
      bool more = false;
      if (ok && (ok = mbar_wait(bar(L::kKFull + 0), 0, abort_flag, P.status))) {
        const int4 e = sched[0];
        more = e.x != kEnd;
        if (more) {
          tc_fence_after();
          *info = make_int2(e.x, e.y);
          mbar_arrive(bar(L::kInfoFull));
          qk(0);
        }
      }
      int c = 0;  // key tiles whose P V has been issued
      while (ok && more) {
        const int ns = (c + 1) & 1, nuse = (c + 1) >> 1;
        if (!(ok = mbar_wait(bar(L::kKFull + ns), nuse & 1, abort_flag, P.status))) break;
        const int4 e = sched[ns];
        more = e.x != kEnd;
        if (more) {
          // S(c) is in the softmax's registers (and the softmax has read
          // the entry of tile c): the next tile's S may take its columns
          if (!(ok = mbar_wait(bar(L::kSFree), c & 1, abort_flag, P.status))) break;
          tc_fence_after();
          *info = make_int2(e.x, e.y);
          mbar_arrive(bar(L::kInfoFull));
          qk(ns);
        }
        // the V^T slot (usually loaded long before) first, so that its check
        // is not added to the wait for P
        const int slot = c & 1, use = c >> 1;
        if (!(ok = mbar_wait(bar(L::kVFull + slot), use & 1, abort_flag, P.status))) break;
        if (!(ok = mbar_wait(bar(L::kPFull), c & 1, abort_flag, P.status))) break;
        tc_fence_after();
        const uint64_t vd = sdesc_add(dv0, slot * L::kTileBytes);
#pragma unroll
        for (int kk = 0; kk < kBN / 32; ++kk)
          mma_ss_f8(o_tm, sdesc_add(dp0, 32 * kk), sdesc_add(vd, 32 * kk), kIdPV,
                    (c > 0 || kk > 0) ? 1u : 0u);
        mma_commit(bar(L::kPFree));
        mma_commit(bar(L::kVEmpty + slot));
        ++c;
      }
      mma_commit(bar(L::kOFull));
      // every entry has been read (the last tile's P was waited for)
      *info = make_int2(kEnd, 0);
      mbar_arrive(bar(L::kInfoFull));
      // nothing of ours may still run on the tensor core when TMEM is freed
      mma_commit(bar(L::kMmaDone));
      mbar_wait_drain(bar(L::kMmaDone), 0);
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;       // row within the tile = TMEM lane
    const int prow = qbase + r;              // permuted query row
    const RowMask rm = row_mask(P, nat_pos(P, prow));
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t s_tm = tmem + lane_off, o_tm = tmem + lane_off + 128;
    uint8_t* p_row = sm + L::kP + r * 128;
    float m_run = -INFINITY, l_run = 0.f;  // l_run sums 2^4 p
    int c = 0;
    bool ok = true;
    uint32_t ahead = 0;  // bit 0 / 1: tile c's entry / S found there ahead
    while (true) {
      ok = (ahead & 1u) || mbar_wait(bar(L::kInfoFull), c & 1, abort_flag, P.status);
      if (!(ok = __all_sync(0xffffffffu, ok))) break;
      const int2 inf = *info;
      if (inf.x == kEnd) break;
      uint32_t vis[4] = {~0u, ~0u, ~0u, ~0u};
      if (inf.y == kMasked) {
        const TileSpan ks = tile_span(P, inf.x * kBN);
        const ColRange c0 = tile_cols(ks, rm.lo, rm.hi);
        const ColRange c1 = tile_cols(ks, rm.qs, min(rm.sink_end - 1, rm.causal_hi));
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) vis[ch] = col_bits(c0, 32 * ch) | col_bits(c1, 32 * ch);
      }
      ok = (ahead & 2u) || mbar_wait(bar(L::kSFull), c & 1, abort_flag, P.status);
      if (!(ok = __all_sync(0xffffffffu, ok))) break;
      tc_fence_after();
      uint32_t sr[4][32];
#pragma unroll
      for (int ch = 0; ch < 4; ++ch) tmem_ld32(s_tm + 32 * ch, sr[ch]);
      tmem_wait_ld();
      // S is in registers: the next key tile's Q K^T may overwrite it
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(L::kSFree));
      if (inf.y == kMasked) {
#pragma unroll
        for (int ch = 0; ch < 4; ++ch)
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (!((vis[ch] >> j) & 1u)) sr[ch][j] = __float_as_uint(-INFINITY);
      }
      // row max as 8 independent chains of three-input maxima (a single
      // chain is latency-bound)
      float m8[8];
#pragma unroll
      for (int t = 0; t < 8; ++t) m8[t] = __uint_as_float(sr[t >> 5][t & 31]);
#pragma unroll
      for (int j = 8; j < 128; j += 2)
        m8[(j >> 1) & 7] = fmax3(m8[(j >> 1) & 7], __uint_as_float(sr[j >> 5][j & 31]),
                                 __uint_as_float(sr[(j + 1) >> 5][(j + 1) & 31]));
      float mx = fmax3(fmax3(m8[0], m8[1], m8[2]), fmax3(m8[3], m8[4], m8[5]),
                       fmaxf(m8[6], m8[7]));
      mx *= P.scale_log2;
      const bool need = mx > m_run + kRescaleThreshold;
      float alpha = 1.f;
      if (need) {
        alpha = (m_run == -INFINITY) ? 0.f : ex2(m_run - mx);
        m_run = mx;
      }
      l_run *= alpha;
      const float msub = (m_run == -INFINITY) ? 0.f : m_run;
      // the previous tile's P V is usually done by the end of this tile's
      // exponentials: its phase is tested now, the test's latency
      // overlapping them, and waited for afterwards only if it was not
      const uint32_t p_free = (c == 0) ? 1u : mbar_test1(bar(L::kPFree), (c - 1) & 1);
      // 2^4 p = exp2(s * scale_log2 - m + 4) <= 2^8, on packed fp32 pairs,
      // as e4m3 codes held in registers (w[4 ck + q]: keys 16 ck + 4 q ..
      // 16 ck + 4 q + 3) until the previous tile's P V has read the P tile
      const uint64_t sc2 = f2_pack(P.scale_log2, P.scale_log2);
      const uint64_t nm2 = f2_pack(kPLog2 - msub, kPLog2 - msub);
      uint64_t ls2[4] = {0, 0, 0, 0};
      uint32_t w[32];
#pragma unroll
      for (int ck = 0; ck < 8; ++ck) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          float pp[4];
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            const int j0 = 16 * ck + 4 * q + 2 * t;
            const uint64_t x = f2_fma(f2_pack(__uint_as_float(sr[j0 >> 5][j0 & 31]),
                                              __uint_as_float(sr[(j0 + 1) >> 5][(j0 + 1) & 31])),
                                      sc2, nm2);
            float x0, x1;
            f2_unpack(x, x0, x1);
            pp[2 * t] = ex2(x0);
            pp[2 * t + 1] = ex2(x1);
            ls2[(2 * q + t) & 3] = f2_add(ls2[(2 * q + t) & 3], f2_pack(pp[2 * t], pp[2 * t + 1]));
          }
          w[4 * ck + q] = pack_e4m3x4(pp[0], pp[1], pp[2], pp[3]);
        }
      }
      {
        float a0, a1, b0, b1, c0, c1, d0, d1;
        f2_unpack(ls2[0], a0, a1);
        f2_unpack(ls2[1], b0, b1);
        f2_unpack(ls2[2], c0, c1);
        f2_unpack(ls2[3], d0, d1);
        l_run += ((a0 + a1) + (b0 + b1)) + ((c0 + c1) + (d0 + d1));
      }
      // the previous tile's P V has read the P tile and added into O (so the
      // P tile and O may be written)
      // the next tile's entry and S (its Q K^T was issued when this S was
      // loaded) are tested now, the tests' latency overlapping the P stores;
      // the next iteration waits only for what was not there
      ahead = mbar_test2(bar(L::kInfoFull), (c + 1) & 1, bar(L::kSFull), (c + 1) & 1);
      if (!__all_sync(0xffffffffu, p_free != 0u)) {
        ok = mbar_wait(bar(L::kPFree), (c - 1) & 1, abort_flag, P.status);
        if (!(ok = __all_sync(0xffffffffu, ok))) break;
      }
      tc_fence_after();
      // this row of the P tile, 16 keys per 16-byte chunk, in the 128-byte
      // swizzle (chunk k of row r at k ^ (r & 7))
#pragma unroll
      for (int ck = 0; ck < 8; ++ck)
        *reinterpret_cast<uint4*>(p_row + ((ck ^ (r & 7)) << 4)) =
            make_uint4(w[4 * ck], w[4 * ck + 1], w[4 * ck + 2], w[4 * ck + 3]);
      // rescale O (the previous tiles' P V, complete) to the new max before
      // this tile's P V adds onto it
      if (__any_sync(0xffffffffu, need && c > 0)) {
#pragma unroll
        for (int ch = 0; ch < kD / 32; ++ch) {
          uint32_t o[32];
          tmem_ld32(o_tm + 32 * ch, o);
          tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 32; ++j)
            o[j] = __float_as_uint(__uint_as_float(o[j]) * alpha);
          tmem_st32(o_tm + 32 * ch, o);
        }
        tmem_wait_st();
      }
      fence_proxy_async_smem();  // the P tile is read next by the tensor core
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(L::kPFull));
      ++c;
    }
    // epilogue: v_descale * O / l -> bf16 rows, LSE = (m + log2 l - 4) ln 2.
    // The 64-column halves of the bf16 tile are staged in the 128-byte
    // swizzle in the Q and P tiles (free: every MMA is done when O is) and
    // one thread stores them with TMA.
    if (ok) ok = mbar_wait(bar(L::kOFull), 0, abort_flag, P.status);
    ok = __all_sync(0xffffffffu, ok);
    tc_fence_after();
    // the CTA's head and batch, recomputed (not kept live through the loop)
    const int unit = batched_order(blockIdx.x, P.Hq * P.Bt, P.S / kBM, P.unit_batch).unit;
    const int h = fwd_head(P, unit), bt = fwd_batch(P, unit);
    if (ok) {
      const float mul = (l_run > 0.f) ? o_mul / l_run : 0.f;
      uint8_t* stage[2] = {sm + L::kQ, sm + L::kP};
#pragma unroll
      for (int ch = 0; ch < kD / 32; ++ch) {
        uint32_t o[32];
        tmem_ld32(o_tm + 32 * ch, o);
        tmem_wait_ld();
        uint32_t wp[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const float a = (c > 0) ? __uint_as_float(o[2 * j]) * mul : 0.f;
          const float b = (c > 0) ? __uint_as_float(o[2 * j + 1]) * mul : 0.f;
          wp[j] = pack_bf16(a, b);
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int c8 = 4 * ch + q, hf = c8 >> 3, chunk = c8 & 7;
          *reinterpret_cast<uint4*>(stage[hf] + r * 128 + ((chunk ^ (r & 7)) << 4)) =
              make_uint4(wp[4 * q], wp[4 * q + 1], wp[4 * q + 2], wp[4 * q + 3]);
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(L::kOStaged));
      if (quarter == 0 && lane == 0) {
        if (mbar_wait(bar(L::kOStaged), 0, abort_flag, P.status)) {
          for (int hf = 0; hf < 2; ++hf)
            tma_store_4d(&tm_o, smem_u32(stage[hf]), hf * 64, h, qbase, bt);
          bulk_commit_group();
          // the tile has been read out of shared memory before the CTA exits
          // (the global writes complete on their own)
          bulk_wait_group_read0();
        }
      }
      P.lse[lse_index(P, bt, h, prow)] =
          (l_run > 0.f) ? (m_run + log2f(l_run) - kPLog2) * kLn2 : -INFINITY;
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp) tmem_dealloc(tmem, 256);
}

// [Bt][S][H][128] codes (tokens tok bytes apart) -> [Bt][H][128][S]: one
// block moves 128 tokens x 128 d of one (batch, head) through shared memory.
__global__ void __launch_bounds__(256) v_transpose_kernel(const uint8_t* __restrict__ v,
                                                          uint8_t* __restrict__ vt, int S,
                                                          int H, long long tok) {
  __shared__ __align__(16) uint8_t tile[128][128 + 16];
  const int t0 = blockIdx.x * 128, hh = blockIdx.y, b = blockIdx.z;
  const uint8_t* src = v + ((long long)b * S + t0) * tok + (long long)hh * kD;
  for (int e = threadIdx.x; e < 128 * 8; e += 256) {
    const int row = e >> 3, c16 = e & 7;
    *reinterpret_cast<uint4*>(&tile[row][16 * c16]) =
        *reinterpret_cast<const uint4*>(src + (long long)row * tok + 16 * c16);
  }
  __syncthreads();
  uint8_t* dst = vt + (((long long)b * H + hh) * kD) * S + t0;
  for (int e = threadIdx.x; e < 128 * 8; e += 256) {
    const int d = e & 127, c16 = e >> 7;  // 16 tokens from 16 * c16
    uint32_t w[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int t = 16 * c16 + 4 * k;
      w[k] = (uint32_t)tile[t][d] | ((uint32_t)tile[t + 1][d] << 8) |
             ((uint32_t)tile[t + 2][d] << 16) | ((uint32_t)tile[t + 3][d] << 24);
    }
    *reinterpret_cast<uint4*>(dst + (long long)d * S + 16 * c16) =
        make_uint4(w[0], w[1], w[2], w[3]);
  }
}

// bf16 -> e4m3 codes of x * inv_scale (the product in fp32), 8 per thread
// and step; the tail past a multiple of 8 one by one.
__global__ void __launch_bounds__(256) quantize_e4m3_kernel(const uint16_t* __restrict__ x,
                                                            uint8_t* __restrict__ out,
                                                            long long n, float inv_scale) {
  const long long n8 = n / 8;
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x; e < n8; e += stride) {
    const uint4 a = reinterpret_cast<const uint4*>(x)[e];
    const uint32_t wv[4] = {a.x, a.y, a.z, a.w};
    float f[8];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      f[2 * k] = __uint_as_float(wv[k] << 16) * inv_scale;
      f[2 * k + 1] = __uint_as_float(wv[k] & 0xFFFF0000u) * inv_scale;
    }
    reinterpret_cast<uint2*>(out)[e] =
        make_uint2(pack_e4m3(f[0], f[1]) | (pack_e4m3(f[2], f[3]) << 16),
                   pack_e4m3(f[4], f[5]) | (pack_e4m3(f[6], f[7]) << 16));
  }
  for (long long e = 8 * n8 + (long long)blockIdx.x * blockDim.x + threadIdx.x; e < n;
       e += stride) {
    const float f = __uint_as_float((uint32_t)x[e] << 16) * inv_scale;
    out[e] = (uint8_t)(pack_e4m3(f, 0.f) & 0xFFu);
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

bool encode(CUtensorMap* m, CUtensorMapDataType type, const void* base, const cuuint64_t* dims,
            const cuuint64_t* strides, const cuuint32_t* box) {
  auto fn = encode_fn();
  if (!fn) {
    fail_cuda_msg("cuTensorMapEncodeTiled", "driver entry point not found");
    return false;
  }
  cuuint32_t es[4] = {1, 1, 1, 1};
  CUresult r = fn(m, type, 4, const_cast<void*>(base), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    char msg[64];
    std::snprintf(msg, sizeof(msg), "CUresult %d", (int)r);
    fail_cuda_msg("cuTensorMapEncodeTiled", msg);
    return false;
  }
  return true;
}

}  // namespace

int read_clear_fwd_fp8_status() {
  int v = 0, z = 0;
  if (cudaMemcpyFromSymbol(&v, g_fwd_fp8_status, sizeof(int)) != cudaSuccess) return -1;
  if (v != 0) cudaMemcpyToSymbol(g_fwd_fp8_status, &z, sizeof(int));
  return v;
}

bool fwd_fp8_supported(const AttnParams& P) {
  if (P.D != kD) return false;
  if (P.shard % kBM != 0) return false;
  if (P.layout == kZigzag && P.chunk % kBM != 0) return false;
  return true;
}

usp_status_t launch_v_transpose(const void* v, void* vt, int Bt, int S, int H, cudaStream_t st) {
  if (Bt == 0 || S == 0) return USP_OK;
  {
    ProfScope ps(st, "fp8_v_transpose");
    v_transpose_kernel<<<dim3((unsigned)(S / 128), (unsigned)H, (unsigned)Bt), 256, 0, st>>>(
        static_cast<const uint8_t*>(v), static_cast<uint8_t*>(vt), S, H, (long long)H * kD);
  }
  note_launch();
  return check_launch();
}

usp_status_t launch_quantize_e4m3(const void* x, void* out, long long n, float inv_scale,
                                  cudaStream_t st) {
  if (n == 0) return USP_OK;
  long long blocks = (n / 8 + 255) / 256;
  const long long cap = (long long)sm_count() * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  {
    ProfScope ps(st, "fp8_quantize");
    quantize_e4m3_kernel<<<(unsigned)blocks, 256, 0, st>>>(
        static_cast<const uint16_t*>(x), static_cast<uint8_t*>(out), n, inv_scale);
  }
  note_launch();
  return check_launch();
}

// P.q, P.k: e4m3 [Bt][S][H][128]; P.v: the transposed values [Bt][Hkv][128][S];
// P.o: bf16 [Bt][S][Hq][128]; P.scale_log2 already includes q and k descales.
usp_status_t launch_fwd_fp8(const AttnParams& P, float v_descale, cudaStream_t st) {
  CUtensorMap mq, mk, mvt, mo;
  {
    const cuuint64_t dq[4] = {(cuuint64_t)kD, (cuuint64_t)P.Hq, (cuuint64_t)P.S,
                              (cuuint64_t)P.Bt};
    const cuuint64_t sq[3] = {(cuuint64_t)kD, (cuuint64_t)P.Hq * kD,
                              (cuuint64_t)P.S * P.Hq * kD};
    const cuuint64_t dk[4] = {(cuuint64_t)kD, (cuuint64_t)P.Hkv, (cuuint64_t)P.S,
                              (cuuint64_t)P.Bt};
    const cuuint64_t sk[3] = {(cuuint64_t)kD, (cuuint64_t)P.Hkv * kD,
                              (cuuint64_t)P.S * P.Hkv * kD};
    const cuuint64_t dv[4] = {(cuuint64_t)P.S, (cuuint64_t)kD, (cuuint64_t)P.Hkv,
                              (cuuint64_t)P.Bt};
    const cuuint64_t sv[3] = {(cuuint64_t)P.S, (cuuint64_t)kD * P.S,
                              (cuuint64_t)P.Hkv * kD * P.S};
    const cuuint64_t sodims[4] = {(cuuint64_t)kD, (cuuint64_t)P.Hq, (cuuint64_t)P.S,
                                  (cuuint64_t)P.Bt};
    const cuuint64_t so[3] = {(cuuint64_t)kD * 2, (cuuint64_t)P.Hq * kD * 2,
                              (cuuint64_t)P.S * P.Hq * kD * 2};
    const cuuint32_t box_qk[4] = {128, 1, (cuuint32_t)kBM, 1};
    const cuuint32_t box_v[4] = {(cuuint32_t)kBN, 128, 1, 1};
    const cuuint32_t box_o[4] = {64, 1, (cuuint32_t)kBM, 1};
    if (!encode(&mq, CU_TENSOR_MAP_DATA_TYPE_UINT8, P.q, dq, sq, box_qk) ||
        !encode(&mk, CU_TENSOR_MAP_DATA_TYPE_UINT8, P.k, dk, sk, box_qk) ||
        !encode(&mvt, CU_TENSOR_MAP_DATA_TYPE_UINT8, P.v, dv, sv, box_v) ||
        !encode(&mo, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, P.o, sodims, so, box_o))
      return USP_ERR_CUDA;
  }
  static int* status = nullptr;
  if (status == nullptr) {
    cudaError_t e = cudaGetSymbolAddress(reinterpret_cast<void**>(&status), g_fwd_fp8_status);
    if (e != cudaSuccess) return fail_cuda("cudaGetSymbolAddress(status)", e);
  }
  AttnParams Pk = P;
  Pk.status = status;
  // L2 batches as in the bf16 forward: about eight waves of CTAs (two per
  // SM), in whole GQA groups
  {
    const int ntiles = P.S / kBM;
    int per = (16 * sm_count() + ntiles - 1) / ntiles;
    per = (per + P.G - 1) / P.G * P.G;
    Pk.unit_batch = per < P.Hq * P.Bt ? per : P.Hq * P.Bt;
  }
  const int smem = Smem8::kAlloc;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(attn_fwd_fp8_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return fail_cuda("cudaFuncSetAttribute(smem)", e);
    attr_set = true;
  }
  const long long blocks = (long long)(P.S / kBM) * P.Hq * P.Bt;
  {
    ProfScope ps(st, "attn_fwd_fp8");
    attn_fwd_fp8_kernel<<<(unsigned)blocks, kThreads, smem, st>>>(Pk, v_descale, mq, mk, mvt,
                                                                  mo);
  }
  note_launch();
  return check_launch();
}

}  // namespace usp
