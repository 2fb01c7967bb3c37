// Decode-step attention over a sharded KV cache: split-KV partials, then the
// log-sum-exp merge.
//
// "Long Context Attention" notes, "Ring Attention" (flash decoding is ring
// attention at inference time) and "Tree Attention" (the partials of one
// decoding step combine by a tree reduction, logsumexp being associative):
// the newest Tq tokens of each sequence attend to all S cached keys. The
// cache is in rank-major contiguous order, rank r holding keys
// [r S/cp, (r+1) S/cp). Every rank's shard is cut into `splits` equal pieces
// and one CTA computes the partial (O, LSE) of one piece for all the query
// rows that read one KV head (G query heads x Tq tokens). The standalone
// merge then combines the pieces in key order (tree order: pairwise levels,
// so the pieces of one shard meet first, then the shards).
//
// HBM-bound: every cached key and value is read once. A CTA (one per SM)
// streams its piece through shared memory in tiles of 64 keys (TMA, 128-byte
// swizzle, six stages for up to four query rows per KV head, else five,
// filled by a producer warp). Tile i belongs to the pair of compute warps
// i mod stages, each taking 32 of its keys; every warp runs its
// own online softmax over its keys, so no block-wide barrier is needed
// inside the loop:
//   scores   a lane pair per key, each lane of the pair takes half of D and
//            keys p and p + 16 of the warp's 32 (one at a time when there
//            are more than eight query rows), so a chunk of q, held in
//            shared memory pre-scaled by scale * log2(e), is read once for
//            two keys
//   softmax  running max m and sum l per query row by warp shuffles,
//            P = 2^(s - m) to a warp-private buffer (key-major: a key's row
//            values are one vector read), O rescaled
//   P V      lanes own output columns
// At the end the warps' (m, l, O) are merged with the log-sum-exp rule.
#include <cudaTypedefs.h>

#include <cstdio>

#include "internal.h"
#include "tc_ptx.cuh"

namespace usp {
namespace {

using namespace tc;

__device__ int g_decode_status = 0;

constexpr int kKeys = 64;           // keys per tile
constexpr int kMaxRows = 16;        // G * Tq
constexpr int kWarpsPerTile = 2;    // a tile's keys are split between two warps
constexpr int kWarpKeys = kKeys / kWarpsPerTile;

// K/V tiles in flight per CTA (one CTA per SM), and so compute warps. With
// at most four query rows per KV head the rows' accumulators leave room for
// six stages (thirteen warps: four share a 16K-register sub-partition, so
// <= 128 registers each); with more rows five (eleven warps, <= 168).
template <int R>
__host__ __device__ constexpr int stages_for() { return R <= 4 ? 6 : 5; }
template <int R>
__host__ __device__ constexpr int threads_for() { return 32 * (stages_for<R>() * kWarpsPerTile + 1); }

// keys scored together by a lane pair (sharing each chunk of q): both of
// its keys, or one when the rows' accumulators would not fit the registers
template <int R>
__host__ __device__ constexpr int keys_together() { return R <= 8 ? 2 : 1; }

struct DecodeParams {
  const __nv_bfloat16* q;  // [B][Tq][Hq][D]
  float* o_part;           // [n_part][B*Tq*Hq][D]
  float* lse_part;         // [n_part][B*Tq*Hq]
  int* status;
  int B, Tq, S, Hq, Hkv, G, R;
  int n_part, piece;  // pieces and keys per piece
  float scale_log2;
  int causal;
};

// q rows in shared memory: the second half of each row is shifted by 16
// bytes so that the two lane halves of a warp, which read the same chunk of
// the two halves, hit different banks (one wavefront instead of two).
template <int D>
__host__ __device__ constexpr int kQStride() { return D + 8; }
template <int D>
__device__ __forceinline__ int q_index(int r, int d) {
  return r * kQStride<D>() + d + (d >= D / 2 ? 4 : 0);
}

template <int D, int R>
struct DSmem {
  static constexpr int kStages = stages_for<R>();
  static constexpr int kComputeWarps = kStages * kWarpsPerTile;
  static constexpr int kThreads = threads_for<R>();  // + one producer warp
  static constexpr int kTileBytes = kKeys * D * 2;  // one K or V tile
  static constexpr int kBoxBytes = kKeys * 128;     // 64 columns x 64 keys
  static constexpr int kK = 0;                      // kStages stages
  static constexpr int kV = kK + kStages * kTileBytes;
  static constexpr int kQ = kV + kStages * kTileBytes;  // [R] padded rows, fp32
  static constexpr int kP = kQ + R * kQStride<D>() * 4;  // per warp [kWarpKeys][R] fp32
  static constexpr int kMerge = kP + kComputeWarps * kWarpKeys * R * 4;  // per warp m, l [R]
  static constexpr int kBar = kMerge + 2 * kComputeWarps * kMaxRows * 4;
  static constexpr int kMisc = kBar + 8 * 2 * kStages;  // abort flag
  static constexpr int kBytes = kMisc + 16;
  static constexpr int kAlloc = kBytes + 1024;
  static_assert(kBar % 8 == 0, "barriers need 8-byte alignment");
  static_assert(kComputeWarps * R * D * 4 <= 2 * kStages * kTileBytes,
                "the final merge fits the tiles");
  static_assert(kP % 16 == 0, "vector reads of P");
  static_assert(kAlloc <= 232448, "exceeds the per-CTA shared memory limit");
};

template <int D>
__device__ __forceinline__ const uint8_t* tile_row(const uint8_t* tile, int key, int chunk) {
  // 16-byte chunk `chunk` (0 .. D/8-1) of key row `key` in a 128-byte swizzled
  // tile stored as D/64 boxes of 64 keys x 128 bytes
  const int box = chunk >> 3, c = chunk & 7;
  return tile + box * (kKeys * 128) + key * 128 + ((c ^ (key & 7)) << 4);
}

// bf16 pair (one 32-bit word) -> packed fp32 pair (low element first)
__device__ __forceinline__ uint64_t bf2_to_f2(uint32_t w) {
  return (static_cast<uint64_t>(w & 0xffff0000u) << 32) | static_cast<uint64_t>(w << 16);
}

// R: query rows per KV head, padded to a compiled size (rows >= P.R are
// zero queries whose results are never written).
template <int D, int R>
__global__ void __launch_bounds__(threads_for<R>())
decode_split_kernel(const DecodeParams P, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v) {
  using L = DSmem<D, R>;
  constexpr int kStages = L::kStages, kComputeWarps = L::kComputeWarps, kThreads = L::kThreads;
  static_assert(R <= kMaxRows, "rows");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(sm);
  auto full = [&](int s) { return sbase + L::kBar + 8 * s; };
  auto empty = [&](int s) { return sbase + L::kBar + 8 * (kStages + s); };
  float* qs = reinterpret_cast<float*>(sm + L::kQ);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + L::kMisc);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // KV heads innermost: the CTAs of one piece, which together read whole
  // cache rows (all heads of each key), run side by side
  const int g = blockIdx.x, piece = blockIdx.y, b = blockIdx.z;
  const int key0 = piece * P.piece;
  const int ntiles = P.piece / kKeys;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), kWarpsPerTile);  // the warps that share the stage's tile
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  // query rows r = hh * Tq + t (query head g*G + hh, token t), pre-scaled;
  // padding rows are zero
  for (int idx = threadIdx.x; idx < R * D; idx += kThreads) {
    const int r = idx / D, d = idx - r * D;
    float x = 0.f;
    if (r < P.R) {
      const int hh = r / P.Tq, t = r - hh * P.Tq;
      x = __bfloat162float(P.q[(((long long)b * P.Tq + t) * P.Hq + g * P.G + hh) * D + d]) *
          P.scale_log2;
    }
    qs[q_index<D>(r, d)] = x;
  }
  __syncthreads();

  constexpr int kCols = D / 32, kPairs = kCols / 2;
  if (warp == kComputeWarps) {
    // ---------------------------------------------------------- producer
    if (lane == 0) {
      tma_prefetch(&tm_k);
      tma_prefetch(&tm_v);
      int issued = 0;
      for (int i = 0; i < ntiles; ++i) {
        const int st = i % kStages;
        // the stage is free once its warps have released tile i - kStages
        if (i >= kStages &&
            !mbar_wait(empty(st), (i / kStages - 1) & 1, abort_flag, P.status))
          break;
        mbar_expect_tx(full(st), 2 * L::kTileBytes);
        for (int hf = 0; hf < D / 64; ++hf) {
          tma_load_4d(sbase + L::kK + st * L::kTileBytes + hf * L::kBoxBytes, &tm_k, full(st),
                      hf * 64, g, key0 + i * kKeys, b);
          tma_load_4d(sbase + L::kV + st * L::kTileBytes + hf * L::kBoxBytes, &tm_v, full(st),
                      hf * 64, g, key0 + i * kKeys, b);
        }
        issued = i + 1;
      }
      if (*abort_flag) {
        // aborted: let the copies already issued land before the tiles are reused
        for (int i = (issued >= kStages ? issued - kStages : 0); i < issued; ++i)
          mbar_wait_drain(full(i % kStages), (i / kStages) & 1);
      }
    }
  } else {
    // ---------------------------------------------------------- compute warps
    // Each warp runs its own online softmax over its keys of its tiles
    // (tiles i = warp / 2, warp / 2 + stages, ..., keys [32 h, 32 h + 32) with
    // h = warp mod 2): running max m, running sum l and the O accumulator
    // (packed fp32 pairs, lane owns columns kCols*lane ..), merged across
    // warps at the end.
    constexpr int KG = keys_together<R>();
    constexpr int kPasses = kWarpKeys / 16;
    const int kbase = (warp % kWarpsPerTile) * kWarpKeys;
    float* pw = reinterpret_cast<float*>(sm + L::kP) + warp * kWarpKeys * R;  // [kWarpKeys][R]
    float m[R], l[R];
    uint64_t o2[R][kPairs];
#pragma unroll
    for (int r = 0; r < R; ++r) {
      m[r] = -INFINITY;
      l[r] = 0.f;
#pragma unroll
      for (int j = 0; j < kPairs; ++j) o2[r][j] = 0ull;
    }
    const int qpos0 = P.S - P.Tq;  // position of token t = 0
    const int pr = lane & 15, hs = lane >> 4;
    const int col = kCols * lane;
    for (int i = warp / kWarpsPerTile; i < ntiles; i += kStages) {
      const int st = i % kStages;
      bool ok = true;
      if (lane == 0) ok = mbar_wait(full(st), (i / kStages) & 1, abort_flag, P.status);
      if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) break;
      const uint8_t* kt = sm + L::kK + st * L::kTileBytes;
      const uint8_t* vt = sm + L::kV + st * L::kTileBytes;
      // the warp's keys in passes of 16 KG: the lane pair's keys
      // kbase + pr + 16 (jb + g), g < KG
#pragma unroll
      for (int jb = 0; jb < kPasses; jb += KG) {
        // scores: a lane pair per key, each lane half of D
        uint64_t acc2[KG][R];
#pragma unroll
        for (int g = 0; g < KG; ++g)
#pragma unroll
          for (int r = 0; r < R; ++r) acc2[g][r] = 0ull;
#pragma unroll
        for (int c = 0; c < D / 16; ++c) {
          const int chunk = hs * (D / 16) + c;
          uint64_t kr[KG][4];
#pragma unroll
          for (int g = 0; g < KG; ++g) {
            const uint4 raw = *reinterpret_cast<const uint4*>(
                tile_row<D>(kt, kbase + pr + 16 * (jb + g), chunk));
            kr[g][0] = bf2_to_f2(raw.x);
            kr[g][1] = bf2_to_f2(raw.y);
            kr[g][2] = bf2_to_f2(raw.z);
            kr[g][3] = bf2_to_f2(raw.w);
          }
#pragma unroll
          for (int r = 0; r < R; ++r) {
            const float* qp = qs + q_index<D>(r, chunk * 8);
            const ulonglong2 qa = *reinterpret_cast<const ulonglong2*>(qp);
            const ulonglong2 qb = *reinterpret_cast<const ulonglong2*>(qp + 4);
#pragma unroll
            for (int g = 0; g < KG; ++g) {
              acc2[g][r] = f2_fma(qa.x, kr[g][0], acc2[g][r]);
              acc2[g][r] = f2_fma(qa.y, kr[g][1], acc2[g][r]);
              acc2[g][r] = f2_fma(qb.x, kr[g][2], acc2[g][r]);
              acc2[g][r] = f2_fma(qb.y, kr[g][3], acc2[g][r]);
            }
          }
        }
        // softmax over the pass's 16 KG keys (both lane halves hold the same
        // values after the first reduction; later ones stay within a half)
#pragma unroll
        for (int r = 0; r < R; ++r) {
          float sc[KG];
          float mx = -INFINITY;
#pragma unroll
          for (int g = 0; g < KG; ++g) {
            float lo, hi;
            f2_unpack(acc2[g][r], lo, hi);
            float x = lo + hi;
            x += __shfl_xor_sync(0xffffffffu, x, 16);
            const int kpos = key0 + i * kKeys + kbase + pr + 16 * (jb + g);
            if (P.causal && kpos > qpos0 + r % P.Tq) x = -INFINITY;
            sc[g] = x;
            mx = fmaxf(mx, x);
          }
#pragma unroll
          for (int off = 8; off > 0; off >>= 1)
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
          const float m_new = fmaxf(m[r], mx);
          float a = 1.f, sum = 0.f;
          float pg[KG];
#pragma unroll
          for (int g = 0; g < KG; ++g) pg[g] = 0.f;
          if (m_new != -INFINITY) {
            a = (m[r] == -INFINITY) ? 0.f : ex2(m[r] - m_new);
#pragma unroll
            for (int g = 0; g < KG; ++g) {
              pg[g] = (sc[g] == -INFINITY) ? 0.f : ex2(sc[g] - m_new);
              sum += pg[g];
            }
          }
#pragma unroll
          for (int off = 8; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
          l[r] = l[r] * a + sum;
          m[r] = m_new;
          const uint64_t a2 = f2_pack(a, a);
#pragma unroll
          for (int j = 0; j < kPairs; ++j) o2[r][j] = f2_fma(o2[r][j], a2, 0ull);
          if (hs == 0) {
#pragma unroll
            for (int g = 0; g < KG; ++g) pw[(pr + 16 * (jb + g)) * R + r] = pg[g];
          }
        }
        __syncwarp();
        // P V over the pass's keys, lane owns columns
#pragma unroll 4
        for (int kk = 16 * jb; kk < 16 * (jb + KG); ++kk) {
          const uint8_t* src = tile_row<D>(vt, kbase + kk, col >> 3) + (col & 7) * 2;
          uint64_t v2[kPairs];
          if constexpr (kPairs == 2) {
            const uint2 raw = *reinterpret_cast<const uint2*>(src);
            v2[0] = bf2_to_f2(raw.x);
            v2[1] = bf2_to_f2(raw.y);
          } else {
            v2[0] = bf2_to_f2(*reinterpret_cast<const uint32_t*>(src));
          }
          float pv[R];
          if constexpr (R % 4 == 0) {
#pragma unroll
            for (int r4 = 0; r4 < R / 4; ++r4) {
              const float4 x = *reinterpret_cast<const float4*>(pw + kk * R + 4 * r4);
              pv[4 * r4] = x.x; pv[4 * r4 + 1] = x.y; pv[4 * r4 + 2] = x.z; pv[4 * r4 + 3] = x.w;
            }
          } else {
#pragma unroll
            for (int r = 0; r < R; ++r) pv[r] = pw[kk * R + r];
          }
#pragma unroll
          for (int r = 0; r < R; ++r) {
            const uint64_t p2 = f2_pack(pv[r], pv[r]);
#pragma unroll
            for (int j = 0; j < kPairs; ++j) o2[r][j] = f2_fma(p2, v2[j], o2[r][j]);
          }
        }
        __syncwarp();  // the P buffer is reused by the next pass
      }
      if (lane == 0) mbar_arrive(empty(st));  // this warp is done with the stage
    }
    // every compute warp is done with the tiles (named barrier of the four
    // compute warps, reached on the abort path too) before the partials
    // overwrite them
    asm volatile("bar.sync 1, %0;" ::"r"(kComputeWarps * 32) : "memory");
    // this warp's partial: m, l per row and its O columns (through the
    // now idle tiles)
    float* mw = reinterpret_cast<float*>(sm + L::kMerge);
    float* lw = mw + kComputeWarps * kMaxRows;
    float* red = reinterpret_cast<float*>(sm + L::kK);  // [warps][R][D]
    if (lane == 0) {
#pragma unroll
      for (int r = 0; r < R; ++r) {
        mw[warp * kMaxRows + r] = m[r];
        lw[warp * kMaxRows + r] = l[r];
      }
    }
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
      for (int j = 0; j < kPairs; ++j)
        *reinterpret_cast<uint64_t*>(red + (warp * R + r) * D + col + 2 * j) = o2[r][j];
  }
  __syncthreads();
  if (*abort_flag) return;
  // merge the warps' partials with the log-sum-exp rule (log2 units)
  const float* mw = reinterpret_cast<const float*>(sm + L::kMerge);
  const float* lw = mw + kComputeWarps * kMaxRows;
  const float* red = reinterpret_cast<const float*>(sm + L::kK);
  const long long rows = (long long)P.B * P.Tq * P.Hq;
  for (int idx = threadIdx.x; idx < P.R * D; idx += kThreads) {
    const int r = idx / D, d = idx - r * D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kComputeWarps; ++w) M = fmaxf(M, mw[w * kMaxRows + r]);
    float Ls = 0.f, Os = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kComputeWarps; ++w) {
        const float mwr = mw[w * kMaxRows + r];
        const float f = (mwr == -INFINITY) ? 0.f : ex2(mwr - M);
        Ls += lw[w * kMaxRows + r] * f;
        Os += red[(w * R + r) * D + d] * f;
      }
    }
    const int hh = r / P.Tq, t = r - hh * P.Tq;
    const long long row = ((long long)b * P.Tq + t) * P.Hq + g * P.G + hh;
    P.o_part[((long long)piece * rows + row) * D + d] = Ls > 0.f ? Os / Ls : 0.f;
    if (d == 0)
      P.lse_part[(long long)piece * rows + row] =
          Ls > 0.f ? (M + log2f(Ls)) * 0.6931471805599453f : -INFINITY;
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

// [B][S][Hkv][D] bf16 cache -> 4-D map (D, Hkv, S, B), box (64, 1, 64, 1).
bool make_cache_map(CUtensorMap* m, const void* base, int B, int S, int H, int D) {
  auto fn = encode_fn();
  if (!fn) {
    fail_cuda_msg("cuTensorMapEncodeTiled", "driver entry point not found");
    return false;
  }
  cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)S, (cuuint64_t)B};
  cuuint64_t strides[3] = {(cuuint64_t)D * 2, (cuuint64_t)H * D * 2,
                           (cuuint64_t)S * H * D * 2};
  cuuint32_t box[4] = {64, 1, (cuuint32_t)kKeys, 1};
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
usp_status_t launch_d(const DecodeParams& P, const void* k, const void* v, cudaStream_t st) {
  CUtensorMap mk, mv;
  if (!make_cache_map(&mk, k, P.B, P.S, P.Hkv, D) || !make_cache_map(&mv, v, P.B, P.S, P.Hkv, D))
    return USP_ERR_CUDA;
  static int* status = nullptr;
  if (status == nullptr) {
    cudaError_t e = cudaGetSymbolAddress(reinterpret_cast<void**>(&status), g_decode_status);
    if (e != cudaSuccess) return fail_cuda("cudaGetSymbolAddress(status)", e);
  }
  DecodeParams Pk = P;
  Pk.status = status;
  dim3 grid(P.Hkv, P.n_part, P.B);
  auto go = [&](auto kernel, int smem, int threads) -> usp_status_t {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         smem);
    if (e != cudaSuccess) return fail_cuda("cudaFuncSetAttribute(smem)", e);
    {
      ProfScope ps(st, "attn_decode_split");
      kernel<<<grid, threads, smem, st>>>(Pk, mk, mv);
    }
    note_launch();
    return check_launch();
  };
  if (P.R <= 1) return go(decode_split_kernel<D, 1>, DSmem<D, 1>::kAlloc, DSmem<D, 1>::kThreads);
  if (P.R <= 2) return go(decode_split_kernel<D, 2>, DSmem<D, 2>::kAlloc, DSmem<D, 2>::kThreads);
  if (P.R <= 4) return go(decode_split_kernel<D, 4>, DSmem<D, 4>::kAlloc, DSmem<D, 4>::kThreads);
  if (P.R <= 8) return go(decode_split_kernel<D, 8>, DSmem<D, 8>::kAlloc, DSmem<D, 8>::kThreads);
  return go(decode_split_kernel<D, 16>, DSmem<D, 16>::kAlloc, DSmem<D, 16>::kThreads);
}

}  // namespace

int read_clear_decode_status() {
  int v = 0, z = 0;
  if (cudaMemcpyFromSymbol(&v, g_decode_status, sizeof(int)) != cudaSuccess) return -1;
  if (v != 0) cudaMemcpyToSymbol(g_decode_status, &z, sizeof(int));
  return v;
}

int decode_max_rows() { return kMaxRows; }
int decode_keys_per_tile() { return kKeys; }

usp_status_t launch_decode_split(const void* q, const void* k, const void* v, float* o_part,
                                 float* lse_part, int B, int Tq, int S, int Hq, int Hkv, int D,
                                 float scale, int causal, int n_part, cudaStream_t st) {
  DecodeParams P{};
  P.q = reinterpret_cast<const __nv_bfloat16*>(q);
  P.o_part = o_part;
  P.lse_part = lse_part;
  P.B = B;
  P.Tq = Tq;
  P.S = S;
  P.Hq = Hq;
  P.Hkv = Hkv;
  P.G = Hq / Hkv;
  P.R = P.G * Tq;
  P.n_part = n_part;
  P.piece = S / n_part;
  P.scale_log2 = scale * 1.4426950408889634f;
  P.causal = causal;
  return D == 128 ? launch_d<128>(P, k, v, st) : launch_d<64>(P, k, v, st);
}

}  // namespace usp
