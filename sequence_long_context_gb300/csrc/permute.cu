// Layout permutes and the Ulysses all-to-all, emulated in device memory.
//
// Both are pure data movement, so they are HBM-bound: each token row
// (H*D*elem bytes, a multiple of 16) is moved with 16-byte vector loads and
// stores, several vectors in flight per thread, over a grid sized to the SM
// count. Results are bit-exact copies.
//
// EXTRACT/RESTORE reorder the sequence into rank-major order for the
// contiguous, zigzag and stripe layouts (YunChang README "2. Usage":
// inputs are reordered with the extract function before load-balanced ring
// attention; "Long Context Attention" notes, "Solution" and "Zig-Zag
// Attention"). The Ulysses exchange (DeepSpeed-Ulysses all-to-all used by
// USP) turns sequence shards with all heads into head groups with all of the
// ring rank's tokens: dst[u][b][p][h][d] = src[b][p][u*H/ud + h][d].
#include "internal.h"

namespace usp {
namespace {

constexpr int kThreads = 256;
constexpr int kVecPerThread = 4;

int grid_for(long long work_items) {
  static int sms = 0;
  if (sms == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (sms <= 0) sms = 1;
  }
  long long per_block = (long long)kThreads * kVecPerThread;
  long long need = (work_items + per_block - 1) / per_block;
  long long cap = (long long)sms * 8;  // 8 resident 256-thread blocks per SM
  return (int)(need < cap ? (need < 1 ? 1 : need) : cap);
}

// dst row p <- src row nat(p) (extract) or dst row nat(p) <- src row p.
__global__ void __launch_bounds__(kThreads)
permute_layout_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst,
                      unsigned rows, unsigned S, unsigned rv, int layout,
                      int cp, int shard, int chunk, int restore) {
  const unsigned total = rows * rv;
  const unsigned stride = gridDim.x * blockDim.x;
  unsigned f = blockIdx.x * blockDim.x + threadIdx.x;
  for (; f < total; f += stride * kVecPerThread) {
    uint4 val[kVecPerThread];
    unsigned dsti[kVecPerThread];
#pragma unroll
    for (int u = 0; u < kVecPerThread; ++u) {
      unsigned g = f + u * stride;
      if (g < total) {
        unsigned r = g / rv, c = g - r * rv;
        unsigned b = r / S, p = r - b * S;
        unsigned np = (unsigned)nat_pos((int)p, layout, cp, shard, chunk);
        unsigned a = (b * S + np) * rv + c;
        if (restore) {
          val[u] = __ldg(src + g);
          dsti[u] = a;
        } else {
          val[u] = __ldg(src + a);
          dsti[u] = g;
        }
      }
    }
#pragma unroll
    for (int u = 0; u < kVecPerThread; ++u) {
      unsigned g = f + u * stride;
      if (g < total) dst[dsti[u]] = val[u];
    }
  }
}

// Ulysses: src [B][S][ud*rvu] <-> dst [ud][B][S][rvu] (16-byte vectors).
__global__ void __launch_bounds__(kThreads)
ulysses_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst,
               unsigned BS, unsigned rvu, unsigned ud, int seq2head) {
  const unsigned total = BS * rvu * ud;
  const unsigned stride = gridDim.x * blockDim.x;
  unsigned f = blockIdx.x * blockDim.x + threadIdx.x;
  for (; f < total; f += stride * kVecPerThread) {
    uint4 val[kVecPerThread];
    unsigned dsti[kVecPerThread];
#pragma unroll
    for (int u = 0; u < kVecPerThread; ++u) {
      unsigned g = f + u * stride;  // index in the head-grouped tensor
      if (g < total) {
        unsigned grp = g / (BS * rvu);
        unsigned rem = g - grp * (BS * rvu);
        unsigned r = rem / rvu, c = rem - r * rvu;
        unsigned a = (r * ud + grp) * rvu + c;  // index in [B][S][H] order
        if (seq2head) {
          val[u] = __ldg(src + a);
          dsti[u] = g;
        } else {
          val[u] = __ldg(src + g);
          dsti[u] = a;
        }
      }
    }
#pragma unroll
    for (int u = 0; u < kVecPerThread; ++u) {
      unsigned g = f + u * stride;
      if (g < total) dst[dsti[u]] = val[u];
    }
  }
}

}  // namespace

usp_status_t launch_permute_layout(const void* src, void* dst, int B, int S,
                                   int row_bytes, int layout, int cp,
                                   int restore, cudaStream_t st) {
  unsigned rv = (unsigned)(row_bytes / 16);
  unsigned rows = (unsigned)B * (unsigned)S;
  long long total = (long long)rows * rv;
  if (total == 0) return USP_OK;
  int shard = S / cp;
  int chunk = layout == kZigzag ? S / (2 * cp) : shard;
  {
    ProfScope ps(st, "permute_layout");
    permute_layout_kernel<<<grid_for(total), kThreads, 0, st>>>(
        reinterpret_cast<const uint4*>(src), reinterpret_cast<uint4*>(dst),
        rows, (unsigned)S, rv, layout, cp, shard, chunk, restore);
  }
  note_launch();
  return check_launch();
}

usp_status_t launch_ulysses(const void* src, void* dst, int B, int S,
                            int row_bytes, int ud, int seq2head,
                            cudaStream_t st) {
  unsigned rvu = (unsigned)(row_bytes / ud / 16);
  unsigned BS = (unsigned)B * (unsigned)S;
  long long total = (long long)BS * rvu * ud;
  if (total == 0) return USP_OK;
  {
    ProfScope ps(st, "permute_ulysses");
    ulysses_kernel<<<grid_for(total), kThreads, 0, st>>>(
        reinterpret_cast<const uint4*>(src), reinterpret_cast<uint4*>(dst),
        BS, rvu, (unsigned)ud, seq2head);
  }
  note_launch();
  return check_launch();
}

}  // namespace usp
