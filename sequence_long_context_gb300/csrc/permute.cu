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

int grid_for(long long warp_units) {
  static int sms = 0;
  if (sms == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (sms <= 0) sms = 1;
  }
  constexpr long long kWarpsPerBlock = kThreads / 32;
  long long need = (warp_units + kWarpsPerBlock - 1) / kWarpsPerBlock;
  long long cap = (long long)sms * 8;  // 8 resident 256-thread blocks per SM
  return (int)(need < cap ? (need < 1 ? 1 : need) : cap);
}

// One warp copies one contiguous run of n 16-byte vectors, four per lane in
// flight.
__device__ __forceinline__ void warp_copy(const uint4* __restrict__ s,
                                          uint4* __restrict__ d, unsigned n,
                                          unsigned lane) {
  unsigned c = lane;
  for (; c + 96 < n; c += 128) {
    const uint4 a = __ldg(s + c), b = __ldg(s + c + 32), e = __ldg(s + c + 64),
                f = __ldg(s + c + 96);
    d[c] = a;
    d[c + 32] = b;
    d[c + 64] = e;
    d[c + 96] = f;
  }
  for (; c < n; c += 32) d[c] = __ldg(s + c);
}

// Token row p of the rank-major tensor <-> token row nat(p) of the natural
// tensor; a row (H*D elements) is rv vectors. One warp per row.
__global__ void __launch_bounds__(kThreads)
permute_layout_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst,
                      unsigned rows, unsigned S, unsigned rv, int layout,
                      int cp, int shard, int chunk, int restore) {
  const unsigned lane = threadIdx.x & 31;
  const unsigned nwarps = gridDim.x * (kThreads / 32);
  for (unsigned r = blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5); r < rows;
       r += nwarps) {
    const unsigned b = r / S, p = r - b * S;
    const unsigned other = b * S + (unsigned)nat_pos((int)p, layout, cp, shard, chunk);
    const size_t so = (size_t)(restore ? r : other) * rv;
    const size_t dof = (size_t)(restore ? other : r) * rv;
    warp_copy(src + so, dst + dof, rv, lane);
  }
}

// Ulysses exchange: src [B*S][ud][rvu] <-> dst [ud][B*S][rvu] (16-byte
// vectors); one warp per (group, token row). With layout >= 0 the flat side
// is in natural sequence order and the grouped side in rank-major order:
// the layout's extract (seq2head) or restore (head2seq) rides along with the
// exchange, so the tensor is moved once instead of twice.
__global__ void __launch_bounds__(kThreads)
ulysses_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst,
               unsigned BS, unsigned rvu, unsigned ud, int seq2head,
               unsigned flat_stride, unsigned flat_off, unsigned S, int layout,
               int cp, int shard, int chunk) {
  const unsigned lane = threadIdx.x & 31;
  const unsigned nwarps = gridDim.x * (kThreads / 32);
  const unsigned units = BS * ud;
  for (unsigned t = blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5); t < units;
       t += nwarps) {
    const unsigned grp = t / BS, r = t - grp * BS;
    const size_t grouped = (size_t)(grp * BS + r) * rvu;  // [ud][B*S] order
    // token row of the flat side: the same row, or (natural order) the row
    // of the rank-major row's natural position
    unsigned fr = r;
    if (layout >= 0) {
      const unsigned b = r / S, p = r - b * S;
      fr = b * S + (unsigned)nat_pos((int)p, layout, cp, shard, chunk);
    }
    // [B*S][ud] order; a token's row may sit inside a wider one (flat_stride
    // vectors per token, starting flat_off vectors in: a packed q/k/v tensor)
    const size_t flat = (size_t)fr * flat_stride + flat_off + (size_t)grp * rvu;
    if (seq2head)
      warp_copy(src + flat, dst + grouped, rvu, lane);
    else
      warp_copy(src + grouped, dst + flat, rvu, lane);
  }
}

}  // namespace

usp_status_t launch_permute_layout(const void* src, void* dst, int B, int S,
                                   int row_bytes, int layout, int cp,
                                   int restore, cudaStream_t st) {
  unsigned rv = (unsigned)(row_bytes / 16);
  unsigned rows = (unsigned)B * (unsigned)S;
  if ((long long)rows * rv == 0) return USP_OK;
  int shard = S / cp;
  int chunk = layout == kZigzag ? S / (2 * cp) : shard;
  {
    ProfScope ps(st, "permute_layout");
    permute_layout_kernel<<<grid_for(rows), kThreads, 0, st>>>(
        reinterpret_cast<const uint4*>(src), reinterpret_cast<uint4*>(dst),
        rows, (unsigned)S, rv, layout, cp, shard, chunk, restore);
  }
  note_launch();
  return check_launch();
}

usp_status_t launch_ulysses(const void* src, void* dst, int B, int S,
                            int row_bytes, int ud, int seq2head,
                            cudaStream_t st, int flat_row_bytes, int flat_off_bytes,
                            int natural_layout, int cp) {
  unsigned rvu = (unsigned)(row_bytes / ud / 16);
  if (flat_row_bytes == 0) flat_row_bytes = row_bytes;
  unsigned BS = (unsigned)B * (unsigned)S;
  if ((long long)BS * rvu * ud == 0) return USP_OK;
  {
    ProfScope ps(st, "permute_ulysses");
    ulysses_kernel<<<grid_for((long long)BS * ud), kThreads, 0, st>>>(
        reinterpret_cast<const uint4*>(src), reinterpret_cast<uint4*>(dst),
        BS, rvu, (unsigned)ud, seq2head, (unsigned)(flat_row_bytes / 16),
        (unsigned)(flat_off_bytes / 16), (unsigned)S, natural_layout, cp, S / cp,
        natural_layout == kZigzag ? S / (2 * cp) : S / cp);
  }
  note_launch();
  return check_launch();
}

}  // namespace usp
