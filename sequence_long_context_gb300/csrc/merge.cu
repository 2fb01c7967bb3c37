// Standalone log-sum-exp merge of n attention partials.
//
// "Long Context Attention" notes, "Tree Attention": logsumexp and max are
// associative, so partial results over disjoint key sets can be reduced in
// any order, e.g. along a tree. For two partials (O_a, L_a), (O_b, L_b):
//   m = max(L_a, L_b), L = m + log(exp(L_a - m) + exp(L_b - m)),
//   O = exp(L_a - L) O_a + exp(L_b - L) O_b;  L = -inf is the identity.
//
// Layout: o_parts [n][rows][D] fp32, lse_parts [n][rows]. A thread owns 4
// consecutive floats (16 bytes) of a row, so D/4 consecutive threads read one
// partial row as one coalesced 256/512-byte segment. HBM-bound: the kernels
// keep many 16-byte loads in flight per thread (every partial of two rows for
// n <= 8) and size the grid to exactly fill the SMs.
//
// Ring order folds left to right. Tree order (pairwise levels, an odd last
// partial carried up unchanged) builds the same tree as a binary counter:
// push each partial, merge the top two while they have equal level, and at
// the end fold the stack from the top down. That needs a stack of at most
// log2(n)+1 entries. For n <= 8 the levels are unrolled at compile time
// (stride doubling), which gives the same tree.
#include "internal.h"

namespace usp {
namespace {

constexpr int kThreads = 256;
constexpr int kRegParts = 8;       // partials loaded together (one aligned block)
constexpr int kMaxBlockDepth = 4;  // counter stack over blocks of 8: n <= 64

// rows in flight per thread on the register path: two rows while that keeps
// the registers low enough for four blocks per SM
template <int NP>
__host__ __device__ constexpr int rows_per_thread() { return NP <= 4 ? 2 : 1; }

__device__ __forceinline__ float4 ld_stream(const float* p) {
  return __ldcs(reinterpret_cast<const float4*>(p));
}

__device__ __forceinline__ void merge_into(float4& oa, float& la, const float4& ob,
                                           float lb) {
  // (oa, la) <- (oa, la) (+) (ob, lb); an empty partial is the identity and
  // its O is never read.
  if (lb == -INFINITY) return;
  if (la == -INFINITY) {
    oa = ob;
    la = lb;
    return;
  }
  float m = fmaxf(la, lb);
  float ea = expf(la - m);
  float eb = expf(lb - m);
  float tot = ea + eb;
  float inv = 1.f / tot;
  float wa = ea * inv, wb = eb * inv;
  oa.x = wa * oa.x + wb * ob.x;
  oa.y = wa * oa.y + wb * ob.y;
  oa.z = wa * oa.z + wb * ob.z;
  oa.w = wa * oa.w + wb * ob.w;
  la = m + logf(tot);
}

__device__ __forceinline__ void store4(float* d, const float4& v) {
  __stcs(reinterpret_cast<float4*>(d), v);
}
__device__ __forceinline__ void store4(__nv_bfloat16* d, const float4& v) {
  __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y);
  __nv_bfloat162 b = __floats2bfloat162_rn(v.z, v.w);
  uint2 x;
  x.x = *reinterpret_cast<unsigned*>(&a);
  x.y = *reinterpret_cast<unsigned*>(&b);
  __stcs(reinterpret_cast<uint2*>(d), x);
}

// n = NP <= 8 partials: every partial of rows_per_thread<NP>() rows is loaded
// before any arithmetic, then merged in registers.
template <int D, int NP, typename TO>
__global__ void __launch_bounds__(kThreads)
merge_reg_kernel(const float* __restrict__ o_parts, const float* __restrict__ lse_parts,
                 long long rows, int tree, TO* __restrict__ o_out,
                 float* __restrict__ lse_out) {
  constexpr int kLPR = D / 4;               // threads per row
  constexpr int kRPB = kThreads / kLPR;     // rows per block and pass
  constexpr int kRowsPerThread = rows_per_thread<NP>();
  const int sub = threadIdx.x / kLPR, c = (threadIdx.x % kLPR) * 4;
  const long long step = (long long)gridDim.x * kRPB * kRowsPerThread;
  for (long long r0 = (long long)blockIdx.x * kRPB * kRowsPerThread; r0 < rows; r0 += step) {
    float4 part[kRowsPerThread][NP];
    float pl[kRowsPerThread][NP];
#pragma unroll
    for (int j = 0; j < kRowsPerThread; ++j) {
      const long long row = r0 + j * kRPB + sub;
      if (row < rows) {
#pragma unroll
        for (int i = 0; i < NP; ++i) {
          part[j][i] = ld_stream(o_parts + ((long long)i * rows + row) * D + c);
          pl[j][i] = __ldg(lse_parts + (long long)i * rows + row);
        }
      }
    }
#pragma unroll
    for (int j = 0; j < kRowsPerThread; ++j) {
      const long long row = r0 + j * kRPB + sub;
      if (row >= rows) continue;
#pragma unroll
      for (int i = 0; i < NP; ++i)
        if (pl[j][i] == -INFINITY) part[j][i] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (!tree) {
#pragma unroll
        for (int i = 1; i < NP; ++i) merge_into(part[j][0], pl[j][0], part[j][i], pl[j][i]);
      } else {
        // pairwise levels: at stride s, slot i absorbs slot i + s; a slot
        // without a partner is carried up unchanged
#pragma unroll
        for (int s = 1; s < NP; s *= 2)
#pragma unroll
          for (int i = 0; i + s < NP; i += 2 * s)
            merge_into(part[j][i], pl[j][i], part[j][i + s], pl[j][i + s]);
      }
      store4(o_out + row * D + c, part[j][0]);
      if (c == 0) lse_out[row] = pl[j][0];
    }
  }
}

// Per-row state of merge_stack_kernel: the binary-counter stack of block
// results (and an accumulator, used when the kernel folds in linear order).
struct StackState {
  float4 acc;
  float L;
  float4 st_o[kMaxBlockDepth];
  float st_l[kMaxBlockDepth];
  int st_lv[kMaxBlockDepth];
  int top;
};

// Loads and reduces one aligned block of partials [b0, b0 + r); kFull means
// r == kRegParts, known at compile time, so the loads carry no predicate.
template <bool kFull>
__device__ __forceinline__ void merge_block(const float* op, const float* lse, long long pstride,
                                            long long rows, long long row, int b0, int r,
                                            int tree, StackState& S) {
  if (kFull) r = kRegParts;
  float4 part[kRegParts];
  float pl[kRegParts];
#pragma unroll
  for (int i = 0; i < kRegParts; ++i)
    if (i < r) {
      part[i] = ld_stream(op + (b0 + i) * pstride);
      pl[i] = __ldg(lse + (long long)(b0 + i) * rows + row);
    }
#pragma unroll
  for (int i = 0; i < kRegParts; ++i)
    if (i < r && pl[i] == -INFINITY) part[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  if (!tree) {
#pragma unroll
    for (int i = 0; i < kRegParts; ++i)
      if (i < r) merge_into(S.acc, S.L, part[i], pl[i]);
    return;
  }
#pragma unroll
  for (int s = 1; s < kRegParts; s *= 2)
#pragma unroll
    for (int i = 0; i + s < kRegParts; i += 2 * s)
      if (i + s < r) merge_into(part[i], pl[i], part[i + s], pl[i + s]);
  float4 cur = part[0];
  float cl = pl[0];
  int lv = 0;
  while (S.top > 0 && S.st_lv[S.top - 1] == lv) {
    // (stack top) (+) cur, left operand first
    float4 lo = S.st_o[S.top - 1];
    float ll = S.st_l[S.top - 1];
    merge_into(lo, ll, cur, cl);
    cur = lo;
    cl = ll;
    ++lv;
    --S.top;
  }
  S.st_o[S.top] = cur;
  S.st_l[S.top] = cl;
  S.st_lv[S.top] = lv;
  ++S.top;
}

// any n, linear order: fold left to right with two partials in flight (few
// registers, so many rows per SM are in flight instead).
template <int D, typename TO>
__global__ void __launch_bounds__(kThreads)
merge_linear_kernel(const float* __restrict__ o_parts, const float* __restrict__ lse_parts,
                    int n, long long rows, TO* __restrict__ o_out,
                    float* __restrict__ lse_out) {
  constexpr int kLPR = D / 4;
  constexpr int kRPB = kThreads / kLPR;
  const int sub = threadIdx.x / kLPR, c = (threadIdx.x % kLPR) * 4;
  for (long long row = (long long)blockIdx.x * kRPB + sub; row < rows;
       row += (long long)gridDim.x * kRPB) {
    const float* op = o_parts + row * D + c;
    const long long pstride = rows * D;
    float4 acc = ld_stream(op);
    float L = __ldg(lse_parts + row);
    if (L == -INFINITY) acc = make_float4(0.f, 0.f, 0.f, 0.f);
    int i = 1;
    for (; i + 1 < n; i += 2) {
      const float4 b0 = ld_stream(op + i * pstride);
      const float4 b1 = ld_stream(op + (i + 1) * pstride);
      const float l0 = __ldg(lse_parts + (long long)i * rows + row);
      const float l1 = __ldg(lse_parts + (long long)(i + 1) * rows + row);
      merge_into(acc, L, b0, l0);
      merge_into(acc, L, b1, l1);
    }
    for (; i < n; ++i)
      merge_into(acc, L, ld_stream(op + i * pstride),
                 __ldg(lse_parts + (long long)i * rows + row));
    store4(o_out + row * D + c, acc);
    if (c == 0) lse_out[row] = L;
  }
}

// any n, tree order: partials are loaded in aligned blocks of 8 (eight loads
// in flight). Each block is reduced by pairwise levels (an aligned block of 8
// leaves is one subtree of the pairwise-level tree; a short last block is the
// same tree on its leaves) and combines the blocks with the binary-counter
// stack.
template <int D, typename TO>
__global__ void __launch_bounds__(kThreads)
merge_stack_kernel(const float* __restrict__ o_parts, const float* __restrict__ lse_parts,
                   int n, long long rows, int tree, TO* __restrict__ o_out,
                   float* __restrict__ lse_out) {
  constexpr int kLPR = D / 4;
  constexpr int kRPB = kThreads / kLPR;
  const int sub = threadIdx.x / kLPR, c = (threadIdx.x % kLPR) * 4;
  for (long long row = (long long)blockIdx.x * kRPB + sub; row < rows;
       row += (long long)gridDim.x * kRPB) {
    const float* op = o_parts + row * D + c;
    const long long pstride = rows * D;
    StackState S;
    S.acc = make_float4(0.f, 0.f, 0.f, 0.f);
    S.L = -INFINITY;  // the identity
    S.top = 0;
    int b0 = 0;
    for (; b0 + kRegParts <= n; b0 += kRegParts)
      merge_block<true>(op, lse_parts, pstride, rows, row, b0, kRegParts, tree, S);
    if (b0 < n) merge_block<false>(op, lse_parts, pstride, rows, row, b0, n - b0, tree, S);
    if (tree) {
      // fold from the top: (s0 + (s1 + (s2 + ...)))
      S.acc = S.st_o[S.top - 1];
      S.L = S.st_l[S.top - 1];
      for (int t = S.top - 2; t >= 0; --t) {
        float4 lo = S.st_o[t];
        float ll = S.st_l[t];
        merge_into(lo, ll, S.acc, S.L);
        S.acc = lo;
        S.L = ll;
      }
    }
    store4(o_out + row * D + c, S.acc);
    if (c == 0) lse_out[row] = S.L;
  }
}

// Grid: enough blocks to cover the rows, at most the resident capacity of
// the device (one wave of persistent blocks).
template <typename K>
int grid_for(K kernel, long long units) {
  int dev = 0, sms = 0, per_sm = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kThreads, 0);
  long long cap = (long long)(sms > 0 ? sms : 1) * (per_sm > 0 ? per_sm : 1);
  return (int)(units < cap ? units : cap);
}

template <int D, typename TO>
usp_status_t launch_d(const float* o, const float* l, int n, long long rows, int tree,
                      TO* oo, float* lo, cudaStream_t st) {
  constexpr int kRPB = kThreads / (D / 4);
  ProfScope ps(st, tree ? "merge_tree" : "merge_linear");
  if (n <= kRegParts) {
    switch (n) {
#define USP_MERGE_CASE(NP)                                                           \
  case NP: {                                                                         \
    constexpr long long rpp = (long long)kRPB * rows_per_thread<NP>();               \
    auto k = merge_reg_kernel<D, NP, TO>;                                            \
    k<<<grid_for(k, (rows + rpp - 1) / rpp), kThreads, 0, st>>>(o, l, rows, tree,    \
                                                               oo, lo);             \
    break;                                                                           \
  }
      USP_MERGE_CASE(1) USP_MERGE_CASE(2) USP_MERGE_CASE(3) USP_MERGE_CASE(4)
      USP_MERGE_CASE(5) USP_MERGE_CASE(6) USP_MERGE_CASE(7) USP_MERGE_CASE(8)
#undef USP_MERGE_CASE
    }
  } else if (!tree) {
    const long long units = (rows + kRPB - 1) / kRPB;
    auto k = merge_linear_kernel<D, TO>;
    k<<<grid_for(k, units), kThreads, 0, st>>>(o, l, n, rows, oo, lo);
  } else {
    const long long units = (rows + kRPB - 1) / kRPB;
    auto k = merge_stack_kernel<D, TO>;
    k<<<grid_for(k, units), kThreads, 0, st>>>(o, l, n, rows, 1, oo, lo);
  }
  note_launch();
  return check_launch();
}

}  // namespace

usp_status_t launch_merge(const float* o_parts, const float* lse_parts, int n,
                          long long rows, int D, int tree, void* o_out,
                          int out_bf16, float* lse_out, cudaStream_t st) {
  if (rows == 0) return USP_OK;
  if (D == 128)
    return out_bf16 ? launch_d<128>(o_parts, lse_parts, n, rows, tree,
                                    reinterpret_cast<__nv_bfloat16*>(o_out), lse_out, st)
                    : launch_d<128>(o_parts, lse_parts, n, rows, tree,
                                    reinterpret_cast<float*>(o_out), lse_out, st);
  return out_bf16 ? launch_d<64>(o_parts, lse_parts, n, rows, tree,
                                 reinterpret_cast<__nv_bfloat16*>(o_out), lse_out, st)
                  : launch_d<64>(o_parts, lse_parts, n, rows, tree,
                                 reinterpret_cast<float*>(o_out), lse_out, st);
}

}  // namespace usp
