// Standalone log-sum-exp merge of n attention partials.
//
// "Long Context Attention" notes, "Tree Attention": logsumexp and max are
// associative, so partial results over disjoint key sets can be reduced in
// any order, e.g. along a tree. For two partials (O_a, L_a), (O_b, L_b):
//   m = max(L_a, L_b), L = m + log(exp(L_a - m) + exp(L_b - m)),
//   O = exp(L_a - L) O_a + exp(L_b - L) O_b;  L = -inf is the identity.
//
// Layout: o_parts [n][rows][D] fp32, lse_parts [n][rows]. One warp merges
// one row: each lane owns D/32 consecutive floats (16 or 8 bytes), so every
// partial row is one coalesced 512/256-byte read. HBM-bound.
//
// Ring order folds left to right. Tree order (pairwise levels, an odd last
// partial carried up unchanged) builds the same tree as a binary counter:
// push each partial, merge the top two while they have equal level, and at
// the end fold the stack from the top down. That needs a stack of at most
// log2(n)+1 entries, held in registers.
#include "internal.h"

namespace usp {
namespace {

constexpr int kWarps = 8;
constexpr int kMaxTreeDepth = 7;  // n <= 64
constexpr int kRegParts = 8;      // up to this many partials merge in registers

template <int E>
__device__ __forceinline__ void merge_into(float* oa, float& la, const float* ob,
                                           float lb) {
  // (oa, la) <- (oa, la) (+) (ob, lb); an empty partial is the identity and
  // its O is never read.
  if (lb == -INFINITY) return;
  if (la == -INFINITY) {
#pragma unroll
    for (int e = 0; e < E; ++e) oa[e] = ob[e];
    la = lb;
    return;
  }
  float m = fmaxf(la, lb);
  float ea = expf(la - m);
  float eb = expf(lb - m);
  float tot = ea + eb;
  float inv = 1.f / tot;
  float wa = ea * inv, wb = eb * inv;
#pragma unroll
  for (int e = 0; e < E; ++e) oa[e] = wa * oa[e] + wb * ob[e];
  la = m + logf(tot);
}

template <int E, typename TO>
__global__ void __launch_bounds__(kWarps * 32)
merge_kernel(const float* __restrict__ o_parts, const float* __restrict__ lse_parts,
             int n, long long rows, int tree, TO* __restrict__ o_out,
             float* __restrict__ lse_out) {
  constexpr int D = E * 32;
  const int lane = threadIdx.x & 31;
  long long row = (long long)blockIdx.x * kWarps + (threadIdx.x >> 5);
  const long long rstride = (long long)gridDim.x * kWarps;
  for (; row < rows; row += rstride) {
    const float* op = o_parts + row * D + lane * E;
    float acc[E];
    float L;
    if (n <= kRegParts) {
      // all partials of the row are loaded at once (n loads in flight) and
      // merged in registers; indices are static after unrolling
      float part[kRegParts][E], pl[kRegParts];
#pragma unroll
      for (int i = 0; i < kRegParts; ++i) {
        if (i < n) {
          load_row<float, E>(op + (long long)i * rows * D, part[i]);
          pl[i] = __ldg(lse_parts + (long long)i * rows + row);
          if (pl[i] == -INFINITY) {
#pragma unroll
            for (int e = 0; e < E; ++e) part[i][e] = 0.f;
          }
        }
      }
      if (!tree) {
#pragma unroll
        for (int i = 1; i < kRegParts; ++i)
          if (i < n) merge_into<E>(part[0], pl[0], part[i], pl[i]);
      } else {
        // pairwise levels: at stride s, slot i absorbs slot i + s; a slot
        // without a partner is carried up unchanged
#pragma unroll
        for (int s = 1; s < kRegParts; s *= 2)
#pragma unroll
          for (int i = 0; i + s < kRegParts; i += 2 * s)
            if (i + s < n) merge_into<E>(part[i], pl[i], part[i + s], pl[i + s]);
      }
#pragma unroll
      for (int e = 0; e < E; ++e) acc[e] = part[0][e];
      L = pl[0];
    } else if (!tree) {
      load_row<float, E>(op, acc);
      L = __ldg(lse_parts + row);
      if (L == -INFINITY) {
#pragma unroll
        for (int e = 0; e < E; ++e) acc[e] = 0.f;
      }
      int i = 1;
      // two partials per iteration keep two row loads in flight
      for (; i + 1 < n; i += 2) {
        float b0[E], b1[E];
        load_row<float, E>(op + (long long)i * rows * D, b0);
        load_row<float, E>(op + (long long)(i + 1) * rows * D, b1);
        float l0 = __ldg(lse_parts + (long long)i * rows + row);
        float l1 = __ldg(lse_parts + (long long)(i + 1) * rows + row);
        merge_into<E>(acc, L, b0, l0);
        merge_into<E>(acc, L, b1, l1);
      }
      for (; i < n; ++i) {
        float b0[E];
        load_row<float, E>(op + (long long)i * rows * D, b0);
        float l0 = __ldg(lse_parts + (long long)i * rows + row);
        merge_into<E>(acc, L, b0, l0);
      }
    } else {
      float st_o[kMaxTreeDepth][E];
      float st_l[kMaxTreeDepth];
      int st_lv[kMaxTreeDepth];
      int top = 0;
      for (int i = 0; i < n; ++i) {
        float cur[E];
        load_row<float, E>(op + (long long)i * rows * D, cur);
        float cl = __ldg(lse_parts + (long long)i * rows + row);
        if (cl == -INFINITY) {
#pragma unroll
          for (int e = 0; e < E; ++e) cur[e] = 0.f;
        }
        int lv = 0;
        while (top > 0 && st_lv[top - 1] == lv) {
          // (stack top) (+) cur, left operand first
          float lo[E];
#pragma unroll
          for (int e = 0; e < E; ++e) lo[e] = st_o[top - 1][e];
          float ll = st_l[top - 1];
          merge_into<E>(lo, ll, cur, cl);
#pragma unroll
          for (int e = 0; e < E; ++e) cur[e] = lo[e];
          cl = ll;
          ++lv;
          --top;
        }
#pragma unroll
        for (int e = 0; e < E; ++e) st_o[top][e] = cur[e];
        st_l[top] = cl;
        st_lv[top] = lv;
        ++top;
      }
      // fold from the top: (s0 + (s1 + (s2 + ...)))
      float cur[E];
#pragma unroll
      for (int e = 0; e < E; ++e) cur[e] = st_o[top - 1][e];
      float cl = st_l[top - 1];
      for (int t = top - 2; t >= 0; --t) {
        float lo[E];
#pragma unroll
        for (int e = 0; e < E; ++e) lo[e] = st_o[t][e];
        float ll = st_l[t];
        merge_into<E>(lo, ll, cur, cl);
#pragma unroll
        for (int e = 0; e < E; ++e) cur[e] = lo[e];
        cl = ll;
      }
#pragma unroll
      for (int e = 0; e < E; ++e) acc[e] = cur[e];
      L = cl;
    }
    store_row<TO, E>(o_out + row * D + lane * E, acc);
    if (lane == 0) lse_out[row] = L;
  }
}

template <int E>
usp_status_t launch_e(const float* o, const float* l, int n, long long rows,
                      int tree, void* oo, int bf16, float* lo, cudaStream_t st) {
  static int sms = 0;
  if (sms == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (sms <= 0) sms = 1;
  }
  long long need = (rows + kWarps - 1) / kWarps;
  long long cap = (long long)sms * 8;
  int grid = (int)(need < cap ? need : cap);
  ProfScope ps(st, tree ? "merge_tree" : "merge_linear");
  if (bf16)
    merge_kernel<E, __nv_bfloat16><<<grid, kWarps * 32, 0, st>>>(
        o, l, n, rows, tree, reinterpret_cast<__nv_bfloat16*>(oo), lo);
  else
    merge_kernel<E, float><<<grid, kWarps * 32, 0, st>>>(
        o, l, n, rows, tree, reinterpret_cast<float*>(oo), lo);
  note_launch();
  return check_launch();
}

}  // namespace

usp_status_t launch_merge(const float* o_parts, const float* lse_parts, int n,
                          long long rows, int D, int tree, void* o_out,
                          int out_bf16, float* lse_out, cudaStream_t st) {
  if (rows == 0) return USP_OK;
  if (D == 128)
    return launch_e<4>(o_parts, lse_parts, n, rows, tree, o_out, out_bf16,
                       lse_out, st);
  return launch_e<2>(o_parts, lse_parts, n, rows, tree, o_out, out_bf16,
                     lse_out, st);
}

}  // namespace usp
