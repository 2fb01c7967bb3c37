// Shared device/host definitions of the sequence-parallel attention kernels.
//
// Positions. Kernels index tensors by the permuted ("rank-major") sequence
// index p; the mask is defined on natural positions. nat_pos() maps p to the
// natural position for the three ring layouts:
//   contiguous  rank r holds [r*S/cp, (r+1)*S/cp)            (ring-sliding-
//               window README: chunk i on rank i)
//   zigzag      rank r holds chunk r then chunk 2cp-1-r of 2cp chunks
//               ("Long Context Attention" notes, "Zig-Zag Attention")
//   stripe      rank r holds r, r+cp, r+2cp, ...             (same notes,
//               "Solution": striped permutation)
// Visibility (query natural position i, key natural position j, both in the
// same packed sequence starting at qs):
//   (!causal || j <= i) && (window <= 0 || i - j < window || j - qs < sink)
// and keys outside [qs, qe) are hidden.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace usp {

enum Layout : int { kContiguous = 0, kZigzag = 1, kStripe = 2 };

// Kernel-side view of one attention problem. Tensors seen by the kernels are
// [Bt][S][H][D] contiguous with Bt = ud * B (Ulysses groups outermost, each
// group holding H = heads/ud heads). LSE/Delta are addressed as
//   lse[b * lse_sb + u * lse_su + h * lse_sh + p],  u = bt / B, b = bt % B.
struct AttnParams {
  const void* q;
  const void* k;
  const void* v;
  void* o;          // forward output / backward: saved forward output
  float* lse;       // forward: written; backward: read
  const void* dout; // backward only
  float* delta;     // backward: rowsum(dO * O), [Bt][Hq][S]
  float* lse2;      // backward (tensor-core path): LSE * log2(e), [Bt][Hq][S]
  void* dq;
  void* dk;
  void* dv;
  float* dq_acc;    // backward (tensor-core path): fp32 dQ accumulator
  int* status;      // device status word (USP_ERR_TIMEOUT from waits)

  int Bt, B, S, Hq, Hkv, D, G, ud;
  long long lse_sb, lse_su, lse_sh;
  float scale;       // softmax scale
  float scale_log2;  // scale * log2(e)
  int causal, window, sink;
  const int* cu;     // varlen boundaries [nseq + 1] or nullptr
  int nseq;
  int cp, layout, shard, chunk;
  int unit_batch;    // tensor-core kernels: (batch, head) units per L2 batch
  // elements between consecutive tokens of q, k, v, dq, dk, dv: 0 = dense
  // ([.., H, D] rows of H*D); 3*H*D for a packed [B, S, 3, H, D] tensor
  long long qkv_tok;
  // 1: q, k, v, o, dout, dq, dk, dv are the caller's natural-order tensors
  // [B][S][ud*H][D], read and written in place (tensor-core kernels, layouts
  // whose 128-row tiles are runs of natural positions); 0: the kernels' own
  // rank-major head groups [Bt][S][H][D]
  int nat;
};

// Token stride of q/k/v/dq/dk/dv rows with H heads.
__host__ __device__ __forceinline__ long long qkv_stride(const AttnParams& P, int H) {
  return P.qkv_tok ? P.qkv_tok : (long long)H * P.D;
}

__host__ __device__ __forceinline__ int nat_pos(int p, int layout, int cp,
                                                int shard, int chunk) {
  if (layout == kContiguous) return p;
  int r = p / shard;
  int i = p - r * shard;
  if (layout == kZigzag)
    return i < chunk ? r * chunk + i : (2 * cp - 1 - r) * chunk + (i - chunk);
  return i * cp + r;
}

__device__ __forceinline__ int nat_pos(const AttnParams& P, int p) {
  return nat_pos(p, P.layout, P.cp, P.shard, P.chunk);
}

// Index n with cu[n] <= pos < cu[n+1] (varlen), by binary search. Only
// values of cu are compared; no index leaves [0, nseq].
__device__ __forceinline__ int seg_of(const int* __restrict__ cu, int nseq,
                                      int pos) {
  int lo = 0, hi = nseq - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (__ldg(cu + mid) <= pos) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Per-query mask description: key natural position j is visible iff
//   (j >= lo && j <= hi) || (j >= qs && j < sink_end && j <= causal_hi)
struct RowMask {
  int lo, hi;        // main visible interval (inclusive); lo > hi: empty
  int qs, sink_end;  // sink interval [qs, sink_end)
  int causal_hi;     // last key a sink may be (causal bound or segment end)
};

__device__ __forceinline__ RowMask row_mask(const AttnParams& P, int i) {
  int qs = 0, qe = P.S;
  if (P.cu != nullptr) {
    int n = seg_of(P.cu, P.nseq, i);
    qs = __ldg(P.cu + n);
    qe = __ldg(P.cu + n + 1);
  }
  RowMask m;
  int hi = P.causal ? i : qe - 1;
  int lo = qs;
  if (P.window > 0) lo = max(lo, i - P.window + 1);
  m.lo = lo;
  m.hi = hi;
  m.qs = qs;
  m.sink_end = (P.window > 0) ? min(qs + P.sink, qe) : qs;
  m.causal_hi = hi;
  return m;
}

__device__ __forceinline__ bool row_visible(const RowMask& m, int j) {
  return (j >= m.lo && j <= m.hi) ||
         (j >= m.qs && j < m.sink_end && j <= m.causal_hi);
}

__device__ __forceinline__ float bf16_to_f(__nv_bfloat16 x) {
  return __bfloat162float(x);
}

// Load E consecutive elements (E*sizeof(T) a multiple of 8 bytes) as floats.
template <typename T, int E>
__device__ __forceinline__ void load_row(const T* __restrict__ src, float* dst);

template <>
__device__ __forceinline__ void load_row<float, 4>(const float* __restrict__ s,
                                                   float* d) {
  float4 x = __ldg(reinterpret_cast<const float4*>(s));
  d[0] = x.x; d[1] = x.y; d[2] = x.z; d[3] = x.w;
}
template <>
__device__ __forceinline__ void load_row<float, 2>(const float* __restrict__ s,
                                                   float* d) {
  float2 x = __ldg(reinterpret_cast<const float2*>(s));
  d[0] = x.x; d[1] = x.y;
}
template <>
__device__ __forceinline__ void load_row<__nv_bfloat16, 4>(
    const __nv_bfloat16* __restrict__ s, float* d) {
  uint2 x = __ldg(reinterpret_cast<const uint2*>(s));
  __nv_bfloat162 a = *reinterpret_cast<__nv_bfloat162*>(&x.x);
  __nv_bfloat162 b = *reinterpret_cast<__nv_bfloat162*>(&x.y);
  float2 fa = __bfloat1622float2(a), fb = __bfloat1622float2(b);
  d[0] = fa.x; d[1] = fa.y; d[2] = fb.x; d[3] = fb.y;
}
template <>
__device__ __forceinline__ void load_row<__nv_bfloat16, 2>(
    const __nv_bfloat16* __restrict__ s, float* d) {
  unsigned x = __ldg(reinterpret_cast<const unsigned*>(s));
  __nv_bfloat162 a = *reinterpret_cast<__nv_bfloat162*>(&x);
  float2 fa = __bfloat1622float2(a);
  d[0] = fa.x; d[1] = fa.y;
}

template <typename T, int E>
__device__ __forceinline__ void store_row(T* dst, const float* s);

template <>
__device__ __forceinline__ void store_row<float, 4>(float* d, const float* s) {
  *reinterpret_cast<float4*>(d) = make_float4(s[0], s[1], s[2], s[3]);
}
template <>
__device__ __forceinline__ void store_row<float, 2>(float* d, const float* s) {
  *reinterpret_cast<float2*>(d) = make_float2(s[0], s[1]);
}
template <>
__device__ __forceinline__ void store_row<__nv_bfloat16, 4>(__nv_bfloat16* d,
                                                            const float* s) {
  __nv_bfloat162 a = __floats2bfloat162_rn(s[0], s[1]);
  __nv_bfloat162 b = __floats2bfloat162_rn(s[2], s[3]);
  uint2 x;
  x.x = *reinterpret_cast<unsigned*>(&a);
  x.y = *reinterpret_cast<unsigned*>(&b);
  *reinterpret_cast<uint2*>(d) = x;
}
template <>
__device__ __forceinline__ void store_row<__nv_bfloat16, 2>(__nv_bfloat16* d,
                                                            const float* s) {
  __nv_bfloat162 a = __floats2bfloat162_rn(s[0], s[1]);
  *reinterpret_cast<__nv_bfloat162*>(d) = a;
}

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// Where head h of head group bt (= u*B + b) at rank-major row p sits in a
// q/k/v/o/dout-like tensor with H heads per group: (head, row, batch) of the
// kernels' own layout, or with P.nat of the caller's natural-order tensor
// (global head u*H + h, natural row). A 128-row tile of a contiguous or
// zigzag layout is a run of natural rows, so a tile's first row gives its
// TMA coordinate.
struct TensorPos {
  int h, row, b;
};
__host__ __device__ __forceinline__ TensorPos tensor_pos(const AttnParams& P, int h, int p,
                                                         int bt, int H) {
  if (!P.nat) return {h, p, bt};
  const int u = bt / P.B;
  return {u * H + h, nat_pos(p, P.layout, P.cp, P.shard, P.chunk), bt - u * P.B};
}

__host__ __device__ __forceinline__ long long lse_index(const AttnParams& P,
                                                        int bt, int h, int p) {
  int u = bt / P.B, b = bt - u * P.B;
  return b * P.lse_sb + u * P.lse_su + h * P.lse_sh + p;
}

}  // namespace usp
