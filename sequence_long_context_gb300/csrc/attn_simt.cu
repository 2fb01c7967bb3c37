// CUDA-core attention kernels in fp32 arithmetic (any supported shape).
//
// These serve the fp32 inputs (whose 1e-5 tolerance rules out TF32 tensor
// cores) and every shape the tensor-core kernels do not take, and they are
// the cross-check for the tensor-core kernels. They compute exactly what
// the tensor-core kernels compute, in the same ring order:
//
// Forward ("Long Context Attention" notes, "Ring Attention"): ring rank rho
// owns permuted rows [rho*S/cp, (rho+1)*S/cp); at step s it meets the KV
// shard of rank (rho - s) mod cp. The per-step partial is folded into the
// running partial with the log-sum-exp rule ("Tree Attention":
// associativity), keeping the running partial unnormalised as (m, l, acc).
//
// One warp owns one query row. Keys are taken 32 at a time, one per lane:
// each lane tests its key's visibility and forms its score; the warp then
// folds the 32 scores into (m, l) and the 32 value rows into acc, where lane
// t owns output features [t*D/32, (t+1)*D/32). Groups with no visible key
// are skipped after a ballot.
//
// Backward (gradient of the above; the LSE is kept for it, "Long Context
// Attention" notes, "Motivation"): Delta_i = <dO_i, O_i>;
// dQ rows are formed by one warp per query row over keys in ring order;
// dK/dV rows by one warp per key row over every query rank that sees the
// shard (the shard's ring return) and every query head of its GQA group.
#include <type_traits>

#include "internal.h"

namespace usp {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr int kRowsPerBlock = 4;  // warps per block; one row per warp

template <typename T>
__device__ __forceinline__ const T* row_ptr(const void* base, const AttnParams& P,
                                            int bt, int p, int h, long long tok) {
  // token stride tok elements: H*D dense, 3*H*D in a packed q/k/v tensor
  return reinterpret_cast<const T*>(base) + ((long long)bt * P.S + p) * tok +
         (long long)h * P.D;
}

// <x, y> over D with x a float row in shared memory and y a tensor row.
template <typename T, int D>
__device__ __forceinline__ float dot_row(const float* __restrict__ xs,
                                         const T* __restrict__ y) {
  float acc = 0.f;
#pragma unroll 8
  for (int d = 0; d < D; d += 4) {
    float yv[4];
    load_row<T, 4>(y + d, yv);
    float4 xv = *reinterpret_cast<const float4*>(xs + d);
    acc = fmaf(xv.x, yv[0], acc);
    acc = fmaf(xv.y, yv[1], acc);
    acc = fmaf(xv.z, yv[2], acc);
    acc = fmaf(xv.w, yv[3], acc);
  }
  return acc;
}

template <typename T, int D>
__global__ void __launch_bounds__(kRowsPerBlock * 32)
fwd_simt_kernel(AttnParams P) {
  constexpr int E = D / 32;
  __shared__ __align__(16) float qs[kRowsPerBlock][D];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row = blockIdx.x * kRowsPerBlock + warp;
  const int h = blockIdx.y, bt = blockIdx.z;
  if (row >= P.S) return;
  const int g = h / P.G;
  {
    float x[E];
    load_row<T, E>(row_ptr<T>(P.q, P, bt, row, h, qkv_stride(P, P.Hq)) + lane * E, x);
#pragma unroll
    for (int e = 0; e < E; ++e) qs[warp][lane * E + e] = x[e] * P.scale_log2;
  }
  __syncwarp();
  const int i = nat_pos(P, row);
  const RowMask rm = row_mask(P, i);
  const int rho = row / P.shard;
  float m = -INFINITY, l = 0.f, acc[E];
#pragma unroll
  for (int e = 0; e < E; ++e) acc[e] = 0.f;

  for (int s = 0; s < P.cp; ++s) {
    const int kap = (rho - s + P.cp) % P.cp;
    const int k0 = kap * P.shard, k1 = k0 + P.shard;
    for (int kb = k0; kb < k1; kb += 32) {
      const int kidx = kb + lane;
      const bool vis = kidx < k1 && row_visible(rm, nat_pos(P, kidx));
      const unsigned mask = __ballot_sync(0xffffffffu, vis);
      if (mask == 0u) continue;
      float sc = -INFINITY;
      if (vis) sc = dot_row<T, D>(qs[warp], row_ptr<T>(P.k, P, bt, kidx, g, qkv_stride(P, P.Hkv)));
      const float m_new = fmaxf(m, warp_max(sc));
      const float alpha = exp2f(m - m_new);
      const float pj = vis ? exp2f(sc - m_new) : 0.f;
      l = l * alpha + warp_sum(pj);
#pragma unroll
      for (int e = 0; e < E; ++e) acc[e] *= alpha;
      unsigned mm = mask;
      while (mm) {
        const int t = __ffs(mm) - 1;
        mm &= mm - 1;
        const float pt = __shfl_sync(0xffffffffu, pj, t);
        float vv[E];
        load_row<T, E>(row_ptr<T>(P.v, P, bt, kb + t, g, qkv_stride(P, P.Hkv)) + lane * E, vv);
#pragma unroll
        for (int e = 0; e < E; ++e) acc[e] = fmaf(pt, vv[e], acc[e]);
      }
      m = m_new;
    }
  }
  const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
  for (int e = 0; e < E; ++e) acc[e] *= inv;
  T* orow = const_cast<T*>(row_ptr<T>(P.o, P, bt, row, h, (long long)P.Hq * D)) + lane * E;
  store_row<T, E>(orow, acc);
  if (lane == 0)
    P.lse[lse_index(P, bt, h, row)] = l > 0.f ? (m + log2f(l)) * kLn2 : -INFINITY;
}

// Delta[bt][h][p] = <dO, O> per row (and, for the tensor-core path, the LSE
// in log2 units in the same layout); optionally zeroes the fp32 dQ
// accumulator rows of the same (bt, p, h).
template <typename T, int D>
__global__ void __launch_bounds__(256)
bwd_preprocess_kernel(AttnParams P, int zero_dq) {
  constexpr int E = D / 32;
  const int lane = threadIdx.x & 31;
  const long long nrows = (long long)P.Bt * P.S * P.Hq;
  long long r = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  for (; r < nrows; r += (long long)gridDim.x * 8) {
    // r enumerates [bt][p][h] (the tensor order)
    const int h = (int)(r % P.Hq);
    const long long bp = r / P.Hq;
    const int p = (int)(bp % P.S);
    const int bt = (int)(bp / P.S);
    float o[E], d[E];
    // the caller's natural-order out and dout in place (tensor-core path),
    // else the kernels' own [bt][p][h] rows
    long long src = r;
    if (P.nat) {
      const TensorPos t = tensor_pos(P, h, p, bt, P.Hq);
      src = ((long long)t.b * P.S + t.row) * ((long long)P.ud * P.Hq) + t.h;
    }
    load_row<T, E>(reinterpret_cast<const T*>(P.o) + src * D + lane * E, o);
    load_row<T, E>(reinterpret_cast<const T*>(P.dout) + src * D + lane * E, d);
    float acc = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) acc = fmaf(o[e], d[e], acc);
    acc = warp_sum(acc);
    if (lane == 0) {
      const long long di = ((long long)bt * P.Hq + h) * P.S + p;
      P.delta[di] = acc;
      if (P.lse2 != nullptr) P.lse2[di] = P.lse[lse_index(P, bt, h, p)] * kLog2e;
    }
    if (zero_dq) {
      float z[E];
#pragma unroll
      for (int e = 0; e < E; ++e) z[e] = 0.f;
      store_row<float, E>(P.dq_acc + r * D + lane * E, z);
    }
  }
}

// bf16 rows with 16-byte accesses: D/8 lanes per row (8 elements each), so
// a warp covers 256/D rows per load instruction; the row's lanes reduce the
// dot product among themselves. Same results and outputs as
// bwd_preprocess_kernel.
template <int D>
__global__ void __launch_bounds__(256)
bwd_preprocess_bf16_kernel(AttnParams P, int zero_dq) {
  constexpr int kLanes = D / 8, kRowsPerWarp = 32 / kLanes;
  const int lane = threadIdx.x & 31;
  const int sub = lane % kLanes, grp = lane / kLanes;
  const long long nrows = (long long)P.Bt * P.S * P.Hq;
  const long long stride = (long long)gridDim.x * 8 * kRowsPerWarp;
  for (long long r = ((long long)blockIdx.x * 8 + (threadIdx.x >> 5)) * kRowsPerWarp + grp;
       r - grp < nrows; r += stride) {
    const bool valid = r < nrows;
    const int h = (int)(r % P.Hq);
    const long long bp = r / P.Hq;
    const int p = (int)(bp % P.S), bt = (int)(bp / P.S);
    long long src = r;
    if (P.nat) {
      const TensorPos t = tensor_pos(P, h, p, bt, P.Hq);
      src = ((long long)t.b * P.S + t.row) * ((long long)P.ud * P.Hq) + t.h;
    }
    float acc = 0.f;
    if (valid) {
      const uint4 a = __ldg(reinterpret_cast<const uint4*>(
          reinterpret_cast<const __nv_bfloat16*>(P.o) + src * D) + sub);
      const uint4 b = __ldg(reinterpret_cast<const uint4*>(
          reinterpret_cast<const __nv_bfloat16*>(P.dout) + src * D) + sub);
      const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, bw[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 af = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&aw[e]));
        const float2 bf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&bw[e]));
        acc = fmaf(af.x, bf.x, acc);
        acc = fmaf(af.y, bf.y, acc);
      }
    }
#pragma unroll
    for (int off = kLanes / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (!valid) continue;
    if (sub == 0) {
      const long long di = ((long long)bt * P.Hq + h) * P.S + p;
      P.delta[di] = acc;
      if (P.lse2 != nullptr) P.lse2[di] = P.lse[lse_index(P, bt, h, p)] * kLog2e;
    }
    if (zero_dq) {
      float4* z = reinterpret_cast<float4*>(P.dq_acc + r * D) + 2 * sub;
      z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
      z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
}

template <typename T, int D>
__global__ void __launch_bounds__(kRowsPerBlock * 32)
bwd_dq_simt_kernel(AttnParams P) {
  constexpr int E = D / 32;
  __shared__ __align__(16) float qs[kRowsPerBlock][D];
  __shared__ __align__(16) float ds[kRowsPerBlock][D];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row = blockIdx.x * kRowsPerBlock + warp;
  const int h = blockIdx.y, bt = blockIdx.z;
  if (row >= P.S) return;
  const int g = h / P.G;
  {
    float x[E], y[E];
    load_row<T, E>(row_ptr<T>(P.q, P, bt, row, h, qkv_stride(P, P.Hq)) + lane * E, x);
    load_row<T, E>(row_ptr<T>(P.dout, P, bt, row, h, (long long)P.Hq * D) + lane * E, y);
#pragma unroll
    for (int e = 0; e < E; ++e) {
      qs[warp][lane * E + e] = x[e] * P.scale_log2;
      ds[warp][lane * E + e] = y[e];
    }
  }
  __syncwarp();
  const int i = nat_pos(P, row);
  const RowMask rm = row_mask(P, i);
  const int rho = row / P.shard;
  const float lse2 = P.lse[lse_index(P, bt, h, row)] * kLog2e;
  const float delta = P.delta[((long long)bt * P.Hq + h) * P.S + row];
  float acc[E];
#pragma unroll
  for (int e = 0; e < E; ++e) acc[e] = 0.f;
  for (int s = 0; s < P.cp; ++s) {
    const int kap = (rho - s + P.cp) % P.cp;
    const int k0 = kap * P.shard, k1 = k0 + P.shard;
    for (int kb = k0; kb < k1; kb += 32) {
      const int kidx = kb + lane;
      const bool vis = kidx < k1 && row_visible(rm, nat_pos(P, kidx));
      const unsigned mask = __ballot_sync(0xffffffffu, vis);
      if (mask == 0u) continue;
      float dsj = 0.f;
      if (vis) {
        const float sc = dot_row<T, D>(qs[warp], row_ptr<T>(P.k, P, bt, kidx, g, qkv_stride(P, P.Hkv)));
        const float pj = exp2f(sc - lse2);
        const float dp = dot_row<T, D>(ds[warp], row_ptr<T>(P.v, P, bt, kidx, g, qkv_stride(P, P.Hkv)));
        dsj = pj * (dp - delta);
      }
      unsigned mm = mask;
      while (mm) {
        const int t = __ffs(mm) - 1;
        mm &= mm - 1;
        const float w = __shfl_sync(0xffffffffu, dsj, t);
        float kv[E];
        load_row<T, E>(row_ptr<T>(P.k, P, bt, kb + t, g, qkv_stride(P, P.Hkv)) + lane * E, kv);
#pragma unroll
        for (int e = 0; e < E; ++e) acc[e] = fmaf(w, kv[e], acc[e]);
      }
    }
  }
#pragma unroll
  for (int e = 0; e < E; ++e) acc[e] *= P.scale;
  T* out = reinterpret_cast<T*>(P.dq) + ((long long)bt * P.S + row) * qkv_stride(P, P.Hq) +
           (long long)h * D + lane * E;
  store_row<T, E>(out, acc);
}

template <typename T, int D>
__global__ void __launch_bounds__(kRowsPerBlock * 32)
bwd_dkdv_simt_kernel(AttnParams P) {
  constexpr int E = D / 32;
  __shared__ __align__(16) float ks[kRowsPerBlock][D];
  __shared__ __align__(16) float vs[kRowsPerBlock][D];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int krow = blockIdx.x * kRowsPerBlock + warp;
  const int g = blockIdx.y, bt = blockIdx.z;
  if (krow >= P.S) return;
  {
    float x[E], y[E];
    load_row<T, E>(row_ptr<T>(P.k, P, bt, krow, g, qkv_stride(P, P.Hkv)) + lane * E, x);
    load_row<T, E>(row_ptr<T>(P.v, P, bt, krow, g, qkv_stride(P, P.Hkv)) + lane * E, y);
#pragma unroll
    for (int e = 0; e < E; ++e) {
      ks[warp][lane * E + e] = x[e] * P.scale_log2;
      vs[warp][lane * E + e] = y[e];
    }
  }
  __syncwarp();
  const int j = nat_pos(P, krow);
  const int kap = krow / P.shard;
  float dk[E], dv[E];
#pragma unroll
  for (int e = 0; e < E; ++e) { dk[e] = 0.f; dv[e] = 0.f; }
  for (int hh = 0; hh < P.G; ++hh) {
    const int h = g * P.G + hh;
    // the shard travels the ring: at step s it is on rank kap + s
    for (int s = 0; s < P.cp; ++s) {
      const int rho = (kap + s) % P.cp;
      const int q0 = rho * P.shard, q1 = q0 + P.shard;
      for (int qb = q0; qb < q1; qb += 32) {
        const int qidx = qb + lane;
        bool vis = false;
        if (qidx < q1) {
          const RowMask rm = row_mask(P, nat_pos(P, qidx));
          vis = row_visible(rm, j);
        }
        const unsigned mask = __ballot_sync(0xffffffffu, vis);
        if (mask == 0u) continue;
        float pj = 0.f, dsj = 0.f;
        if (vis) {
          const float sc = dot_row<T, D>(ks[warp], row_ptr<T>(P.q, P, bt, qidx, h, qkv_stride(P, P.Hq)));
          const float lse2 = P.lse[lse_index(P, bt, h, qidx)] * kLog2e;
          pj = exp2f(sc - lse2);
          const float dp = dot_row<T, D>(vs[warp], row_ptr<T>(P.dout, P, bt, qidx, h, (long long)P.Hq * D));
          const float delta = P.delta[((long long)bt * P.Hq + h) * P.S + qidx];
          dsj = pj * (dp - delta);
        }
        unsigned mm = mask;
        while (mm) {
          const int t = __ffs(mm) - 1;
          mm &= mm - 1;
          const float wp = __shfl_sync(0xffffffffu, pj, t);
          const float wd = __shfl_sync(0xffffffffu, dsj, t);
          float qv[E], dov[E];
          load_row<T, E>(row_ptr<T>(P.q, P, bt, qb + t, h, qkv_stride(P, P.Hq)) + lane * E, qv);
          load_row<T, E>(row_ptr<T>(P.dout, P, bt, qb + t, h, (long long)P.Hq * D) + lane * E, dov);
#pragma unroll
          for (int e = 0; e < E; ++e) {
            dk[e] = fmaf(wd, qv[e], dk[e]);
            dv[e] = fmaf(wp, dov[e], dv[e]);
          }
        }
      }
    }
  }
#pragma unroll
  for (int e = 0; e < E; ++e) dk[e] *= P.scale;
  const long long off =
      ((long long)bt * P.S + krow) * qkv_stride(P, P.Hkv) + (long long)g * D + lane * E;
  store_row<T, E>(reinterpret_cast<T*>(P.dk) + off, dk);
  store_row<T, E>(reinterpret_cast<T*>(P.dv) + off, dv);
}

template <typename T, int D>
usp_status_t fwd_t(const AttnParams& P, cudaStream_t st) {
  dim3 grid((P.S + kRowsPerBlock - 1) / kRowsPerBlock, P.Hq, P.Bt);
  {
    ProfScope ps(st, "attn_fwd_simt");
    fwd_simt_kernel<T, D><<<grid, kRowsPerBlock * 32, 0, st>>>(P);
  }
  note_launch();
  return check_launch();
}

template <typename T, int D>
usp_status_t pre_t(const AttnParams& P, int zero, cudaStream_t st) {
  long long rows = (long long)P.Bt * P.S * P.Hq;
  if constexpr (std::is_same<T, __nv_bfloat16>::value) {
    const long long blocks = (rows + 8 * (256 / D) - 1) / (8 * (256 / D));
    const int grid = (int)(blocks < 152LL * 16 ? blocks : 152LL * 16);
    ProfScope ps(st, "attn_bwd_preprocess");
    bwd_preprocess_bf16_kernel<D><<<grid, 256, 0, st>>>(P, zero);
  } else {
    long long blocks = (rows + 7) / 8;
    int grid = (int)(blocks < 152LL * 16 ? blocks : 152LL * 16);
    ProfScope ps(st, "attn_bwd_preprocess");
    bwd_preprocess_kernel<T, D><<<grid, 256, 0, st>>>(P, zero);
  }
  note_launch();
  return check_launch();
}

template <typename T, int D>
usp_status_t bwd_t(const AttnParams& P, cudaStream_t st) {
  dim3 gq((P.S + kRowsPerBlock - 1) / kRowsPerBlock, P.Hq, P.Bt);
  {
    ProfScope ps(st, "attn_bwd_dq_simt");
    bwd_dq_simt_kernel<T, D><<<gq, kRowsPerBlock * 32, 0, st>>>(P);
  }
  note_launch();
  usp_status_t r = check_launch();
  if (r != USP_OK) return r;
  dim3 gk((P.S + kRowsPerBlock - 1) / kRowsPerBlock, P.Hkv, P.Bt);
  {
    ProfScope ps(st, "attn_bwd_dkdv_simt");
    bwd_dkdv_simt_kernel<T, D><<<gk, kRowsPerBlock * 32, 0, st>>>(P);
  }
  note_launch();
  return check_launch();
}

}  // namespace

usp_status_t launch_fwd_simt(const AttnParams& P, int bf16, cudaStream_t st) {
  if (P.S == 0) return USP_OK;
  if (bf16) return P.D == 128 ? fwd_t<__nv_bfloat16, 128>(P, st) : fwd_t<__nv_bfloat16, 64>(P, st);
  return P.D == 128 ? fwd_t<float, 128>(P, st) : fwd_t<float, 64>(P, st);
}

usp_status_t launch_bwd_preprocess(const AttnParams& P, int bf16, int zero,
                                   cudaStream_t st) {
  if (P.S == 0) return USP_OK;
  if (bf16) return P.D == 128 ? pre_t<__nv_bfloat16, 128>(P, zero, st) : pre_t<__nv_bfloat16, 64>(P, zero, st);
  return P.D == 128 ? pre_t<float, 128>(P, zero, st) : pre_t<float, 64>(P, zero, st);
}

usp_status_t launch_bwd_simt(const AttnParams& P, int bf16, cudaStream_t st) {
  if (P.S == 0) return USP_OK;
  if (bf16) return P.D == 128 ? bwd_t<__nv_bfloat16, 128>(P, st) : bwd_t<__nv_bfloat16, 64>(P, st);
  return P.D == 128 ? bwd_t<float, 128>(P, st) : bwd_t<float, 64>(P, st);
}

}  // namespace usp
