// C ABI entry points: argument validation, workspace carving, dispatch.
//
// Every check happens on the host before any launch, so a call that returns
// an error has enqueued nothing. The library allocates no device memory;
// scratch is carved out of the caller's workspace in 256-byte aligned slices.
#include <atomic>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <map>
#include <string>
#include <vector>

#include "internal.h"

namespace usp {

static std::atomic<unsigned long long> g_launches{0};

namespace {
struct ProfRec {
  const char* name;
  cudaEvent_t a, b;
};
bool g_prof_on = false;
std::vector<ProfRec> g_prof_recs;
std::vector<cudaEvent_t> g_prof_pool;

cudaEvent_t prof_event() {
  if (!g_prof_pool.empty()) {
    cudaEvent_t e = g_prof_pool.back();
    g_prof_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}
}  // namespace

ProfScope::ProfScope(cudaStream_t s, const char* name) : idx(-1), st(s) {
  if (!g_prof_on) return;
  ProfRec r{name, prof_event(), prof_event()};
  if (!r.a || !r.b) return;
  cudaEventRecord(r.a, st);
  g_prof_recs.push_back(r);
  idx = (int)g_prof_recs.size() - 1;
}

ProfScope::~ProfScope() {
  if (idx >= 0) cudaEventRecord(g_prof_recs[idx].b, st);
}

void note_launch(int n) { g_launches.fetch_add((unsigned long long)n); }

int sm_count() {
  constexpr int kMaxDevices = 64;
  static std::atomic<int> cache[kMaxDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 1;
  if (dev < kMaxDevices) {
    const int c = cache[dev].load(std::memory_order_relaxed);
    if (c > 0) return c;
  }
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    n = 1;
  if (dev < kMaxDevices) cache[dev].store(n, std::memory_order_relaxed);
  return n;
}

static thread_local char g_detail[256] = "";

usp_status_t fail_cuda_msg(const char* where, const char* msg) {
  std::snprintf(g_detail, sizeof(g_detail), "%s: %s", where, msg);
  return USP_ERR_CUDA;
}

void set_error_detail(const char* msg) {
  std::snprintf(g_detail, sizeof(g_detail), "%s", msg);
}

usp_status_t fail_cuda(const char* where, cudaError_t e) {
  return fail_cuda_msg(where, cudaGetErrorString(e));
}

usp_status_t check_launch() {
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? USP_OK : fail_cuda("kernel launch", e);
}

namespace {

constexpr size_t kAlign = 256;

size_t round_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

bool aligned16(const void* p) {
  return (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}

struct Shape {
  int B, S, Hq, Hkv, D, cp, ud, layout, dtype, varlen;
  // USP_FLAG_NATURAL_ORDER: the caller's q, k, v, out, dout, dq, dk, dv are
  // in natural sequence order (the kernels' copies in the workspace are
  // rank-major)
  int natural = 0;
  // the kernels need workspace copies of the caller's tensors
  bool staged() const { return ud > 1 || natural; }
  size_t elem() const { return dtype == USP_FP32 ? 4 : 2; }
  size_t q_bytes() const { return (size_t)B_eff() * S * Hq * D * elem(); }
  size_t kv_bytes() const { return (size_t)B_eff() * S * Hkv * D * elem(); }
  int B_eff() const { return varlen ? 1 : B; }
};

usp_status_t validate(const Shape& s, int window, int sink) {
  if (s.B < 0 || s.S < 0 || s.Hq <= 0 || s.Hkv <= 0) return USP_ERR_INVALID_ARG;
  if (s.varlen && s.B < 1) return USP_ERR_INVALID_ARG;
  if (s.D != 64 && s.D != 128) return USP_ERR_UNSUPPORTED;
  if (s.Hq % s.Hkv != 0) return USP_ERR_INVALID_ARG;
  if (s.cp < 1 || s.ud < 1) return USP_ERR_INVALID_ARG;
  if (s.Hq % s.ud != 0 || s.Hkv % s.ud != 0) return USP_ERR_INVALID_ARG;
  if (s.layout < USP_LAYOUT_CONTIGUOUS || s.layout > USP_LAYOUT_STRIPE)
    return USP_ERR_INVALID_ARG;
  if (s.dtype != USP_BF16 && s.dtype != USP_FP32) return USP_ERR_INVALID_ARG;
  int div = s.cp * s.ud * (s.layout == USP_LAYOUT_ZIGZAG ? 2 : 1);
  if (s.S % div != 0) return USP_ERR_INVALID_ARG;
  if (sink < 0) return USP_ERR_INVALID_ARG;
  (void)window;
  // 32-bit element offsets inside the copy kernels and grid limits
  if ((double)s.B_eff() * s.S * s.Hq * s.D >= 2147483647.0 * 8.0)
    return USP_ERR_UNSUPPORTED;
  if ((long long)s.B_eff() * s.ud > 65535 || s.Hq > 65535)
    return USP_ERR_UNSUPPORTED;
  return USP_OK;
}

AttnParams make_params(const Shape& s, float scale, int causal, int window,
                       int sink, const int32_t* cu) {
  AttnParams P{};
  P.B = s.B_eff();
  P.ud = s.ud;
  P.Bt = P.B * s.ud;
  P.S = s.S;
  P.Hq = s.Hq / s.ud;
  P.Hkv = s.Hkv / s.ud;
  P.D = s.D;
  P.G = s.Hq / s.Hkv;
  // LSE [B][Hq_total][S]: u-th group's head h is global head u*Hq/ud + h
  P.lse_sh = s.S;
  P.lse_su = (long long)P.Hq * s.S;
  P.lse_sb = (long long)s.Hq * s.S;
  P.scale = scale > 0.f ? scale : 1.0f / std::sqrt((float)s.D);
  P.scale_log2 = P.scale * 1.4426950408889634f;
  P.causal = causal ? 1 : 0;
  P.window = window > 0 ? window : 0;
  P.sink = sink;
  P.cu = cu;
  P.nseq = cu ? s.B : 0;
  P.cp = s.cp;
  P.layout = s.layout;
  P.shard = s.S / s.cp;
  P.chunk = s.layout == USP_LAYOUT_ZIGZAG ? s.S / (2 * s.cp) : P.shard;
  return P;
}

struct Carve {
  char* base;
  size_t used = 0;
  explicit Carve(void* b) : base(static_cast<char*>(b)) {}
  void* take(size_t bytes) {
    void* p = base ? base + used : nullptr;
    used += round_up(bytes);
    return p;
  }
};

// Workspace slices, in order. Only the sizes matter when base == nullptr.
struct FwdWs {
  void *q, *k, *v, *o;
};
FwdWs carve_fwd(Carve& c, const Shape& s) {
  FwdWs w{};
  if (s.staged()) {
    w.q = c.take(s.q_bytes());
    w.k = c.take(s.kv_bytes());
    w.v = c.take(s.kv_bytes());
    w.o = c.take(s.q_bytes());
  }
  return w;
}

struct BwdWs {
  float* delta;
  float* lse2;
  float* dq_acc;
  void *q, *k, *v, *o, *dout, *dq, *dk, *dv;
};
// The head-sharded q, k, v, o come first, at carve_fwd's offsets, so that a
// forward's workspace handed to the backward (USP_FLAG_SAVED_EXCHANGE) still
// holds them where the backward reads them.
BwdWs carve_bwd(Carve& c, const Shape& s, bool tc) {
  BwdWs w{};
  if (s.staged()) {
    w.q = c.take(s.q_bytes());
    w.k = c.take(s.kv_bytes());
    w.v = c.take(s.kv_bytes());
    w.o = c.take(s.q_bytes());
  }
  w.delta = static_cast<float*>(c.take((size_t)s.B_eff() * s.Hq * s.S * 4));
  if (tc) {
    w.lse2 = static_cast<float*>(c.take((size_t)s.B_eff() * s.Hq * s.S * 4));
    w.dq_acc = static_cast<float*>(c.take((size_t)s.B_eff() * s.S * s.Hq * s.D * 4));
  }
  if (s.staged()) {
    w.dout = c.take(s.q_bytes());
    w.dq = c.take(s.q_bytes());
    w.dk = c.take(s.kv_bytes());
    w.dv = c.take(s.kv_bytes());
  }
  return w;
}

Shape shape_of(int B, int S, int Hq, int Hkv, int D, int cp, int ud,
               int layout, int dtype, int varlen) {
  Shape s{B, S, Hq, Hkv, D, cp, ud, layout, dtype, varlen};
  return s;
}

// Parameters of a natural-order call run in place: every head of the
// caller's tensors is attended as it stands. Attention is per head, so the
// Ulysses head groups (a batch view of the exchanged tensors) are not
// formed: one group of all heads, whose [B][S][H][D] tensors differ from the
// kernels' own layout only by the order of their rows.
AttnParams inplace_params(const Shape& s, float scale, int causal, int window, int sink,
                          const int32_t* cu) {
  Shape one = s;
  one.ud = 1;
  AttnParams P = make_params(one, scale, causal, window, sink, cu);
  P.nat = 1;
  return P;
}

// Natural-order calls read and write the caller's tensors in place where a
// 128-row tile is a run of natural rows (contiguous, zigzag) and the problem
// is short per token: the kernels take 1-4 % longer on the caller's tensors
// than on rank-major copies, which pays while the copies (linear in the
// sequence) cost more than that share of the attention (quadratic): windows,
// packed batches (sequences of at most a few 10K tokens) and dense
// sequences up to 16K tokens (measured: S=8K in place saves 0.07 ms of
// 1.9, S=32K loses 0.15 ms of 26.5). The rule depends only on the call's
// arguments, so forward and backward decide alike.
bool natural_in_place(const Shape& s, int window, const int32_t* cu, long long tok) {
  if (!s.natural || s.layout == USP_LAYOUT_STRIPE || tok != 0) return false;
  return window > 0 || cu != nullptr || s.S <= 16384;
}

bool use_tc_fwd(const AttnParams& P, const Shape& s, unsigned flags) {
  return s.dtype == USP_BF16 && !(flags & USP_FLAG_FORCE_SIMT) &&
         fwd_tc_supported(P);
}
bool use_tc_bwd(const AttnParams& P, const Shape& s, unsigned flags) {
  return s.dtype == USP_BF16 && !(flags & USP_FLAG_FORCE_SIMT) &&
         bwd_tc_supported(P);
}

// Ulysses exchange of one [B,S,H,D] tensor (row = H*D*elem bytes).
// tok: elements between tokens of the flat side (0: dense H*D; 3*H*D when
// the flat side is one of q/k/v (or dq/dk/dv) inside a packed tensor).
usp_status_t a2a(const void* src, void* dst, const Shape& s, int H, int s2h,
                 cudaStream_t st, long long tok = 0) {
  return launch_ulysses(src, dst, s.B_eff(), s.S, (int)(H * s.D * s.elem()),
                        s.ud, s2h, st, (int)(tok * s.elem()), 0,
                        s.natural ? s.layout : -1, s.cp);
}

// Into the kernels' rank-major copy (to_kernel) or back out of it, for one
// [B,S,H,D] tensor of the caller: the Ulysses exchange when ud > 1 (with the
// layout's extract / restore fused in for natural-order tensors), else the
// layout's extract / restore alone.
usp_status_t stage(const void* src, void* dst, const Shape& s, int H, int to_kernel,
                   cudaStream_t st) {
  if (s.ud > 1) return a2a(src, dst, s, H, to_kernel, st);
  return launch_permute_layout(src, dst, s.B_eff(), s.S, (int)(H * s.D * s.elem()), s.layout,
                               s.cp, to_kernel ? 0 : 1, st);
}

}  // namespace
}  // namespace usp

using namespace usp;

extern "C" {

usp_status_t usp_check_cu_seqlens(const int32_t* cu, int nseq, int total) {
  if (cu == nullptr || nseq < 1 || total < 0) return USP_ERR_INVALID_ARG;
  char msg[96];
  if (cu[0] != 0) {
    std::snprintf(msg, sizeof(msg), "cu_seqlens[0] = %d, not 0", (int)cu[0]);
    set_error_detail(msg);
    return USP_ERR_INVALID_ARG;
  }
  for (int i = 0; i < nseq; ++i)
    if (cu[i + 1] < cu[i]) {
      std::snprintf(msg, sizeof(msg), "cu_seqlens[%d] = %d < cu_seqlens[%d] = %d", i + 1,
                    (int)cu[i + 1], i, (int)cu[i]);
      set_error_detail(msg);
      return USP_ERR_INVALID_ARG;
    }
  if (cu[nseq] != total) {
    std::snprintf(msg, sizeof(msg), "cu_seqlens[%d] = %d, not the %d tokens", nseq,
                  (int)cu[nseq], total);
    set_error_detail(msg);
    return USP_ERR_INVALID_ARG;
  }
  return USP_OK;
}

const char* usp_status_string(usp_status_t st) {
  switch (st) {
    case USP_OK: return "USP_OK";
    case USP_ERR_INVALID_ARG: return "USP_ERR_INVALID_ARG";
    case USP_ERR_UNSUPPORTED: return "USP_ERR_UNSUPPORTED";
    case USP_ERR_ALIGNMENT: return "USP_ERR_ALIGNMENT";
    case USP_ERR_WORKSPACE: return "USP_ERR_WORKSPACE";
    case USP_ERR_CUDA: return "USP_ERR_CUDA";
    case USP_ERR_TIMEOUT: return "USP_ERR_TIMEOUT";
  }
  return "USP_ERR_UNKNOWN";
}

uint64_t usp_launch_count(void) { return g_launches.load(); }

const char* usp_last_error_detail(void) { return g_detail; }

usp_status_t usp_device_status(void) {
  if (cudaDeviceSynchronize() != cudaSuccess) return USP_ERR_CUDA;
  const int words[5] = {read_clear_fwd_tc_status(), read_clear_bwd_tc_status(),
                        read_clear_decode_status(), read_clear_selftest_status(),
                        read_clear_fwd_fp8_status()};
  for (int w : words)
    if (w < 0) return USP_ERR_CUDA;
  for (int w : words)
    if (w == USP_ERR_TIMEOUT) return USP_ERR_TIMEOUT;
  for (int w : words)
    if (w != 0) return USP_ERR_CUDA;
  return USP_OK;
}

usp_status_t usp_selftest_wait_timeout(unsigned limit_us, usp_stream_t stream) {
  if (limit_us < 1 || limit_us > 1000000) return USP_ERR_INVALID_ARG;
  return launch_selftest_wait_timeout(limit_us, reinterpret_cast<cudaStream_t>(stream));
}

usp_status_t usp_profile_enable(int on) {
  g_prof_on = on != 0;
  return USP_OK;
}

int usp_profile_read(usp_kernel_stat_t* stats, int max_stats) {
  std::map<std::string, std::pair<uint64_t, double>> agg;
  int rc = 0;
  for (ProfRec& r : g_prof_recs) {
    float ms = 0.f;
    if (cudaEventSynchronize(r.b) != cudaSuccess ||
        cudaEventElapsedTime(&ms, r.a, r.b) != cudaSuccess)
      rc = -1;
    auto& e = agg[r.name];
    e.first += 1;
    e.second += ms;
    g_prof_pool.push_back(r.a);
    g_prof_pool.push_back(r.b);
  }
  g_prof_recs.clear();
  if (rc < 0) return rc;
  int n = 0;
  for (auto& kv : agg) {
    if (n >= max_stats || !stats) break;
    std::memset(stats[n].name, 0, sizeof(stats[n].name));
    std::strncpy(stats[n].name, kv.first.c_str(), sizeof(stats[n].name) - 1);
    stats[n].launches = kv.second.first;
    stats[n].total_ms = kv.second.second;
    ++n;
  }
  return n;
}

size_t usp_attn_fwd_workspace_size(int B, int S, int Hq, int Hkv, int D,
                                   int cp, int ud, usp_dtype_t dtype,
                                   unsigned flags) {
  Shape s = shape_of(B, S, Hq, Hkv, D, cp, ud, 0, dtype, 0);
  s.natural = (flags & USP_FLAG_NATURAL_ORDER) != 0;
  Carve c(nullptr);
  carve_fwd(c, s);
  return c.used;
}

size_t usp_attn_bwd_workspace_size(int B, int S, int Hq, int Hkv, int D,
                                   int cp, int ud, usp_dtype_t dtype,
                                   unsigned flags) {
  Shape s = shape_of(B, S, Hq, Hkv, D, cp, ud, 0, dtype, 0);
  s.natural = (flags & USP_FLAG_NATURAL_ORDER) != 0;
  Carve c(nullptr);
  bool tc = dtype == USP_BF16 && !(flags & USP_FLAG_FORCE_SIMT);
  carve_bwd(c, s, tc);
  return c.used;
}

namespace {
// tok: elements between tokens of q, k, v (0: dense; 3*Hq*D when they are
// the three parts of one packed tensor)
usp_status_t attn_fwd_impl(const void* q, const void* k, const void* v,
                           void* out, float* lse, int B, int S, int Hq, int Hkv,
                           int D, float softmax_scale, int causal, int window,
                           int sink_tokens, const int32_t* cu_seqlens,
                           int cp_size, int ulysses_degree, usp_layout_t layout,
                           usp_dtype_t dtype, unsigned flags, void* workspace,
                           size_t workspace_bytes, usp_stream_t stream, long long tok) {
  Shape s = shape_of(B, S, Hq, Hkv, D, cp_size, ulysses_degree, layout, dtype,
                     cu_seqlens != nullptr);
  s.natural = (flags & USP_FLAG_NATURAL_ORDER) != 0;
  usp_status_t r = validate(s, window, sink_tokens);
  if (r != USP_OK) return r;
  if (s.natural && tok != 0) return USP_ERR_UNSUPPORTED;  // packed q/k/v
  if (S > 0 && (!q || !k || !v || !out || !lse)) return USP_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) ||
      !aligned16(lse) || !aligned16(workspace))
    return USP_ERR_ALIGNMENT;
  if (s.B_eff() == 0 || S == 0) return USP_OK;
  Carve c(workspace);
  FwdWs w = carve_fwd(c, s);
  if (c.used > 0 && (!workspace || workspace_bytes < c.used))
    return USP_ERR_WORKSPACE;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  AttnParams P = make_params(s, softmax_scale, causal, window, sink_tokens,
                             cu_seqlens);
  // natural-order tensors read and written in place by the tensor-core
  // kernel (its 128-row tiles are runs of natural rows except for stripe)
  const bool inplace = natural_in_place(s, window, cu_seqlens, tok) && use_tc_fwd(P, s, flags);
  if (inplace) {
    P = inplace_params(s, softmax_scale, causal, window, sink_tokens, cu_seqlens);
    P.q = q; P.k = k; P.v = v; P.o = out;
  } else if (s.ud > 1 && !s.natural) {
    if ((r = a2a(q, w.q, s, Hq, 1, st, tok)) != USP_OK) return r;
    if ((r = a2a(k, w.k, s, Hkv, 1, st, tok)) != USP_OK) return r;
    if ((r = a2a(v, w.v, s, Hkv, 1, st, tok)) != USP_OK) return r;
    P.q = w.q; P.k = w.k; P.v = w.v; P.o = w.o;  // dense head groups
  } else if (s.staged()) {
    if ((r = stage(q, w.q, s, Hq, 1, st)) != USP_OK) return r;
    if ((r = stage(k, w.k, s, Hkv, 1, st)) != USP_OK) return r;
    if ((r = stage(v, w.v, s, Hkv, 1, st)) != USP_OK) return r;
    P.q = w.q; P.k = w.k; P.v = w.v; P.o = w.o;
  } else {
    P.q = q; P.k = k; P.v = v; P.o = out;
    P.qkv_tok = tok;
  }
  P.lse = lse;
  if (use_tc_fwd(P, s, flags))
    r = launch_fwd_tc(P, st);
  else
    r = launch_fwd_simt(P, dtype == USP_BF16, st);
  if (r != USP_OK) return r;
  if (s.staged() && !inplace) r = stage(w.o, out, s, Hq, 0, st);
  return r;
}

}  // namespace

usp_status_t usp_attn_fwd(const void* q, const void* k, const void* v,
                          void* out, float* lse, int B, int S, int Hq, int Hkv,
                          int D, float softmax_scale, int causal, int window,
                          int sink_tokens, const int32_t* cu_seqlens,
                          int cp_size, int ulysses_degree, usp_layout_t layout,
                          usp_dtype_t dtype, unsigned flags, void* workspace,
                          size_t workspace_bytes, usp_stream_t stream) {
  return attn_fwd_impl(q, k, v, out, lse, B, S, Hq, Hkv, D, softmax_scale, causal, window,
                       sink_tokens, cu_seqlens, cp_size, ulysses_degree, layout, dtype, flags,
                       workspace, workspace_bytes, stream, 0);
}

usp_status_t usp_attn_fwd_qkvpacked(const void* qkv, void* out, float* lse, int B, int S,
                                    int H, int D, float softmax_scale, int causal, int window,
                                    int sink_tokens, const int32_t* cu_seqlens, int cp_size,
                                    int ulysses_degree, usp_layout_t layout, usp_dtype_t dtype,
                                    unsigned flags, void* workspace, size_t workspace_bytes,
                                    usp_stream_t stream) {
  if (H < 1 || D < 1) return USP_ERR_INVALID_ARG;
  const size_t part = (size_t)H * D * (dtype == USP_FP32 ? 4 : 2);
  const char* base = static_cast<const char*>(qkv);
  return attn_fwd_impl(qkv, base ? base + part : nullptr, base ? base + 2 * part : nullptr, out,
                       lse, B, S, H, H, D, softmax_scale, causal, window, sink_tokens,
                       cu_seqlens, cp_size, ulysses_degree, layout, dtype, flags, workspace,
                       workspace_bytes, stream, 3LL * H * D);
}

namespace {
// tok: elements between tokens of q, k, v and dq, dk, dv (0: dense; 3*Hq*D
// for packed tensors)
usp_status_t attn_bwd_impl(const void* q, const void* k, const void* v,
                          const void* out, const float* lse, const void* dout,
                          void* dq, void* dk, void* dv, int B, int S, int Hq,
                          int Hkv, int D, float softmax_scale, int causal,
                          int window, int sink_tokens,
                          const int32_t* cu_seqlens, int cp_size,
                          int ulysses_degree, usp_layout_t layout,
                          usp_dtype_t dtype, unsigned flags, void* workspace,
                          size_t workspace_bytes, usp_stream_t stream, long long tok) {
  Shape s = shape_of(B, S, Hq, Hkv, D, cp_size, ulysses_degree, layout, dtype,
                     cu_seqlens != nullptr);
  s.natural = (flags & USP_FLAG_NATURAL_ORDER) != 0;
  usp_status_t r = validate(s, window, sink_tokens);
  if (r != USP_OK) return r;
  if (s.natural && tok != 0) return USP_ERR_UNSUPPORTED;  // packed q/k/v
  // saved: the workspace holds the forward's copies of q, k, v, out (head
  // groups, or rank-major copies of natural-order tensors)
  const bool saved = (flags & USP_FLAG_SAVED_EXCHANGE) && s.staged();
  // natural-order calls may read q, k, v, out in place, so they always need them
  const bool need_qkvo = !saved || s.natural;
  if (S > 0 && (!lse || !dout || !dq || !dk || !dv || (need_qkvo && (!q || !k || !v || !out))))
    return USP_ERR_INVALID_ARG;
  const void* ptrs[] = {q, k, v, out, lse, dout, dq, dk, dv, workspace};
  for (const void* p : ptrs)
    if (!aligned16(p)) return USP_ERR_ALIGNMENT;
  if (s.B_eff() == 0 || S == 0) return USP_OK;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  AttnParams P = make_params(s, softmax_scale, causal, window, sink_tokens,
                             cu_seqlens);
  const bool tc = use_tc_bwd(P, s, flags);
  Carve c(workspace);
  BwdWs w = carve_bwd(c, s, tc);
  if (!workspace || workspace_bytes < c.used) return USP_ERR_WORKSPACE;
  const bool inplace = natural_in_place(s, window, cu_seqlens, tok) && tc;
  if (inplace) {
    P = inplace_params(s, softmax_scale, causal, window, sink_tokens, cu_seqlens);
    P.q = q; P.k = k; P.v = v; P.o = const_cast<void*>(out); P.dout = dout;
    P.dq = dq; P.dk = dk; P.dv = dv;
  } else if (s.staged()) {
    if (!saved) {
      if (s.natural) {
        if ((r = stage(q, w.q, s, Hq, 1, st)) != USP_OK) return r;
        if ((r = stage(k, w.k, s, Hkv, 1, st)) != USP_OK) return r;
        if ((r = stage(v, w.v, s, Hkv, 1, st)) != USP_OK) return r;
      } else {
        if ((r = a2a(q, w.q, s, Hq, 1, st, tok)) != USP_OK) return r;
        if ((r = a2a(k, w.k, s, Hkv, 1, st, tok)) != USP_OK) return r;
        if ((r = a2a(v, w.v, s, Hkv, 1, st, tok)) != USP_OK) return r;
      }
      if ((r = stage(out, w.o, s, Hq, 1, st)) != USP_OK) return r;
    }
    if ((r = stage(dout, w.dout, s, Hq, 1, st)) != USP_OK) return r;
    P.q = w.q; P.k = w.k; P.v = w.v; P.o = w.o; P.dout = w.dout;
    P.dq = w.dq; P.dk = w.dk; P.dv = w.dv;
  } else {
    P.q = q; P.k = k; P.v = v; P.o = const_cast<void*>(out); P.dout = dout;
    P.dq = dq; P.dk = dk; P.dv = dv;
    P.qkv_tok = tok;
  }
  P.lse = const_cast<float*>(lse);
  P.delta = w.delta;
  P.lse2 = w.lse2;
  P.dq_acc = w.dq_acc;
  if ((r = launch_bwd_preprocess(P, dtype == USP_BF16, tc ? 1 : 0, st)) != USP_OK)
    return r;
  if (tc)
    r = launch_bwd_tc(P, st);
  else
    r = launch_bwd_simt(P, dtype == USP_BF16, st);
  if (r != USP_OK) return r;
  if (inplace) return USP_OK;
  if (s.ud > 1 && !s.natural) {
    if ((r = a2a(w.dq, dq, s, Hq, 0, st, tok)) != USP_OK) return r;
    if ((r = a2a(w.dk, dk, s, Hkv, 0, st, tok)) != USP_OK) return r;
    if ((r = a2a(w.dv, dv, s, Hkv, 0, st, tok)) != USP_OK) return r;
  } else if (s.staged()) {
    if ((r = stage(w.dq, dq, s, Hq, 0, st)) != USP_OK) return r;
    if ((r = stage(w.dk, dk, s, Hkv, 0, st)) != USP_OK) return r;
    if ((r = stage(w.dv, dv, s, Hkv, 0, st)) != USP_OK) return r;
  }
  return USP_OK;
}

}  // namespace

usp_status_t usp_attn_bwd(const void* q, const void* k, const void* v,
                          const void* out, const float* lse, const void* dout,
                          void* dq, void* dk, void* dv, int B, int S, int Hq,
                          int Hkv, int D, float softmax_scale, int causal,
                          int window, int sink_tokens,
                          const int32_t* cu_seqlens, int cp_size,
                          int ulysses_degree, usp_layout_t layout,
                          usp_dtype_t dtype, unsigned flags, void* workspace,
                          size_t workspace_bytes, usp_stream_t stream) {
  return attn_bwd_impl(q, k, v, out, lse, dout, dq, dk, dv, B, S, Hq, Hkv, D, softmax_scale, causal, window, sink_tokens, cu_seqlens, cp_size, ulysses_degree, layout, dtype, flags, workspace, workspace_bytes, stream, 0);
}

usp_status_t usp_attn_bwd_qkvpacked(const void* qkv, const void* out, const float* lse,
                                    const void* dout, void* dqkv, int B, int S, int H, int D,
                                    float softmax_scale, int causal, int window,
                                    int sink_tokens, const int32_t* cu_seqlens, int cp_size,
                                    int ulysses_degree, usp_layout_t layout, usp_dtype_t dtype,
                                    unsigned flags, void* workspace, size_t workspace_bytes,
                                    usp_stream_t stream) {
  if (H < 1 || D < 1) return USP_ERR_INVALID_ARG;
  const size_t part = (size_t)H * D * (dtype == USP_FP32 ? 4 : 2);
  const char* in = static_cast<const char*>(qkv);
  char* g = static_cast<char*>(dqkv);
  return attn_bwd_impl(qkv, in ? in + part : nullptr, in ? in + 2 * part : nullptr, out, lse,
                       dout, dqkv, g ? g + part : nullptr, g ? g + 2 * part : nullptr, B, S, H,
                       H, D, softmax_scale, causal, window, sink_tokens, cu_seqlens, cp_size,
                       ulysses_degree, layout, dtype, flags, workspace, workspace_bytes, stream,
                       3LL * H * D);
}

// Decode workspace: the partials [n_part][rows][D] fp32 and [n_part][rows].
struct DecodeWs {
  float* o_part;
  float* lse_part;
};
DecodeWs carve_decode(Carve& c, long long rows, int D, int n_part) {
  DecodeWs w{};
  w.o_part = static_cast<float*>(c.take((size_t)n_part * rows * D * 4));
  w.lse_part = static_cast<float*>(c.take((size_t)n_part * rows * 4));
  return w;
}

size_t usp_attn_decode_workspace_size(int B, int Tq, int S, int Hq, int Hkv, int D,
                                      int cp_size, int splits_per_shard) {
  (void)S;
  (void)Hkv;
  if (B < 0 || Tq < 1 || Hq < 1 || D < 1 || cp_size < 1 || splits_per_shard < 1) return 0;
  Carve c(nullptr);
  carve_decode(c, (long long)B * Tq * Hq, D, cp_size * splits_per_shard);
  return c.used;
}

usp_status_t usp_attn_decode(const void* q, const void* k, const void* v, void* out,
                             float* lse, int B, int Tq, int S, int Hq, int Hkv, int D,
                             float softmax_scale, int causal, int cp_size,
                             int splits_per_shard, int tree_order, usp_dtype_t dtype,
                             void* workspace, size_t workspace_bytes, usp_stream_t stream) {
  if (B < 0 || Tq < 1 || S < Tq || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || cp_size < 1 ||
      splits_per_shard < 1)
    return USP_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return USP_ERR_INVALID_ARG;
  if (dtype == USP_FP32) return USP_ERR_UNSUPPORTED;
  if (dtype != USP_BF16) return USP_ERR_INVALID_ARG;
  if ((Hq / Hkv) * Tq > decode_max_rows()) return USP_ERR_UNSUPPORTED;
  const long long n_part = (long long)cp_size * splits_per_shard;
  if (S % n_part != 0 || (S / n_part) % decode_keys_per_tile() != 0)
    return USP_ERR_INVALID_ARG;
  if (tree_order && n_part > 64) return USP_ERR_INVALID_ARG;
  if (B > 65535 || n_part > 65535) return USP_ERR_UNSUPPORTED;  // grid z and y
  if (B > 0 && (!q || !k || !v || !out || !lse)) return USP_ERR_INVALID_ARG;
  const void* ptrs[] = {q, k, v, out, lse, workspace};
  for (const void* p : ptrs)
    if (!aligned16(p)) return USP_ERR_ALIGNMENT;
  if (B == 0) return USP_OK;
  const long long rows = (long long)B * Tq * Hq;
  Carve c(workspace);
  DecodeWs w = carve_decode(c, rows, D, (int)n_part);
  if (!workspace || workspace_bytes < c.used) return USP_ERR_WORKSPACE;
  const float scale = softmax_scale > 0.f ? softmax_scale : 1.f / std::sqrt((float)D);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  usp_status_t r = launch_decode_split(q, k, v, w.o_part, w.lse_part, B, Tq, S, Hq, Hkv, D,
                                       scale, causal ? 1 : 0, (int)n_part, st);
  if (r != USP_OK) return r;
  return launch_merge(w.o_part, w.lse_part, (int)n_part, rows, D, tree_order ? 1 : 0, out, 1,
                      lse, st);
}

namespace {
// fp8 forward scratch: the transposed values, then (Ulysses) the head groups
// of the e4m3 q, k, v and of the bf16 output.
struct Fp8Ws {
  void *vt, *q, *k, *v, *o;
};
Fp8Ws carve_fwd_fp8(Carve& c, const Shape& s) {
  Fp8Ws w{};
  const size_t q8 = (size_t)s.B_eff() * s.S * s.Hq * s.D;
  const size_t kv8 = (size_t)s.B_eff() * s.S * s.Hkv * s.D;
  w.vt = c.take(kv8);
  if (s.ud > 1) {
    w.q = c.take(q8);
    w.k = c.take(kv8);
    w.v = c.take(kv8);
    w.o = c.take(2 * q8);
  }
  return w;
}
}  // namespace

size_t usp_attn_fwd_fp8_workspace_size(int B, int S, int Hq, int Hkv, int D, int cp,
                                       int ud) {
  if (B < 0 || S < 0 || Hq < 1 || Hkv < 1 || D < 1 || cp < 1 || ud < 1) return 0;
  Shape s = shape_of(B, S, Hq, Hkv, D, cp, ud, 0, USP_BF16, 0);
  Carve c(nullptr);
  carve_fwd_fp8(c, s);
  return c.used;
}

usp_status_t usp_attn_fwd_fp8(const void* q, const void* k, const void* v, float q_descale,
                              float k_descale, float v_descale, void* out, float* lse, int B,
                              int S, int Hq, int Hkv, int D, float softmax_scale, int causal,
                              int window, int sink_tokens, const int32_t* cu_seqlens,
                              int cp_size, int ulysses_degree, usp_layout_t layout,
                              unsigned flags, void* workspace, size_t workspace_bytes,
                              usp_stream_t stream) {
  Shape s = shape_of(B, S, Hq, Hkv, D, cp_size, ulysses_degree, layout, USP_BF16,
                     cu_seqlens != nullptr);
  usp_status_t r = validate(s, window, sink_tokens);
  if (r != USP_OK) return r;
  if (flags & USP_FLAG_NATURAL_ORDER) return USP_ERR_UNSUPPORTED;
  if (!(q_descale > 0.f) || !(k_descale > 0.f) || !(v_descale > 0.f) ||
      !std::isfinite(q_descale) || !std::isfinite(k_descale) || !std::isfinite(v_descale))
    return USP_ERR_INVALID_ARG;
  if (S > 0 && (!q || !k || !v || !out || !lse)) return USP_ERR_INVALID_ARG;
  const void* ptrs[] = {q, k, v, out, lse, workspace};
  for (const void* p : ptrs)
    if (!aligned16(p)) return USP_ERR_ALIGNMENT;
  AttnParams P = make_params(s, softmax_scale, causal, window, sink_tokens, cu_seqlens);
  if (!fwd_fp8_supported(P)) return USP_ERR_UNSUPPORTED;
  if (s.B_eff() == 0 || S == 0) return USP_OK;
  Carve c(workspace);
  Fp8Ws w = carve_fwd_fp8(c, s);
  if (!workspace || workspace_bytes < c.used) return USP_ERR_WORKSPACE;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  // the codes' scales: s = scale * <q, k> of the real values
  P.scale *= q_descale * k_descale;
  P.scale_log2 *= q_descale * k_descale;
  const void* vsrc = v;
  if (s.ud > 1) {
    const int B_eff = s.B_eff();
    if ((r = launch_ulysses(q, w.q, B_eff, S, Hq * D, s.ud, 1, st)) != USP_OK) return r;
    if ((r = launch_ulysses(k, w.k, B_eff, S, Hkv * D, s.ud, 1, st)) != USP_OK) return r;
    if ((r = launch_ulysses(v, w.v, B_eff, S, Hkv * D, s.ud, 1, st)) != USP_OK) return r;
    P.q = w.q;
    P.k = w.k;
    P.o = w.o;
    vsrc = w.v;
  } else {
    P.q = q;
    P.k = k;
    P.o = out;
  }
  if ((r = launch_v_transpose(vsrc, w.vt, P.Bt, S, P.Hkv, st)) != USP_OK) return r;
  P.v = w.vt;
  P.lse = lse;
  if ((r = launch_fwd_fp8(P, v_descale, st)) != USP_OK) return r;
  if (s.ud > 1) r = launch_ulysses(w.o, out, s.B_eff(), S, Hq * D * 2, s.ud, 0, st);
  return r;
}

usp_status_t usp_quantize_e4m3(const void* x, void* out, int64_t n, float inv_scale,
                               usp_stream_t stream) {
  if (n < 0 || !std::isfinite(inv_scale)) return USP_ERR_INVALID_ARG;
  if (n > 0 && (!x || !out)) return USP_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(out)) return USP_ERR_ALIGNMENT;
  return launch_quantize_e4m3(x, out, n, inv_scale, reinterpret_cast<cudaStream_t>(stream));
}

usp_status_t usp_merge_partials(const float* o_parts, const float* lse_parts,
                                int n, int64_t rows, int D, int tree_order,
                                void* o_out, usp_dtype_t out_dtype,
                                float* lse_out, usp_stream_t stream) {
  if (n < 1 || rows < 0 || (tree_order && n > 64)) return USP_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return USP_ERR_INVALID_ARG;
  if (out_dtype != USP_BF16 && out_dtype != USP_FP32) return USP_ERR_INVALID_ARG;
  if (rows > 0 && (!o_parts || !lse_parts || !o_out || !lse_out))
    return USP_ERR_INVALID_ARG;
  if (!aligned16(o_parts) || !aligned16(lse_parts) || !aligned16(o_out) ||
      !aligned16(lse_out))
    return USP_ERR_ALIGNMENT;
  return launch_merge(o_parts, lse_parts, n, rows, D, tree_order ? 1 : 0, o_out,
                      out_dtype == USP_BF16 ? 1 : 0, lse_out,
                      reinterpret_cast<cudaStream_t>(stream));
}

usp_status_t usp_permute(const void* src, void* dst, usp_permute_kind_t kind,
                         usp_layout_t layout, int B, int S, int H, int D,
                         int cp_size, int ulysses_degree, int elem_bytes,
                         usp_stream_t stream) {
  if (B < 0 || S < 0 || H <= 0 || D <= 0 || cp_size < 1 || ulysses_degree < 1)
    return USP_ERR_INVALID_ARG;
  if (elem_bytes != 1 && elem_bytes != 2 && elem_bytes != 4) return USP_ERR_INVALID_ARG;
  if (layout < USP_LAYOUT_CONTIGUOUS || layout > USP_LAYOUT_STRIPE)
    return USP_ERR_INVALID_ARG;
  long long row = (long long)H * D * elem_bytes;
  int div = cp_size * ulysses_degree * (layout == USP_LAYOUT_ZIGZAG ? 2 : 1);
  if (S % div != 0) return USP_ERR_INVALID_ARG;
  if ((double)B * S * row / 16.0 >= 2147483647.0) return USP_ERR_UNSUPPORTED;
  if (B * (long long)S > 0 && (!src || !dst)) return USP_ERR_INVALID_ARG;
  if (!aligned16(src) || !aligned16(dst)) return USP_ERR_ALIGNMENT;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  switch (kind) {
    case USP_PERMUTE_EXTRACT:
    case USP_PERMUTE_RESTORE:
      if (row % 16 != 0) return USP_ERR_INVALID_ARG;
      return launch_permute_layout(src, dst, B, S, (int)row, layout, cp_size,
                                   kind == USP_PERMUTE_RESTORE, st);
    case USP_PERMUTE_ULYSSES_SEQ2HEAD:
    case USP_PERMUTE_ULYSSES_HEAD2SEQ:
      if (H % ulysses_degree != 0 || (row / ulysses_degree) % 16 != 0)
        return USP_ERR_INVALID_ARG;
      return launch_ulysses(src, dst, B, S, (int)row, ulysses_degree,
                            kind == USP_PERMUTE_ULYSSES_SEQ2HEAD, st);
  }
  return USP_ERR_INVALID_ARG;
}

}  // extern "C"
