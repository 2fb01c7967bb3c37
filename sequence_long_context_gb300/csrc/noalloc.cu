// usp_attn_bwd_noalloc: the backward pass for callers that cannot allocate.
//
// usp_attn_bwd needs scratch (Delta, the LSE in log2 units, the fp32 dQ
// accumulator, and the Ulysses exchange buffers) and takes it from a
// workspace the caller allocates. Some callers cannot do that: a runtime
// that has handed all device memory to its own pools before the attention
// layer runs, or code on a path where calling cudaMalloc is not allowed
// (cudaMalloc may synchronise the device, and some host contexts forbid
// it). For them this entry point takes its scratch from one fixed array in
// device memory, declared below at file scope, and allocates nothing.
//
// The array is shared by every call in the process: calls that overlap on
// the GPU (for example on two streams) race on it. Its contents persist
// between calls; everything the kernels need zeroed (the dQ accumulator) is
// cleared on the device at the start of every call.
//
// When the array takes device memory: it belongs to this file's module,
// which the CUDA runtime loads on a device when something first needs it
// there. With the runtime's default lazy module loading that is the first
// usp_attn_bwd_noalloc call on the device (its cudaGetSymbolAddress), so
// the 64 MiB are reserved then, and stay until the process exits.
#include <cudaTypedefs.h>

#include <mutex>

#include "internal.h"

namespace usp {
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(64) << 20;  // 64 MiB
constexpr int kMaxDevices = 256;

// In host code this name is only a stand-in for the symbol; the device
// address comes from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_mu;
struct DeviceScratch {
  void* addr;
  unsigned long long ctx_id;  // context the address belongs to
};
DeviceScratch g_scratch[kMaxDevices] = {};

// Unique id of the calling thread's current context (0 if there is none or
// the driver cannot say). A device reset destroys the context and the next
// one gets a new id, so an address looked up before the reset is not reused.
unsigned long long current_context_id() {
  static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
  static PFN_cuCtxGetId_v12000 get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
  });
  if (!get_current || !get_id) return 0;
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
  if (get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

// Device address of the scratch array on the current device. It is looked
// up (with that device current) on the first call on each device and again
// whenever the device's context has changed since (after a device reset);
// otherwise the cached address is returned.
usp_status_t scratch_on_current_device(void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail_cuda("cudaGetDevice", e);
  if (dev < 0 || dev >= kMaxDevices)
    return fail_cuda_msg("usp_attn_bwd_noalloc", "device ordinal out of range");
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceScratch& s = g_scratch[dev];
  const unsigned long long ctx = current_context_id();
  if (s.addr == nullptr || ctx == 0 || ctx != s.ctx_id) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return fail_cuda("cudaGetSymbolAddress(scratch)", e);
    s.addr = p;
    // the lookup has made the device's context current if it was not yet
    s.ctx_id = ctx != 0 ? ctx : current_context_id();
  }
  *out = s.addr;
  return USP_OK;
}

}  // namespace
}  // namespace usp

using namespace usp;

extern "C" {

usp_status_t usp_attn_bwd_noalloc(const void* q, const void* k, const void* v,
                                  const void* out, const float* lse,
                                  const void* dout, void* dq, void* dk,
                                  void* dv, int B, int S, int Hq, int Hkv,
                                  int D, float softmax_scale, int causal,
                                  int window, int sink_tokens,
                                  const int32_t* cu_seqlens, int cp_size,
                                  int ulysses_degree, usp_layout_t layout,
                                  usp_dtype_t dtype, unsigned flags,
                                  usp_stream_t stream) {
  if (flags & USP_FLAG_SAVED_EXCHANGE) {
    set_error_detail("usp_attn_bwd_noalloc: USP_FLAG_SAVED_EXCHANGE needs the "
                     "forward's workspace, which this call does not take");
    return USP_ERR_INVALID_ARG;
  }
  // Argument check first, without a workspace: usp_attn_bwd validates every
  // argument and then refuses the missing workspace before it launches
  // anything, or returns USP_OK at once for an empty problem.
  const usp_status_t dry = usp_attn_bwd(q, k, v, out, lse, dout, dq, dk, dv, B, S, Hq, Hkv, D,
                                        softmax_scale, causal, window, sink_tokens, cu_seqlens,
                                        cp_size, ulysses_degree, layout, dtype, flags, nullptr,
                                        0, stream);
  if (dry != USP_OK && dry != USP_ERR_WORKSPACE) return dry;
  void* scratch = nullptr;
  usp_status_t r = scratch_on_current_device(&scratch);
  if (r != USP_OK || dry == USP_OK) return r;  // an empty problem: set-up only
  r = usp_attn_bwd(q, k, v, out, lse, dout, dq, dk, dv, B, S, Hq, Hkv, D, softmax_scale,
                   causal, window, sink_tokens, cu_seqlens, cp_size, ulysses_degree, layout,
                   dtype, flags, scratch, kNoAllocScratchBytes, stream);
  if (r == USP_ERR_WORKSPACE)
    set_error_detail("usp_attn_bwd_noalloc: problem needs more scratch than "
                     "the fixed 64 MiB array holds");
  return r;
}

}  // extern "C"
