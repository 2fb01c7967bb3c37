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
#include <mutex>

#include "internal.h"

namespace usp {
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(64) << 20;  // 64 MiB
constexpr int kMaxDevices = 256;

// Every GPU that loads this library holds these 64 MiB until the process
// exits. In host code this name is only a stand-in for the symbol; the
// device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device, looked up
// once per device (with that device current) and cached.
usp_status_t scratch_on_current_device(void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail_cuda("cudaGetDevice", e);
  if (dev < 0 || dev >= kMaxDevices)
    return fail_cuda_msg("usp_attn_bwd_noalloc", "device ordinal out of range");
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return fail_cuda("cudaGetSymbolAddress(scratch)", e);
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
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
  // Packed batches keep one leading batch row in their tensors.
  const int b_tensor = cu_seqlens != nullptr ? 1 : B;
  const size_t need = usp_attn_bwd_workspace_size(
      b_tensor, S, Hq, Hkv, D, cp_size, ulysses_degree, dtype, flags);
  if (need > kNoAllocScratchBytes) {
    set_error_detail("usp_attn_bwd_noalloc: problem needs more scratch than "
                     "the fixed 64 MiB array holds");
    return USP_ERR_WORKSPACE;
  }
  void* scratch = nullptr;
  usp_status_t r = scratch_on_current_device(&scratch);
  if (r != USP_OK) return r;
  return usp_attn_bwd(q, k, v, out, lse, dout, dq, dk, dv, B, S, Hq, Hkv, D,
                      softmax_scale, causal, window, sink_tokens, cu_seqlens,
                      cp_size, ulysses_degree, layout, dtype, flags, scratch,
                      kNoAllocScratchBytes, stream);
}

}  // extern "C"
