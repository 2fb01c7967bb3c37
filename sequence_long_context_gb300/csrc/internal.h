// Host-side declarations shared between the library's translation units.
#pragma once

#include <cuda_runtime.h>

#include "../../include/usp.h"
#include "common.cuh"

namespace usp {

// Counts kernel launches enqueued by this library (usp_launch_count()).
void note_launch(int n = 1);

// Number of SMs of the current device (cached per device).
int sm_count();

// Converts the last CUDA error (after a launch) into a status.
usp_status_t check_launch();

// Records a human-readable reason for the USP_ERR_CUDA about to be returned
// (usp_last_error_detail()); returns USP_ERR_CUDA.
usp_status_t fail_cuda(const char* where, cudaError_t e);
usp_status_t fail_cuda_msg(const char* where, const char* msg);
// Sets the usp_last_error_detail() text without changing any status.
void set_error_detail(const char* msg);

// Brackets one kernel launch with timing events when the kernel timer is on
// (usp_profile_enable); a no-op otherwise.
struct ProfScope {
  int idx;
  cudaStream_t st;
  ProfScope(cudaStream_t s, const char* name);
  ~ProfScope();
};

// permute.cu
usp_status_t launch_permute_layout(const void* src, void* dst, int B, int S,
                                   int row_bytes, int layout, int cp,
                                   int restore, cudaStream_t st);
// flat_row_bytes / flat_off_bytes: the [B*S] token rows of the flat side
// (the source of seq2head, the destination of head2seq) are flat_row_bytes
// apart and start flat_off_bytes in (0, 0: dense rows of row_bytes).
// natural_layout >= 0: the flat side is in natural sequence order, the
// grouped side rank-major for that layout over cp ring ranks (the layout's
// extract / restore fused into the exchange); -1: both rank-major.
usp_status_t launch_ulysses(const void* src, void* dst, int B, int S,
                            int row_bytes, int ud, int seq2head,
                            cudaStream_t st, int flat_row_bytes = 0,
                            int flat_off_bytes = 0, int natural_layout = -1,
                            int cp = 1);

// merge.cu
usp_status_t launch_merge(const float* o_parts, const float* lse_parts, int n,
                          long long rows, int D, int tree, void* o_out,
                          int out_bf16, float* lse_out, cudaStream_t st);

// attn_simt.cu (CUDA-core kernels, fp32 arithmetic; any supported shape)
usp_status_t launch_fwd_simt(const AttnParams& P, int bf16, cudaStream_t st);
usp_status_t launch_bwd_preprocess(const AttnParams& P, int bf16,
                                   int zero_dq_acc, cudaStream_t st);
usp_status_t launch_bwd_simt(const AttnParams& P, int bf16, cudaStream_t st);

// attn_fwd_tc.cu (tcgen05 tensor-core forward, bf16)
bool fwd_tc_supported(const AttnParams& P);
usp_status_t launch_fwd_tc(const AttnParams& P, cudaStream_t st);

int read_clear_fwd_tc_status();  // -1 on a CUDA error

// attn_fwd_fp8.cu (tcgen05 tensor-core forward, e4m3 q/k/v, D = 128)
bool fwd_fp8_supported(const AttnParams& P);
usp_status_t launch_fwd_fp8(const AttnParams& P, float v_descale, cudaStream_t st);
usp_status_t launch_v_transpose(const void* v, void* vt, int Bt, int S, int H,
                                cudaStream_t st);
usp_status_t launch_quantize_e4m3(const void* x, void* out, long long n, float inv_scale,
                                  cudaStream_t st);
int read_clear_fwd_fp8_status();  // -1 on a CUDA error

// attn_bwd_tc.cu (tcgen05 tensor-core backward, bf16)
usp_status_t launch_decode_split(const void* q, const void* k, const void* v, float* o_part,
                                 float* lse_part, int B, int Tq, int S, int Hq, int Hkv, int D,
                                 float scale, int causal, int n_part, cudaStream_t st);
int read_clear_decode_status();  // -1 on a CUDA error
usp_status_t launch_selftest_wait_timeout(unsigned limit_us, cudaStream_t st);
int read_clear_selftest_status();  // -1 on a CUDA error
int decode_max_rows();
int decode_keys_per_tile();

bool bwd_tc_supported(const AttnParams& P);
usp_status_t launch_bwd_tc(const AttnParams& P, cudaStream_t st);
int read_clear_bwd_tc_status();  // -1 on a CUDA error

}  // namespace usp
