// Self-test of the failure path shared by the tensor-core kernels: a pipeline
// wait that can never complete must give up after its limit, record
// USP_ERR_TIMEOUT in a device status word, and let the kernel exit normally,
// so the context stays usable. One CTA waits, with the kernels' own bounded
// wait, on an mbarrier phase that nothing ever completes.
#include "internal.h"
#include "tc_ptx.cuh"

namespace usp {
namespace {

using namespace tc;

__device__ int g_selftest_status = 0;

__global__ void wait_timeout_kernel(uint64_t limit_ns, int* status) {
  __shared__ __align__(8) uint64_t bar_mem;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    const uint32_t bar = smem_u32(&bar_mem);
    mbar_init(bar, 1);  // one arrival needed; none is ever made
    abort_flag = 0;
    fence_barrier_init();
    mbar_wait(bar, 0, &abort_flag, status, limit_ns);
  }
}

}  // namespace

int read_clear_selftest_status() {
  int v = 0, z = 0;
  if (cudaMemcpyFromSymbol(&v, g_selftest_status, sizeof(int)) != cudaSuccess) return -1;
  if (v != 0) cudaMemcpyToSymbol(g_selftest_status, &z, sizeof(int));
  return v;
}

usp_status_t launch_selftest_wait_timeout(unsigned limit_us, cudaStream_t st) {
  int* status = nullptr;
  cudaError_t e = cudaGetSymbolAddress(reinterpret_cast<void**>(&status), g_selftest_status);
  if (e != cudaSuccess) return fail_cuda("cudaGetSymbolAddress(status)", e);
  wait_timeout_kernel<<<1, 32, 0, st>>>((uint64_t)limit_us * 1000ull, status);
  note_launch();
  return check_launch();
}

}  // namespace usp
