// tcgen05 tensor-core backward (bf16 in, fp32 accumulate). Not yet enabled.
#include "internal.h"

namespace usp {
bool bwd_tc_supported(const AttnParams&) { return false; }
usp_status_t launch_bwd_tc(const AttnParams&, cudaStream_t) { return USP_ERR_UNSUPPORTED; }
int read_clear_bwd_tc_status() { return 0; }
}  // namespace usp
