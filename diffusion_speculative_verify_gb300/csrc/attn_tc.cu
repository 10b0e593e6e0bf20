// tcgen05 / TMEM verify attention (bf16) -- placeholder until the tensor-core kernel lands.
#include "attn_common.cuh"

namespace simsd {
bool attn_tc_supported(const simsd_attn_params*) { return false; }
size_t attn_tc_workspace(const simsd_attn_params*) { return 256; }
simsd_status launch_attn_tc(const simsd_attn_params*, void*, size_t, cudaStream_t) {
  return SIMSD_ERR_UNSUPPORTED;
}
}  // namespace simsd
