// Status strings, version, and the verify-attention entry points (dispatch between the
// tcgen05 bf16 kernel and the CUDA-core kernel).
#include <stdio.h>

#include "attn_common.cuh"

namespace simsd {
simsd_status launch_attn_simt(const simsd_attn_params* p, cudaStream_t stream);
bool attn_tc_supported(const simsd_attn_params* p);
size_t attn_tc_workspace(const simsd_attn_params* p);
simsd_status launch_attn_tc(const simsd_attn_params* p, void* ws, size_t ws_bytes,
                            cudaStream_t stream);
}  // namespace simsd

SIMSD_API const char* simsd_status_str(simsd_status s) {
  switch (s) {
    case SIMSD_OK: return "SIMSD_OK";
    case SIMSD_ERR_INVALID_ARG: return "SIMSD_ERR_INVALID_ARG";
    case SIMSD_ERR_UNSUPPORTED: return "SIMSD_ERR_UNSUPPORTED";
    case SIMSD_ERR_WORKSPACE: return "SIMSD_ERR_WORKSPACE";
    case SIMSD_ERR_CUDA: return "SIMSD_ERR_CUDA";
    case SIMSD_ERR_TIMEOUT: return "SIMSD_ERR_TIMEOUT";
  }
  return "SIMSD_ERR_UNKNOWN";
}

SIMSD_API int simsd_version(void) { return 300; }

namespace simsd {
static thread_local char g_last_error[256];
void record_cuda_error(const char* what, cudaError_t e) {
  snprintf(g_last_error, sizeof(g_last_error), "%s%s%s (%d)", what, what[0] ? ": " : "",
           cudaGetErrorString(e), (int)e);
}
}  // namespace simsd

SIMSD_API const char* simsd_last_cuda_error(void) { return simsd::g_last_error; }

SIMSD_API size_t simsd_verify_attention_workspace(const simsd_attn_params* p) {
  if (simsd::check_attn_sizes(p) != SIMSD_OK) return 0;
  if (p->dtype == SIMSD_DTYPE_BF16 && simsd::attn_tc_supported(p)) return simsd::attn_tc_workspace(p);
  return 256;  // the CUDA-core kernel needs no scratch; keep a non-zero minimum
}

SIMSD_API simsd_status simsd_verify_attention(const simsd_attn_params* p, void* workspace,
                                              size_t workspace_bytes, simsd_stream_t stream) {
  SIMSD_NVTX_RANGE("simsd_verify_attention");
  const simsd_status st = simsd::check_attn_params(p);
  if (st != SIMSD_OK) return st;
  if (p->batch == 0) return SIMSD_OK;
  if (p->dtype == SIMSD_DTYPE_BF16 && simsd::attn_tc_supported(p))
    return simsd::launch_attn_tc(p, workspace, workspace_bytes, (cudaStream_t)stream);
  return simsd::launch_attn_simt(p, (cudaStream_t)stream);
}
