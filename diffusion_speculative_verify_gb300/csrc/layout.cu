// simsd_build_layout: paired data/mask layout, copied RoPE ids, packed step labels.
//
// SimSD notes (papernotes.org), "关键设计" items 1-3: the response part of the input is
// [D_1..D_B | D~_1..D~_B]; D_k holds the draft token, D~_k is the [MASK] prediction slot
// bound to it; every response slot carries a step label tau in 1..B (a permutation, per
// the gist.science summary, section 2), and D~_k reuses the position id of D_k. In a later
// round of the same block the slots committed earlier carry tau = 0, like the prompt
// (item 2), and the R remaining positions (item 4) a permutation of 1..R.
// No mask is materialised: labels are enough to evaluate A_ij on the fly.
// With SIMSD_LAYOUT_PHYSICAL_POSITIONS the mask slots take their own sequence index instead
// (the "Without Aligned RoPE" ablation of the SimSD notes' table), a negative control.
#include "common.cuh"

namespace simsd {

// One warp per request; lane k handles slot k (B <= 32).
__global__ void __launch_bounds__(128) build_layout_kernel(
    const int32_t* __restrict__ tau, const int32_t* __restrict__ prompt_len, int batch, int B,
    int mask_pos_offset, int32_t* __restrict__ pos_ids, uint8_t* __restrict__ labels,
    uint32_t* __restrict__ dev_err) {
  // launched as a programmatic dependent of the stream's previous kernel: let the attention
  // grid be placed at once, and read nothing before the previous grid has completed
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int lane = threadIdx.x & 31;
  const int r = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (r >= batch) return;
  const bool active = lane < B;
  const long long ti = (long long)r * B + lane;
  const int t = active && chk(ti, 1, (long long)batch * B, dev_err) ? tau[ti] : 0;
  const int P = chk(r, 1, batch, dev_err) ? prompt_len[r] : 0;
  // tau = 0 marks a slot committed in an earlier round of the block; the R other labels
  // must be a permutation of 1..R  <=>  every value lies in 0..B and the R nonzero values
  // set R distinct bits, the bits of 1..R.
  const bool in_range = !active || (t >= 0 && t <= B);
  const int R = __popc(__ballot_sync(0xffffffffu, active && t != 0));
  const unsigned bit = (active && t >= 1 && t <= B) ? (1u << (t - 1)) : 0u;
  const unsigned covered = __reduce_or_sync(0xffffffffu, bit);
  const unsigned full = (R == 32) ? 0xffffffffu : ((1u << R) - 1u);
  const bool perm_ok = __all_sync(0xffffffffu, in_range) && covered == full;
  uint32_t bad = 0;
  if (!perm_ok) bad |= SIMSD_DEVERR_TAU;
  if (P < 0) bad |= SIMSD_DEVERR_PROMPT_LEN;
  if (!active) return;
  const size_t row = (size_t)r * 2 * B;
  if (!chk((long long)row + lane, 1, (long long)batch * 2 * B, dev_err) ||
      !chk((long long)row + B + lane, 1, (long long)batch * 2 * B, dev_err))
    return;
  if (bad) {
    pos_ids[row + lane] = -1;
    pos_ids[row + B + lane] = -1;
    labels[row + lane] = kLabelInvalid;
    labels[row + B + lane] = kLabelInvalid;
    if (lane == 0) atomicOr(dev_err, bad);
    return;
  }
  pos_ids[row + lane] = P + lane;      // D_k: next response position
  pos_ids[row + B + lane] = P + mask_pos_offset + lane;  // D~_k: D_k's id (offset 0) or its own
  labels[row + lane] = (uint8_t)t;
  labels[row + B + lane] = (uint8_t)(kSegMask | t);
}

}  // namespace simsd

SIMSD_API simsd_status simsd_build_layout_ex(const int32_t* tau, const int32_t* prompt_len,
                                             int batch, int B, uint32_t flags, int32_t* pos_ids,
                                             uint8_t* labels, uint32_t* dev_err,
                                             simsd_stream_t stream) {
  SIMSD_NVTX_RANGE("simsd_build_layout_ex");
  if (batch < 0 || B < 1 || B > simsd::kMaxB) return SIMSD_ERR_INVALID_ARG;
  if (flags & ~(uint32_t)SIMSD_LAYOUT_PHYSICAL_POSITIONS) return SIMSD_ERR_INVALID_ARG;
  if (batch == 0) return SIMSD_OK;
  if (!tau || !prompt_len || !pos_ids || !labels || !dev_err) return SIMSD_ERR_INVALID_ARG;
  const int warps = 4;
  const int grid = (batch + warps - 1) / warps;
  const int offset = (flags & SIMSD_LAYOUT_PHYSICAL_POSITIONS) ? B : 0;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3((unsigned)(warps * 32));
  cfg.stream = (cudaStream_t)stream;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, simsd::build_layout_kernel, tau, prompt_len, batch, B,
                                           offset, pos_ids, labels, dev_err);
  if (e != cudaSuccess) {
    simsd::record_cuda_error("cudaLaunchKernelEx(build_layout_kernel)", e);
    return SIMSD_ERR_CUDA;
  }
  return simsd::last_launch_status();
}

SIMSD_API simsd_status simsd_build_layout(const int32_t* tau, const int32_t* prompt_len,
                                          int batch, int B, int32_t* pos_ids, uint8_t* labels,
                                          uint32_t* dev_err, simsd_stream_t stream) {
  return simsd_build_layout_ex(tau, prompt_len, batch, B, 0u, pos_ids, labels, dev_err, stream);
}
