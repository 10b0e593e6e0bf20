// Shared device/host helpers of the SimSD verification library (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "simsd.h"

#define SIMSD_API extern "C" __attribute__((visibility("default")))

#include <nvtx3/nvToolsExt.h>

namespace simsd {

constexpr int kMaxB = 32;          // block size limit (labels hold tau in 7 bits; warp scans)
constexpr uint8_t kSegMask = 0x80; // label bit: mask slot D~
constexpr uint8_t kLabelInvalid = 0xFF;

// Records the text of the last CUDA failure seen on this host thread.
void record_cuda_error(const char* what, cudaError_t e);

static inline simsd_status cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return SIMSD_OK;
  record_cuda_error("", e);
  return SIMSD_ERR_CUDA;
}

static inline simsd_status last_launch_status() {
  return cuda_status(cudaGetLastError());
}

static inline int device_sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

static inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// NVTX range around one call of the C interface, named after it, so that a timeline
// profiler shows each call with its kernels (an NVTX call costs a few ns when no tool is
// attached).
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};
#define SIMSD_NVTX_RANGE(name) ::simsd::NvtxRange simsd_nvtx_range_(name)

// --------------------------------------------------------------------- checked build
// Built with -DSIMSD_CHECKED, every kernel checks the index of each global access against
// the extent of the array it addresses (extents follow from the call's sizes; for a row
// read in one piece the row's range is checked); an index outside sets SIMSD_DEVERR_BOUNDS
// in the call's error word and the access is skipped (a skipped load yields a neutral
// value). It stands in for a memory checker where none can run. In the default build every
// check is the constant true and compiles away.
#ifdef SIMSD_CHECKED
constexpr bool kChecked = true;
#else
constexpr bool kChecked = false;
#endif

// True when [i, i + len) lies inside [0, n); otherwise (checked build only) raises
// SIMSD_DEVERR_BOUNDS in *err.
__device__ __forceinline__ bool chk(long long i, long long len, long long n, uint32_t* err) {
  if constexpr (!kChecked) {
    return true;
  } else {
    if (i >= 0 && len >= 0 && i + len <= n) return true;
    atomicOr(err, SIMSD_DEVERR_BOUNDS);
    return false;
  }
}

// ------------------------------------------------------------------------------ Philox
// Philox4x32-10 as defined by Salmon, Moraes, Dror, Shaw (SC'11): each round forms the
// 64-bit products of counter words 0 and 2 with two odd multipliers, and the new counter
// is (hi(c2*M1) ^ c1 ^ k0, lo(c2*M1), hi(c0*M0) ^ c3 ^ k1, lo(c0*M0)); the key is advanced
// by two Weyl increments between rounds.
struct Philox4 {
  uint32_t x, y, z, w;
};

__device__ __forceinline__ Philox4 philox4x32_10(Philox4 c, uint32_t k0, uint32_t k1) {
  const uint32_t kM0 = 0xD2511F53u, kM1 = 0xCD9E8D57u;
  const uint32_t kW0 = 0x9E3779B9u, kW1 = 0xBB67AE85u;
#pragma unroll
  for (int round = 0; round < 10; ++round) {
    if (round) {
      k0 += kW0;
      k1 += kW1;
    }
    const uint32_t hi0 = __umulhi(kM0, c.x), lo0 = kM0 * c.x;
    const uint32_t hi1 = __umulhi(kM1, c.z), lo1 = kM1 * c.z;
    Philox4 n;
    n.x = hi1 ^ c.y ^ k0;
    n.y = lo1;
    n.z = hi0 ^ c.w ^ k1;
    n.w = lo0;
    c = n;
  }
  return c;
}

// Odd multiple of 2^-24 in (0, 1): exact in fp32.
__device__ __forceinline__ float word_to_uniform(uint32_t w) {
  return (float)(((w >> 9) << 1) | 1u) * 5.9604644775390625e-8f;  // * 2^-24
}

__device__ __forceinline__ uint32_t philox_word(const Philox4& r, int i) {
  return i == 0 ? r.x : (i == 1 ? r.y : (i == 2 ? r.z : r.w));
}

constexpr uint32_t kResampleTag = 0x80000000u;
constexpr uint32_t kNoiseTag = 0x40000000u;  // coupled-noise table: (request, position, offset lo, tag | v/4)

}  // namespace simsd
