// Logit loads shared by the acceptance and routing kernels (sm_103a): fp32 or bf16 rows,
// streamed in 16-byte loads and widened exactly to fp32.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "common.cuh"

namespace simsd {

__device__ __forceinline__ uint4 ld_stream16(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ uint32_t word_of(const uint4& w, int i) {
  return i == 0 ? w.x : i == 1 ? w.y : i == 2 ? w.z : w.w;
}

// Logit element types: fp32, or bf16 widened exactly to fp32 (its 16 bits are the top half
// of the fp32 pattern). The streaming passes read kVec consecutive entries per 16-byte load
// (4 fp32 or 8 bf16, so a lane keeps as many bytes in flight for either type) and widen
// each with `entry`; the race reads 4 entries per load (`ldg4`, kAlign bytes).
template <typename LT>
struct LogitIO;
template <>
struct LogitIO<float> {
  static constexpr int kVec = 4;
  static constexpr int kAlign = 16;
  static constexpr uint32_t kNegInfWord = 0xff800000u;  // one -inf entry
  static __device__ __forceinline__ float entry(const uint4& w, int j) { return __uint_as_float(word_of(w, j)); }
  // running maximum over whole loads
  using MaxAcc = float;
  static __device__ __forceinline__ MaxAcc max_init() { return -INFINITY; }
  static __device__ __forceinline__ MaxAcc max_acc(MaxAcc a, const uint4& w) {
    return fmaxf(a, fmaxf(fmaxf(__uint_as_float(w.x), __uint_as_float(w.y)),
                          fmaxf(__uint_as_float(w.z), __uint_as_float(w.w))));
  }
  static __device__ __forceinline__ float max_value(MaxAcc a) { return a; }
  static __device__ __forceinline__ float4 ldg4(const float* row, int i) {
    return __ldg(reinterpret_cast<const float4*>(row) + i);
  }
  // entries 4i .. 4i + 3 as loaded, widened only where they are used (so that a batch of
  // loads is issued before any of them is consumed)
  using Raw4 = float4;
  static __device__ __forceinline__ Raw4 ldraw4(const float* row, int i) { return ldg4(row, i); }
  static __device__ __forceinline__ float4 widen4(const Raw4& w) { return w; }
  // the same four entries from an unaligned row, one load each (0 at and past `end`)
  static __device__ __forceinline__ Raw4 ldraw4_each(const float* row, int i, int end) {
    const int v = 4 * i;
    return make_float4(v < end ? __ldg(row + v) : 0.f, v + 1 < end ? __ldg(row + v + 1) : 0.f,
                       v + 2 < end ? __ldg(row + v + 2) : 0.f, v + 3 < end ? __ldg(row + v + 3) : 0.f);
  }
  static __device__ __forceinline__ float ld1(const float* p) { return __ldg(p); }
};
template <>
struct LogitIO<__nv_bfloat16> {
  static constexpr int kVec = 8;
  static constexpr int kAlign = 8;
  static constexpr uint32_t kNegInfWord = 0xff80ff80u;  // two -inf entries
  static __device__ __forceinline__ float lo(uint32_t x) { return __uint_as_float(x << 16); }
  static __device__ __forceinline__ float hi(uint32_t x) { return __uint_as_float(x & 0xffff0000u); }
  static __device__ __forceinline__ float entry(const uint4& w, int j) {
    const uint32_t x = word_of(w, j >> 1);
    return (j & 1) ? hi(x) : lo(x);
  }
  // running maximum on the packed pairs (widening is exact and monotone, so the maximum of
  // the bf16 values widens to the maximum of the widened values; a NaN operand is skipped)
  using MaxAcc = uint32_t;
  static __device__ __forceinline__ uint32_t max2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
  }
  static __device__ __forceinline__ MaxAcc max_init() { return kNegInfWord; }
  static __device__ __forceinline__ MaxAcc max_acc(MaxAcc a, const uint4& w) {
    return max2(a, max2(max2(w.x, w.y), max2(w.z, w.w)));
  }
  static __device__ __forceinline__ float max_value(MaxAcc a) { return fmaxf(lo(a), hi(a)); }
  static __device__ __forceinline__ float4 ldg4(const __nv_bfloat16* row, int i) {
    return widen4(ldraw4(row, i));
  }
  using Raw4 = uint2;
  static __device__ __forceinline__ Raw4 ldraw4(const __nv_bfloat16* row, int i) {
    return __ldg(reinterpret_cast<const uint2*>(row) + i);
  }
  static __device__ __forceinline__ float4 widen4(const Raw4& w) {
    return make_float4(lo(w.x), hi(w.x), lo(w.y), hi(w.y));
  }
  static __device__ __forceinline__ Raw4 ldraw4_each(const __nv_bfloat16* row, int i, int end) {
    const unsigned short* p = reinterpret_cast<const unsigned short*>(row);
    const int v = 4 * i;
    uint32_t e[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) e[j] = v + j < end ? (uint32_t)__ldg(p + v + j) : 0u;
    return make_uint2(e[0] | (e[1] << 16), e[2] | (e[3] << 16));
  }
  static __device__ __forceinline__ float ld1(const __nv_bfloat16* p) {
    return __uint_as_float((uint32_t)__ldg(reinterpret_cast<const unsigned short*>(p)) << 16);
  }
};

// Rows can be streamed with 16-byte loads: V a multiple of kVec and both bases aligned.
template <typename LT>
__device__ __forceinline__ bool stream_ok(int V, const LT* a, const LT* b) {
  return V % LogitIO<LT>::kVec == 0 && ((((uintptr_t)a) | ((uintptr_t)b)) & 15) == 0;
}

// x / T, correctly rounded (the same value in every kernel that scales a logit).
__device__ __forceinline__ float scale_logit(float x, float T, bool unit_T) {
  return unit_T ? x : __fdiv_rn(x, T);
}

// e^(x - m) for x <= m on the exp2 unit: (x - m) log2 e, then ex2.approx.ftz (relative
// error about 2^-22; underflows to 0 below about -87).
__device__ __forceinline__ float exp_shifted(float x, float m) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"((x - m) * 1.4426950408889634f));
  return y;
}

// Resident blocks per SM of `kernel` x SMs of the current device, cached per device in
// `cache` (64 entries).
template <typename K>
int resident_blocks(K kernel, int threads, int* cache) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) dev = 0;
  // (host threads may race here: each computes the same value; the accesses are atomic)
  int v = __atomic_load_n(&cache[dev], __ATOMIC_ACQUIRE);
  if (v == 0) {
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, 0) != cudaSuccess ||
        per_sm < 1)
      per_sm = 1;
    const int sms = device_sm_count();
    v = per_sm * (sms > 0 ? sms : 148);
    __atomic_store_n(&cache[dev], v, __ATOMIC_RELEASE);
  }
  return v;
}

}  // namespace simsd
