// Pieces shared by the two verify-attention kernels: RoPE angle, the temporal-causal
// visibility rule on packed labels, and the host-side argument checks.
#pragma once

#include <math.h>

#include "common.cuh"

namespace simsd {

constexpr int kMaxHalfD = 64;

// Per-call RoPE constants: c_d = theta^(-2d/D) / (2*pi), split into an fp32 head and
// tail (c_hi + c_lo ~ c_d to ~2^-48 relative) so that the fractional number of turns
// pos * c_d can be formed in fp32 without losing the integer part's precision.
struct RopeTable {
  float c_hi[kMaxHalfD];
  float c_lo[kMaxHalfD];
};

static inline void make_rope_table(RopeTable* t, double theta, int D) {
  const int half = D / 2;
  const double two_pi = 6.283185307179586476925286766559;
  for (int d = 0; d < kMaxHalfD; ++d) {
    double c = d < half ? pow(theta, -2.0 * (double)d / (double)D) / two_pi : 0.0;
    float hi = (float)c;
    t->c_hi[d] = hi;
    t->c_lo[d] = (float)(c - (double)hi);
  }
}

// sin / cos of the RoPE angle pos * omega_d. The product pos * c_hi is split exactly into
// its rounded value and rounding error (fma), the whole turns are dropped, and the
// remaining fraction f in about [-1/2, 1/2] turns is passed to sincospi(2f).
// Requires |pos| < 2^24 (exact as fp32).
__device__ __forceinline__ void rope_sincos(int pos, float c_hi, float c_lo, float* s, float* c) {
  const float x = (float)pos;
  const float a = x * c_hi;
  const float e = fmaf(x, c_hi, -a);
  const float f = (a - rintf(a)) + fmaf(x, c_lo, e);
  sincospif(2.0f * f, s, c);
}

// Visibility of response key slot j for a row with threshold t = tau(row) + [row in D]:
// a data key D_j is visible iff tau(j) < t, a mask key D~_j iff tau(j) >= t. This is the
// four-case A_ij of the SimSD mask equation folded into one comparison.
__device__ __forceinline__ bool response_key_visible(uint8_t label_j, int t) {
  const int tau_j = label_j & 0x7F;
  return (label_j & kSegMask) ? (tau_j >= t) : (tau_j < t);
}

__device__ __forceinline__ int row_threshold(uint8_t label_row) {
  return (label_row & 0x7F) + ((label_row & kSegMask) ? 0 : 1);
}

__device__ __forceinline__ float load_f(const float* p) { return *p; }
__device__ __forceinline__ float load_f(const __nv_bfloat16* p) { return __bfloat162float(*p); }
__device__ __forceinline__ void store_f(float* p, float v) { *p = v; }
__device__ __forceinline__ void store_f(__nv_bfloat16* p, float v) { *p = __float2bfloat16_rn(v); }

// Size checks only (the workspace query needs no pointers).
static inline simsd_status check_attn_sizes(const simsd_attn_params* p) {
  if (!p) return SIMSD_ERR_INVALID_ARG;
  if (p->batch < 0 || p->B < 1 || p->B > kMaxB || p->Hq < 1 || p->Hkv < 1 || p->D < 1)
    return SIMSD_ERR_INVALID_ARG;
  if (p->Hq % p->Hkv) return SIMSD_ERR_INVALID_ARG;
  if (p->cache_tokens < 0) return SIMSD_ERR_INVALID_ARG;
  if (p->dtype != SIMSD_DTYPE_FP32 && p->dtype != SIMSD_DTYPE_BF16) return SIMSD_ERR_INVALID_ARG;
  if (p->cache_layout != SIMSD_CACHE_NHD && p->cache_layout != SIMSD_CACHE_HND)
    return SIMSD_ERR_INVALID_ARG;
  if (!(p->rope_theta > 0.f)) return SIMSD_ERR_INVALID_ARG;
  if (p->D != 64 && p->D != 128) return SIMSD_ERR_UNSUPPORTED;
  return SIMSD_OK;
}

static inline simsd_status check_attn_params(const simsd_attn_params* p) {
  const simsd_status st = check_attn_sizes(p);
  if (st != SIMSD_OK || p->batch == 0) return st;
  if (!p->q || !p->k_resp || !p->v_resp || !p->cache_start || !p->prompt_len || !p->pos_ids ||
      !p->labels || !p->out || !p->dev_err)
    return SIMSD_ERR_INVALID_ARG;
  if (p->cache_tokens > 0 && (!p->k_cache || !p->v_cache)) return SIMSD_ERR_INVALID_ARG;
  return SIMSD_OK;
}

// Element offset of cache row (token, head) in either layout.
__device__ __forceinline__ int64_t cache_index(int layout, int64_t tokens, int Hkv, int D,
                                               int64_t token, int h) {
  return layout == SIMSD_CACHE_NHD ? (token * Hkv + h) * (int64_t)D
                                   : ((int64_t)h * tokens + token) * (int64_t)D;
}

}  // namespace simsd
