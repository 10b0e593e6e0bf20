// simsd_accept: speculative acceptance along the draft's step order + residual resampling.
//
// SimSD notes (papernotes.org), "关键设计" item 4: alpha_r = min(1, p_theta / p_phi) for the
// draft token of step r, the longest accepted prefix is kept, and the first rejected slot
// is resampled in place by the target. The residual is max(0, p - q) normalised (S2D2 page,
// "方法步骤详情" step (5)); it is drawn by the exponential race argmax_v r_v / E_v, the
// Gumbel-max identity of the SPOT page ("Gumbel-Max 技巧与随机耦合"), which needs neither
// the normaliser of the residual nor a prefix scan over the vocabulary.
//
// Two launches:
//   K3a accept_stats    : grid over (request, step, model, vocab chunk); streams the logit
//                         row chunk once and writes its (max, sum exp) pair.
//   K3b accept_finish   : grid over (request, vocab chunk); every CTA merges the chunk
//                         pairs, re-derives the accept decisions (cheap), and if a step was
//                         rejected runs the race over its chunk of the rejected slot's rows;
//                         winners meet in a 64-bit atomicMax; the last CTA of the request
//                         (atomic ticket, no waiting) writes the outputs and re-zeroes the
//                         request's scratch.
#include <float.h>

#include <mutex>

#include "common.cuh"

namespace simsd {

namespace {

constexpr int kStatThreads = 512;
constexpr int kFinishThreads = 256;

struct AcceptWs {
  float2* stats;                // [batch][gamma][2][nchunk]  (max, sum exp) per chunk
  unsigned long long* winners;  // [batch][2]  race winners: residual, target
  unsigned* any_pos;            // [batch]     residual has a positive entry
  unsigned* ticket;             // [batch]     CTAs of K3b finished
};

struct AcceptPlan {
  int nchunk_a, chunk_a;  // K3a: chunks per row, elements per chunk (multiple of 4)
  int nchunk_b, chunk_b;  // K3b: chunks per request, elements per chunk (multiple of 4)
  size_t off_stats, off_winners, off_anypos, off_ticket, bytes;
};

AcceptPlan make_plan(int batch, int gamma, int V) {
  AcceptPlan p;
  const long rows = (long)batch * gamma * 2;
  const long target_ctas = 1216;  // keeps every SM busy several times over
  long na = rows > 0 ? (target_ctas + rows - 1) / rows : 1;
  const long max_na = (V + 4095) / 4096;
  if (na > max_na) na = max_na;
  if (na < 1) na = 1;
  p.nchunk_a = (int)na;
  p.chunk_a = (int)(((V + na - 1) / na + 3) / 4 * 4);
  long nb = batch > 0 ? (608 + batch - 1) / batch : 1;
  const long max_nb = (V + 1023) / 1024;
  if (nb > max_nb) nb = max_nb;
  if (nb < 1) nb = 1;
  p.nchunk_b = (int)nb;
  p.chunk_b = (int)(((V + nb - 1) / nb + 3) / 4 * 4);
  size_t off = 0;
  p.off_stats = off;
  off = align_up(off + (size_t)batch * gamma * 2 * p.nchunk_a * sizeof(float2), 256);
  p.off_winners = off;
  off = align_up(off + (size_t)batch * 2 * sizeof(unsigned long long), 256);
  p.off_anypos = off;
  off = align_up(off + (size_t)batch * sizeof(unsigned), 256);
  p.off_ticket = off;
  off = align_up(off + (size_t)batch * sizeof(unsigned), 256);
  p.bytes = off;
  return p;
}

__device__ __forceinline__ float4 ld_stream4(const float* p) {
  float4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.f32 {%0,%1,%2,%3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ float scale_logit(float x, float T, bool unit_T) {
  return unit_T ? x : __fdiv_rn(x, T);
}

// Merge two (max, sum exp(x - max)) pairs.
__device__ __forceinline__ void lse_merge(float& m, float& s, float m2, float s2) {
  if (m2 == -INFINITY) return;
  if (m == -INFINITY) {
    m = m2;
    s = s2;
    return;
  }
  if (m2 > m) {
    s = s * expf(m - m2) + s2;
    m = m2;
  } else {
    s = s + s2 * expf(m2 - m);
  }
}

// Slot whose data label carries step `step1` (1-based), or -1.
__device__ __forceinline__ int slot_of_step(const uint8_t* lab, int B, int step1) {
  for (int k = 0; k < B; ++k)
    if ((lab[k] & 0x7F) == step1 && !(lab[k] & kSegMask)) return k;
  return -1;
}

// ----------------------------------------------------------------------------- K3a
__global__ void __launch_bounds__(kStatThreads) accept_stats_kernel(
    const float* __restrict__ target, const float* __restrict__ draft,
    const uint8_t* __restrict__ labels, int batch, int B, int gamma, int V, float T,
    AcceptPlan plan, AcceptWs ws) {
  const int nchunk = plan.nchunk_a;
  int idx = blockIdx.x;
  const int chunk = idx % nchunk;
  idx /= nchunk;
  const int model = idx & 1;
  idx >>= 1;
  const int step = idx % gamma;
  const int r = idx / gamma;

  if (blockIdx.x == 0) {  // scratch of K3b starts at zero on every call
    for (int i = threadIdx.x; i < batch; i += blockDim.x) {
      ws.winners[2 * i] = 0ull;
      ws.winners[2 * i + 1] = 0ull;
      ws.any_pos[i] = 0u;
      ws.ticket[i] = 0u;
    }
  }

  __shared__ int s_slot;
  if (threadIdx.x == 0) s_slot = slot_of_step(labels + (size_t)r * 2 * B, B, step + 1);
  __syncthreads();
  const int k = s_slot;
  float m = -INFINITY, s = 0.f;
  if (k >= 0) {
    const float* row = (model ? draft : target) + ((size_t)r * B + k) * (size_t)V;
    const int c0 = chunk * plan.chunk_a;
    const int c1 = min(V, c0 + plan.chunk_a);
    const bool unit_T = (T == 1.f);
    const bool vec = ((V & 3) == 0) && ((((uintptr_t)row) & 15) == 0);
    if (vec) {
      const int n4 = (c1 - c0) >> 2;  // c0 is a multiple of 4; V too
      const float* base = row + c0;
      int i = threadIdx.x;
      for (; i + 3 * kStatThreads < n4; i += 4 * kStatThreads) {
        float4 x[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) x[u] = ld_stream4(base + 4 * (i + u * kStatThreads));
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const float z0 = scale_logit(x[u].x, T, unit_T), z1 = scale_logit(x[u].y, T, unit_T);
          const float z2 = scale_logit(x[u].z, T, unit_T), z3 = scale_logit(x[u].w, T, unit_T);
          const float mx = fmaxf(fmaxf(z0, z1), fmaxf(z2, z3));
          if (mx > m) {
            s *= expf(m - mx);
            m = mx;
          }
          s += expf(z0 - m) + expf(z1 - m) + expf(z2 - m) + expf(z3 - m);
        }
      }
      for (; i < n4; i += kStatThreads) {
        const float4 x = ld_stream4(base + 4 * i);
        const float z0 = scale_logit(x.x, T, unit_T), z1 = scale_logit(x.y, T, unit_T);
        const float z2 = scale_logit(x.z, T, unit_T), z3 = scale_logit(x.w, T, unit_T);
        const float mx = fmaxf(fmaxf(z0, z1), fmaxf(z2, z3));
        if (mx > m) {
          s *= expf(m - mx);
          m = mx;
        }
        s += expf(z0 - m) + expf(z1 - m) + expf(z2 - m) + expf(z3 - m);
      }
    } else {
      for (int v = c0 + threadIdx.x; v < c1; v += kStatThreads) {
        const float z = scale_logit(row[v], T, unit_T);
        if (z > m) {
          s *= expf(m - z);
          m = z;
        }
        s += expf(z - m);
      }
    }
  }
  // block reduction of (m, s)
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
    const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
    lse_merge(m, s, m2, s2);
  }
  __shared__ float sm[kStatThreads / 32], ss[kStatThreads / 32];
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) {
    sm[w] = m;
    ss[w] = s;
  }
  __syncthreads();
  if (w == 0) {
    m = lane < kStatThreads / 32 ? sm[lane] : -INFINITY;
    s = lane < kStatThreads / 32 ? ss[lane] : 0.f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
      const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
      lse_merge(m, s, m2, s2);
    }
    if (lane == 0)
      ws.stats[(((size_t)r * gamma + step) * 2 + model) * nchunk + chunk] = make_float2(m, s);
  }
}

// ----------------------------------------------------------------------------- K3b
__device__ __forceinline__ unsigned long long pack_key(float key, int v) {
  // keys are >= 0, so their bit patterns order like the values; the low word prefers
  // the smaller token id on equal keys
  return ((unsigned long long)__float_as_uint(key) << 32) | (unsigned)(0xFFFFFFFFu - (unsigned)v);
}

__device__ __forceinline__ int unpack_token(unsigned long long w) {
  return (int)(0xFFFFFFFFu - (unsigned)(w & 0xFFFFFFFFull));
}

__global__ void __launch_bounds__(kFinishThreads) accept_finish_kernel(
    const float* __restrict__ target, const float* __restrict__ draft,
    const int32_t* __restrict__ tokens, const uint8_t* __restrict__ labels, int batch, int B,
    int gamma, int V, float T, uint32_t key0, uint32_t key1, uint32_t off_lo, uint32_t off_hi,
    AcceptPlan plan, AcceptWs ws, int32_t* __restrict__ accepted_len,
    int32_t* __restrict__ out_tokens, int32_t* __restrict__ out_pos,
    int32_t* __restrict__ n_commit, uint32_t* __restrict__ dev_err) {
  const int chunk = blockIdx.x % plan.nchunk_b;
  const int r = blockIdx.x / plan.nchunk_b;
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const uint8_t* lab = labels + (size_t)r * 2 * B;
  const bool unit_T = (T == 1.f);

  __shared__ int s_order[kMaxB];
  __shared__ int s_a, s_bad;
  __shared__ float s_mt, s_st, s_md, s_sd;

  if (w == 0) {
    // step labels of the data half -> order o_t; validity of the permutation
    const uint8_t lb = lane < B ? lab[lane] : 0;
    const int tau = lb & 0x7F;
    const bool ok_lane = lane >= B || (lb != kLabelInvalid && !(lb & kSegMask) && tau >= 1 && tau <= B);
    const unsigned bit = (lane < B && tau >= 1 && tau <= B) ? (1u << (tau - 1)) : 0u;
    const unsigned cover = __reduce_or_sync(0xffffffffu, bit);
    const unsigned full = B == 32 ? 0xffffffffu : ((1u << B) - 1u);
    const bool perm = __all_sync(0xffffffffu, ok_lane) && cover == full;
    if (perm && lane < B) s_order[tau - 1] = lane;
    __syncwarp();
    int bad = perm ? 0 : (int)SIMSD_DEVERR_TAU;
    int x = 0, k = 0;
    if (perm && lane < gamma) {
      k = s_order[lane];
      x = tokens[(size_t)r * B + k];
    }
    const bool tok_bad = perm && lane < gamma && (x < 0 || x >= V);
    if (__any_sync(0xffffffffu, tok_bad)) bad |= (int)SIMSD_DEVERR_TOKEN;
    int a = gamma;
    if (!bad) {
      bool acc = true;
      float mt = 0.f, st = 0.f, md = 0.f, sd = 0.f;
      if (lane < gamma) {
        float m1 = -INFINITY, s1 = 0.f, m2 = -INFINITY, s2 = 0.f;
        const float2* st_t = ws.stats + (((size_t)r * gamma + lane) * 2 + 0) * plan.nchunk_a;
        const float2* st_d = ws.stats + (((size_t)r * gamma + lane) * 2 + 1) * plan.nchunk_a;
        for (int c = 0; c < plan.nchunk_a; ++c) {
          const float2 a2 = st_t[c], b2 = st_d[c];
          lse_merge(m1, s1, a2.x, a2.y);
          lse_merge(m2, s2, b2.x, b2.y);
        }
        mt = m1;
        st = s1;
        md = m2;
        sd = s2;
        const size_t rowoff = ((size_t)r * B + k) * (size_t)V + x;
        const float px = __fdiv_rn(expf(scale_logit(target[rowoff], T, unit_T) - mt), st);
        const float qx = __fdiv_rn(expf(scale_logit(draft[rowoff], T, unit_T) - md), sd);
        Philox4 c4 = {(uint32_t)r, off_lo, off_hi, (uint32_t)(lane >> 2)};
        const Philox4 rnd = philox4x32_10(c4, key0, key1);
        const float u = word_to_uniform(philox_word(rnd, lane & 3));
        acc = (px >= qx) || (u * qx < px);
      }
      const unsigned rej = __ballot_sync(0xffffffffu, lane < gamma && !acc);
      a = rej ? (__ffs(rej) - 1) : gamma;
      if (a < gamma && lane == a) {
        s_mt = mt;
        s_st = st;
        s_md = md;
        s_sd = sd;
      }
    }
    if (lane == 0) {
      s_a = a;
      s_bad = bad;
    }
  }
  __syncthreads();
  const int a = s_a;
  const int bad = s_bad;
  if (bad) {
    if (chunk == 0) {
      if (tid == 0) {
        atomicOr(dev_err, (uint32_t)bad);
        accepted_len[r] = -1;
        n_commit[r] = 0;
      }
      for (int i = tid; i < B; i += blockDim.x) {
        out_tokens[(size_t)r * B + i] = -1;
        out_pos[(size_t)r * B + i] = -1;
      }
    }
    return;
  }

  if (a < gamma) {
    // exponential race over this CTA's chunk of the rejected slot's vocabulary
    const int k = s_order[a];
    const float mt = s_mt, st = s_st, md = s_md, sd = s_sd;
    const float* trow = target + ((size_t)r * B + k) * (size_t)V;
    const float* drow = draft + ((size_t)r * B + k) * (size_t)V;
    const int c0 = chunk * plan.chunk_b;
    const int c1 = min(V, c0 + plan.chunk_b);
    unsigned long long best_res = 0ull, best_p = 0ull;
    bool anyp = false;
    for (int g = c0 / 4 + tid; g * 4 < c1; g += blockDim.x) {
      Philox4 c4 = {(uint32_t)r, off_lo, off_hi, kResampleTag | (uint32_t)g};
      const Philox4 rnd = philox4x32_10(c4, key0, key1);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int v = 4 * g + j;
        if (v >= c1) break;
        const float p = __fdiv_rn(expf(scale_logit(trow[v], T, unit_T) - mt), st);
        const float q = __fdiv_rn(expf(scale_logit(drow[v], T, unit_T) - md), sd);
        const float res = fmaxf(p - q, 0.f);
        const float E = -logf(word_to_uniform(philox_word(rnd, j)));
        anyp |= res > 0.f;
        const unsigned long long kr = pack_key(__fdiv_rn(res, E), v);
        const unsigned long long kp = pack_key(__fdiv_rn(p, E), v);
        best_res = kr > best_res ? kr : best_res;
        best_p = kp > best_p ? kp : best_p;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const unsigned long long b1 = __shfl_xor_sync(0xffffffffu, best_res, o);
      const unsigned long long b2 = __shfl_xor_sync(0xffffffffu, best_p, o);
      best_res = b1 > best_res ? b1 : best_res;
      best_p = b2 > best_p ? b2 : best_p;
    }
    anyp = __any_sync(0xffffffffu, anyp);
    if (lane == 0) {
      atomicMax(&ws.winners[2 * r], best_res);
      atomicMax(&ws.winners[2 * r + 1], best_p);
      if (anyp) atomicOr(&ws.any_pos[r], 1u);
    }
  }
  // last CTA of this request writes the outputs
  __shared__ bool s_last;
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    const unsigned done = atomicAdd(&ws.ticket[r], 1u);
    s_last = (done == (unsigned)plan.nchunk_b - 1u);
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  if (tid < B) {
    int tok = -1, pos = -1;
    if (tid < a) {
      pos = s_order[tid];
      tok = tokens[(size_t)r * B + pos];
    } else if (tid == a && a < gamma) {
      pos = s_order[a];
      const unsigned long long wr = atomicAdd(&ws.winners[2 * r], 0ull);
      const unsigned long long wp = atomicAdd(&ws.winners[2 * r + 1], 0ull);
      const unsigned ap = atomicAdd(&ws.any_pos[r], 0u);
      tok = unpack_token(ap ? wr : wp);
    }
    out_tokens[(size_t)r * B + tid] = tok;
    out_pos[(size_t)r * B + tid] = pos;
  }
  if (tid == 0) {
    accepted_len[r] = a;
    n_commit[r] = a + (a < gamma ? 1 : 0);
  }
}

}  // namespace

}  // namespace simsd

SIMSD_API size_t simsd_accept_workspace(int batch, int B, int gamma, int V) {
  if (batch < 0 || B < 1 || gamma < 1 || gamma > B || V < 1) return 0;
  return simsd::make_plan(batch, gamma, V).bytes;
}

SIMSD_API simsd_status simsd_accept(const float* target_logits, const float* draft_logits,
                                    const int32_t* draft_tokens, const uint8_t* labels,
                                    int batch, int B, int gamma, int V, float temperature,
                                    uint64_t seed, uint64_t offset, int32_t* accepted_len,
                                    int32_t* out_tokens, int32_t* out_pos, int32_t* n_commit,
                                    void* workspace, size_t workspace_bytes, uint32_t* dev_err,
                                    simsd_stream_t stream) {
  using namespace simsd;
  if (batch < 0 || B < 1 || B > kMaxB || gamma < 1 || gamma > B || V < 1)
    return SIMSD_ERR_INVALID_ARG;
  if (!(temperature >= 0.f)) return SIMSD_ERR_INVALID_ARG;
  if (temperature == 0.f) return SIMSD_ERR_UNSUPPORTED;
  if (batch == 0) return SIMSD_OK;
  if (!target_logits || !draft_logits || !draft_tokens || !labels || !accepted_len ||
      !out_tokens || !out_pos || !n_commit || !dev_err)
    return SIMSD_ERR_INVALID_ARG;
  if ((size_t)batch * B * (size_t)V >= ((size_t)1 << 40)) return SIMSD_ERR_UNSUPPORTED;
  const AcceptPlan plan = make_plan(batch, gamma, V);
  if (!workspace || workspace_bytes < plan.bytes || (((uintptr_t)workspace) & 255))
    return SIMSD_ERR_WORKSPACE;
  char* base = (char*)workspace;
  AcceptWs ws;
  ws.stats = (float2*)(base + plan.off_stats);
  ws.winners = (unsigned long long*)(base + plan.off_winners);
  ws.any_pos = (unsigned*)(base + plan.off_anypos);
  ws.ticket = (unsigned*)(base + plan.off_ticket);
  const long grid_a = (long)batch * gamma * 2 * plan.nchunk_a;
  const long grid_b = (long)batch * plan.nchunk_b;
  if (grid_a > 0x7fffffffL || grid_b > 0x7fffffffL) return SIMSD_ERR_UNSUPPORTED;
  cudaStream_t s = (cudaStream_t)stream;
  accept_stats_kernel<<<(unsigned)grid_a, kStatThreads, 0, s>>>(
      target_logits, draft_logits, labels, batch, B, gamma, V, temperature, plan, ws);
  simsd_status st = last_launch_status();
  if (st != SIMSD_OK) return st;
  accept_finish_kernel<<<(unsigned)grid_b, kFinishThreads, 0, s>>>(
      target_logits, draft_logits, draft_tokens, labels, batch, B, gamma, V, temperature,
      (uint32_t)(seed & 0xffffffffu), (uint32_t)(seed >> 32), (uint32_t)(offset & 0xffffffffu),
      (uint32_t)(offset >> 32), plan, ws, accepted_len, out_tokens, out_pos, n_commit, dev_err);
  return last_launch_status();
}

// ------------------------------------------------------------------------------------
// Allocation-free variant. Its scratch lives in a fixed device array of this file, so the
// caller passes only inputs and outputs. Every device that loads the library holds the
// array (kNoAllocScratchBytes) until the process exits.
namespace simsd {
namespace {
constexpr size_t kNoAllocScratchBytes = (size_t)1 << 20;  // 1 MiB
static __device__ __align__(256) unsigned char g_accept_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
void* g_scratch_ptr[kMaxDevices];

// Device address of g_accept_scratch on the current device. Resolved on the first call
// per device (with that device current) and cached; the host-side symbol itself is not a
// device address and is never passed to a kernel.
simsd_status noalloc_scratch(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    record_cuda_error("cudaGetDevice", e);
    return SIMSD_ERR_CUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) return SIMSD_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (!g_scratch_ptr[dev]) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_accept_scratch);
    if (e != cudaSuccess || !ptr) {
      record_cuda_error("cudaGetSymbolAddress", e != cudaSuccess ? e : cudaErrorInvalidSymbol);
      return SIMSD_ERR_CUDA;
    }
    g_scratch_ptr[dev] = ptr;
  }
  *out = g_scratch_ptr[dev];
  return SIMSD_OK;
}
}  // namespace
}  // namespace simsd

SIMSD_API size_t simsd_accept_noalloc_max_scratch(void) { return simsd::kNoAllocScratchBytes; }

SIMSD_API simsd_status simsd_accept_noalloc(const float* target_logits, const float* draft_logits,
                                            const int32_t* draft_tokens, const uint8_t* labels,
                                            int batch, int B, int gamma, int V, float temperature,
                                            uint64_t seed, uint64_t offset, int32_t* accepted_len,
                                            int32_t* out_tokens, int32_t* out_pos,
                                            int32_t* n_commit, uint32_t* dev_err,
                                            simsd_stream_t stream) {
  using namespace simsd;
  if (batch < 0 || B < 1 || B > kMaxB || gamma < 1 || gamma > B || V < 1)
    return SIMSD_ERR_INVALID_ARG;
  if (batch > 0 && make_plan(batch, gamma, V).bytes > kNoAllocScratchBytes)
    return SIMSD_ERR_WORKSPACE;  // these sizes need more scratch than the fixed array holds
  void* scratch = nullptr;
  if (batch > 0) {
    const simsd_status st = noalloc_scratch(&scratch);
    if (st != SIMSD_OK) return st;
  }
  return simsd_accept(target_logits, draft_logits, draft_tokens, labels, batch, B, gamma, V,
                      temperature, seed, offset, accepted_len, out_tokens, out_pos, n_commit,
                      scratch, kNoAllocScratchBytes, dev_err, stream);
}
