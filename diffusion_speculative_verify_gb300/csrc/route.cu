// Routing statistic of the verification step (sm_103a): the expected accepted-prefix
// length of every request,
//   K^ = sum_{k=1..L} prod_{i=1..k} alpha_i,   L = min(gamma, R),
// with a margin-based alpha_i = 1[m_i >= tau_margin] or an entropy-based
// alpha_i = exp(-beta H~_i) of the draft distribution p = softmax(z / T) at step i
// (S2D2 page, "方法步骤详情" step (4), the score policy of its routing algorithm).
// m_i = p_(1) - p_(2) and H~_i = H(p) / ln V.
//
// Two launches:
//   K4a  one warp per (verified draft row, chunk): a single streamed pass keeps the two
//        largest scaled logits m1 >= m2 and, relative to m1, S = sum e^(z - m1) and
//        W2 = sum e^(z - m1) (z - m1) log2(e). Then p_(1) = 1 / S, p_(2) = e^(m2 - m1) / S
//        and H = ln S - ln(2) W2 / S.
//   K4b  one CTA per request, a programmatic dependent of K4a: a warp merges the chunks
//        of a step across its lanes and forms alpha_i; K^ is a multiplicative prefix scan
//        and a sum over the steps.
#include <float.h>
#include <math.h>

#include <algorithm>

#include "common.cuh"
#include "logits.cuh"

namespace simsd {
namespace {

constexpr int kKhatThreads = 256;
constexpr int kKhatPer = 16;  // 16-byte loads in flight per lane

struct KhatPlan {
  int nchunk, chunk;  // chunks per row, entries per chunk (multiple of 8)
  size_t bytes;       // workspace: float4 (m1, m2, S, W) per (row, chunk)
};

int resident_khat_warps();

// Rows are cut into the smallest number of equal chunks whose work items fill the last
// round of the resident warps to at least 97 % (chunks of at least 512 entries).
KhatPlan make_khat_plan(int batch, int gamma, int V) {
  KhatPlan p;
  const long rows = (long)batch * gamma;
  const long W = std::max(1, resident_khat_warps());
  const long ncmax = std::max<long>(1, (V + 511) / 512);
  long best_nc = 1;
  double best_fill = -1.0;
  for (long nc = 1; nc <= ncmax && rows > 0; ++nc) {
    const long items = rows * nc;
    const long rounds = (items + W - 1) / W;
    const double fill = (double)items / (double)(rounds * W);
    if (fill > best_fill + 1e-9) {
      best_fill = fill;
      best_nc = nc;
    }
    if (fill >= 0.97) break;
  }
  p.chunk = (int)(((V + best_nc - 1) / best_nc + 7) / 8 * 8);
  p.nchunk = (V + p.chunk - 1) / p.chunk;
  p.bytes = std::max<size_t>(256, align_up((size_t)rows * p.nchunk * sizeof(float4), 256));
  return p;
}

// Running top two of a stream of values: a1 >= a2, a repeated maximum counts twice.
__device__ __forceinline__ void top2_add(float& a1, float& a2, float z) {
  a2 = fmaxf(a2, fminf(a1, z));
  a1 = fmaxf(a1, z);
}

__device__ __forceinline__ void top2_merge(float& a1, float& a2, float b1, float b2) {
  a2 = fmaxf(fmaxf(a2, b2), fminf(a1, b1));
  a1 = fmaxf(a1, b1);
}

// Top two of one batch of 16-byte loads, on the raw values (scaling by 1 / T is monotone,
// so the caller scales the two results). fp32: four independent accumulators (one per
// word of a load); bf16: the same on packed pairs with min/max.bf16x2, then the halves.
template <typename LT>
struct BatchTop2;

template <>
struct BatchTop2<float> {
  template <int K>
  static __device__ __forceinline__ float2 of(const uint4 (&x)[K]) {
    float a1[4], a2[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) a1[j] = a2[j] = -INFINITY;
#pragma unroll
    for (int u = 0; u < K; ++u)
#pragma unroll
      for (int j = 0; j < 4; ++j) top2_add(a1[j], a2[j], __uint_as_float(word_of(x[u], j)));
    top2_merge(a1[0], a2[0], a1[1], a2[1]);
    top2_merge(a1[2], a2[2], a1[3], a2[3]);
    top2_merge(a1[0], a2[0], a1[2], a2[2]);
    return make_float2(a1[0], a2[0]);
  }
};

template <>
struct BatchTop2<__nv_bfloat16> {
  static __device__ __forceinline__ uint32_t max2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
  }
  static __device__ __forceinline__ uint32_t min2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("min.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
  }
  template <int K>
  static __device__ __forceinline__ float2 of(const uint4 (&x)[K]) {
    using IO = LogitIO<__nv_bfloat16>;
    uint32_t a1[4], a2[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) a1[j] = a2[j] = IO::kNegInfWord;
#pragma unroll
    for (int u = 0; u < K; ++u)
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t w = word_of(x[u], j);
        a2[j] = max2(a2[j], min2(a1[j], w));
        a1[j] = max2(a1[j], w);
      }
    float m1 = -INFINITY, m2 = -INFINITY;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      top2_merge(m1, m2, IO::lo(a1[j]), IO::lo(a2[j]));
      top2_merge(m1, m2, IO::hi(a1[j]), IO::hi(a2[j]));
    }
    return make_float2(m1, m2);
  }
};

constexpr float kLog2e = 1.4426950408889634f;

// Row statistic relative to its maximum: (m1, m2, S = sum e^(z - m1),
// W2 = sum e^(z - m1) (z - m1) log2 e). Merging re-bases both parts on the larger maximum:
// a part with maximum m and offset d = (m - m1') log2 e contributes 2^d S and 2^d (W2 + d S).
__device__ __forceinline__ void stat_merge(float4& a, const float4& b) {
  const float n1 = fmaxf(a.x, b.x);
  const float n2 = fmaxf(fmaxf(a.y, b.y), fminf(a.x, b.x));
  float S = 0.f, W = 0.f;
  if (a.x != -INFINITY) {
    const float d = (a.x - n1) * kLog2e, f = exp2f(d);
    S = f * a.z;
    W = f * fmaf(d, a.z, a.w);
  }
  if (b.x != -INFINITY) {
    const float d = (b.x - n1) * kLog2e, f = exp2f(d);
    S = fmaf(f, b.z, S);
    W = fmaf(f, fmaf(d, b.z, b.w), W);
  }
  a = make_float4(n1, n2, S, W);
}

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ----------------------------------------------------------------------------- K4a
template <typename LT>
__global__ void __launch_bounds__(kKhatThreads, 2) khat_stats_kernel(
    const LT* __restrict__ draft, const uint8_t* __restrict__ labels, int batch, int B,
    int gamma, int V, float T, KhatPlan plan, float4* __restrict__ stats, uint32_t* __restrict__ err) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int lane = threadIdx.x & 31;
  const long warp_global = (long)blockIdx.x * (kKhatThreads / 32) + (threadIdx.x >> 5);
  const long nwarps = (long)gridDim.x * (kKhatThreads / 32);
  const int nchunk = plan.nchunk;
  const long items = (long)batch * gamma * nchunk;
  const bool unit_T = (T == 1.f);
  const bool vec_ok = stream_ok(V, draft, draft);
  constexpr int E = LogitIO<LT>::kVec;
  const uint4 neg_inf = make_uint4(LogitIO<LT>::kNegInfWord, LogitIO<LT>::kNegInfWord,
                                   LogitIO<LT>::kNegInfWord, LogitIO<LT>::kNegInfWord);
  for (long item = warp_global; item < items; item += nwarps) {
    const int chunk = (int)(item % nchunk);
    const long row = item / nchunk;
    const int step = (int)(row % gamma);
    const int r = (int)(row / gamma);
    // the data slot labelled step + 1 (none for an invalid request or a step past R)
    const bool lab_ok = chk((long long)r * 2 * B, 2 * B, (long long)batch * 2 * B, err);
    const uint8_t lb = lane < B && lab_ok ? labels[(size_t)r * 2 * B + lane] : (uint8_t)0;
    const unsigned hit = __ballot_sync(0xffffffffu, lane < B && !(lb & kSegMask) && (lb & 0x7F) == step + 1);
    float4 st = make_float4(-INFINITY, -INFINITY, 0.f, 0.f);
    const int c0 = chunk * plan.chunk;
    const int len = min(plan.chunk, V - c0);
    if (hit && len > 0 &&
        chk(((long long)r * B + (__ffs(hit) - 1)) * V + c0, len, (long long)batch * B * V, err)) {
      const LT* rowp = draft + ((size_t)r * B + (__ffs(hit) - 1)) * (size_t)V + c0;
      float s0 = 0.f, s1 = 0.f, w0 = 0.f, w1 = 0.f;  // relative to st.x
      if (vec_ok) {  // c0 is a multiple of 8: every load is 16-byte aligned
        const int nv = len / E;
        for (int base = 0; base < nv; base += 32 * kKhatPer) {
          uint4 x[kKhatPer];
#pragma unroll
          for (int u = 0; u < kKhatPer; ++u) {
            const int i = base + lane + 32 * u;
            x[u] = i < nv ? ld_stream16(rowp + (size_t)E * i) : neg_inf;
          }
          const float2 bt = BatchTop2<LT>::of(x);
          const float b1 = scale_logit(bt.x, T, unit_T), b2 = scale_logit(bt.y, T, unit_T);
          const float n1 = fmaxf(st.x, b1);
          st.y = fmaxf(fmaxf(st.y, b2), fminf(st.x, b1));
          if (n1 > st.x) {  // re-base what was summed so far on the new maximum
            if (st.x == -INFINITY) {
              s0 = s1 = w0 = w1 = 0.f;
            } else {
              const float d = (st.x - n1) * kLog2e, f = exp2f(d);
              w0 = f * fmaf(d, s0, w0);
              w1 = f * fmaf(d, s1, w1);
              s0 *= f;
              s1 *= f;
            }
            st.x = n1;
          }
          if (st.x != -INFINITY) {
            // offset of an entry in log2 units, d = z log2 e - m1 log2 e (one FMA; the
            // rounding of m1 log2 e is common to the whole row and cancels in p = 2^d / S)
            const float mL = st.x * kLog2e;
#pragma unroll
            for (int u = 0; u < kKhatPer; ++u)
#pragma unroll
              for (int j = 0; j < E; j += 2) {
                // a masked entry (-inf) has 2^d = 0; its offset is clamped so that 0 * d = 0
                const float d0 = fmaxf(fmaf(scale_logit(LogitIO<LT>::entry(x[u], j), T, unit_T), kLog2e, -mL), -FLT_MAX);
                const float d1 = fmaxf(fmaf(scale_logit(LogitIO<LT>::entry(x[u], j + 1), T, unit_T), kLog2e, -mL), -FLT_MAX);
                const float e0 = ex2_approx(d0), e1 = ex2_approx(d1);
                s0 += e0;
                s1 += e1;
                w0 = fmaf(e0, d0, w0);
                w1 = fmaf(e1, d1, w1);
              }
          }
        }
      } else {  // unaligned rows or V not a multiple of 8: one entry at a time
        float4 acc = st;
        for (int v = lane; v < len; v += 32) {
          const float z = scale_logit(LogitIO<LT>::ld1(rowp + v), T, unit_T);
          if (z == -INFINITY || z != z) continue;  // no probability mass
          stat_merge(acc, make_float4(z, -INFINITY, 1.f, 0.f));
        }
        st.x = acc.x;
        st.y = acc.y;
        s0 = acc.z;
        w0 = acc.w;
      }
      st.z = s0 + s1;
      st.w = w0 + w1;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      float4 other;
      other.x = __shfl_xor_sync(0xffffffffu, st.x, o);
      other.y = __shfl_xor_sync(0xffffffffu, st.y, o);
      other.z = __shfl_xor_sync(0xffffffffu, st.z, o);
      other.w = __shfl_xor_sync(0xffffffffu, st.w, o);
      stat_merge(st, other);
    }
    if (lane == 0 && chk(item, 1, items, err)) stats[item] = st;
  }
}

// ----------------------------------------------------------------------------- K4b
// One CTA per request, a programmatic dependent of K4a. The labels are checked before the
// grid-dependency wait; then warp w takes the steps w, w + 8, ...: its lanes load that
// step's chunk statistics side by side and merge them in a shuffle tree, so no lane walks
// the chunks one load after another. Warp 0 then scans the alphas.
constexpr int kFinishWarps = 8;

__global__ void __launch_bounds__(32 * kFinishWarps) khat_finish_kernel(
    const uint8_t* __restrict__ labels, int batch, int B, int gamma, int V, int mode,
    float tau_margin, float beta, KhatPlan plan, const float4* __restrict__ stats,
    float* __restrict__ khat, float* __restrict__ alpha_out, uint32_t* __restrict__ dev_err) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int r = blockIdx.x;
  // checked build: the request's labels, chunk statistics and outputs lie inside their
  // arrays (block-uniform; else the block does nothing)
  if (!chk(r, 1, batch, dev_err) || !chk((long long)r * 2 * B, 2 * B, (long long)batch * 2 * B, dev_err) ||
      !chk((long long)r * gamma * plan.nchunk, (long long)gamma * plan.nchunk,
           (long long)batch * gamma * plan.nchunk, dev_err))
    return;
  __shared__ float s_alpha[kMaxB];
  // open slots carry the labels 1..R (0: committed in an earlier round); every warp
  // reaches the same decision
  const uint8_t lb = lane < B ? labels[(size_t)r * 2 * B + lane] : 0;
  const int tau = lb & 0x7F;
  const bool ok_lane = lane >= B || (lb != kLabelInvalid && !(lb & kSegMask) && tau <= B);
  const int R = __popc(__ballot_sync(0xffffffffu, lane < B && tau != 0));
  const unsigned bit = (lane < B && tau >= 1 && tau <= B) ? (1u << (tau - 1)) : 0u;
  const unsigned cover = __reduce_or_sync(0xffffffffu, bit);
  const unsigned full = R == 32 ? 0xffffffffu : ((1u << R) - 1u);
  const bool perm = __all_sync(0xffffffffu, ok_lane) && cover == full;
  const int gr = min(gamma, R);  // steps estimated
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (!perm) {  // block-uniform
    if (threadIdx.x == 0) {
      atomicOr(dev_err, SIMSD_DEVERR_TAU);
      khat[r] = -1.f;
    }
    if (alpha_out && threadIdx.x < gamma) alpha_out[(size_t)r * gamma + threadIdx.x] = 0.f;
    return;
  }
  for (int t = warp; t < kMaxB; t += kFinishWarps) {
    float a = 0.f;  // alpha of step t + 1 (0 past gr)
    if (t < gr) {   // warp-uniform
      const float4* src = stats + ((size_t)r * gamma + t) * plan.nchunk;
      float4 st = make_float4(-INFINITY, -INFINITY, 0.f, 0.f);
      for (int c = lane; c < plan.nchunk; c += 32) stat_merge(st, src[c]);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        float4 other;
        other.x = __shfl_xor_sync(0xffffffffu, st.x, o);
        other.y = __shfl_xor_sync(0xffffffffu, st.y, o);
        other.z = __shfl_xor_sync(0xffffffffu, st.z, o);
        other.w = __shfl_xor_sync(0xffffffffu, st.w, o);
        stat_merge(st, other);
      }
      if (mode == SIMSD_KHAT_MARGIN) {
        // p_(1) - p_(2) = (1 - e^(m2 - m1)) / S
        const float margin = st.y == -INFINITY ? 1.f / st.z : -expm1f(st.y - st.x) / st.z;
        a = margin >= tau_margin ? 1.f : 0.f;
      } else {
        const float H = logf(st.z) - 0.69314718055994531f * (st.w / st.z);
        const float Hn = V > 1 ? fminf(fmaxf(H / logf((float)V), 0.f), 1.f) : 0.f;
        a = expf(-beta * Hn);
      }
    }
    if (lane == 0) s_alpha[t] = a;
  }
  __syncthreads();
  if (warp == 0) {
    // K^ = sum over steps of the inclusive prefix products (0 from step gr on)
    const float a = s_alpha[lane];
    float prod = a;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float v = __shfl_up_sync(0xffffffffu, prod, o);
      if (lane >= o) prod *= v;
    }
    float sum = prod;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    if (lane == 0) khat[r] = sum;
    if (alpha_out && lane < gamma) alpha_out[(size_t)r * gamma + lane] = a;
  }
}

int resident_khat_warps() {
  static int cache_f[64], cache_h[64];
  return std::min(resident_blocks(khat_stats_kernel<float>, kKhatThreads, cache_f),
                  resident_blocks(khat_stats_kernel<__nv_bfloat16>, kKhatThreads, cache_h)) *
         (kKhatThreads / 32);
}

template <typename LT>
simsd_status expected_prefix_impl(const LT* draft, const uint8_t* labels, int batch, int B, int gamma,
                                  int V, float T, int mode, float tau_margin, float beta, float* khat,
                                  float* alpha, void* workspace, size_t workspace_bytes,
                                  uint32_t* dev_err, cudaStream_t s) {
  const KhatPlan plan = make_khat_plan(batch, gamma, V);
  if (!workspace || workspace_bytes < plan.bytes || (((uintptr_t)workspace) & 255))
    return SIMSD_ERR_WORKSPACE;
  const long items = (long)batch * gamma * plan.nchunk;
  if (items > 0x7fffffffL) return SIMSD_ERR_UNSUPPORTED;
  float4* stats = (float4*)workspace;
  const long max_ctas = std::max(1, resident_khat_warps() / (kKhatThreads / 32));
  const long grid = std::max<long>(1, std::min<long>((items + kKhatThreads / 32 - 1) / (kKhatThreads / 32), max_ctas));
  khat_stats_kernel<LT><<<(unsigned)grid, kKhatThreads, 0, s>>>(draft, labels, batch, B, gamma, V, T, plan, stats,
                                                                dev_err);
  simsd_status st = last_launch_status();
  if (st != SIMSD_OK) return st;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3((unsigned)batch);
  cfg.blockDim = dim3(32 * kFinishWarps);
  cfg.stream = s;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, khat_finish_kernel, labels, batch, B, gamma, V, mode,
                                           tau_margin, beta, plan, (const float4*)stats, khat, alpha, dev_err);
  if (e != cudaSuccess) {
    record_cuda_error("cudaLaunchKernelEx(khat_finish_kernel)", e);
    return SIMSD_ERR_CUDA;
  }
  return last_launch_status();
}

}  // namespace
}  // namespace simsd

SIMSD_API size_t simsd_expected_prefix_workspace(int batch, int B, int gamma, int V) {
  using namespace simsd;
  if (batch < 0 || B < 1 || B > kMaxB || gamma < 1 || gamma > B || V < 1) return 0;
  return make_khat_plan(batch, gamma, V).bytes;
}

SIMSD_API simsd_status simsd_expected_prefix(const void* draft_logits, simsd_dtype logit_dtype,
                                             const uint8_t* labels, int batch, int B, int gamma, int V,
                                             float temperature, simsd_khat_mode mode, float tau_margin,
                                             float beta, float* khat, float* alpha, void* workspace,
                                             size_t workspace_bytes, uint32_t* dev_err,
                                             simsd_stream_t stream) {
  SIMSD_NVTX_RANGE("simsd_expected_prefix");
  using namespace simsd;
  if (batch < 0 || B < 1 || B > kMaxB || gamma < 1 || gamma > B || V < 1)
    return SIMSD_ERR_INVALID_ARG;
  if (!(temperature > 0.f) || !(beta >= 0.f) || tau_margin != tau_margin)
    return SIMSD_ERR_INVALID_ARG;
  if (mode != SIMSD_KHAT_MARGIN && mode != SIMSD_KHAT_ENTROPY) return SIMSD_ERR_INVALID_ARG;
  if (logit_dtype != SIMSD_DTYPE_FP32 && logit_dtype != SIMSD_DTYPE_BF16) return SIMSD_ERR_INVALID_ARG;
  if (batch == 0) return SIMSD_OK;
  if (!draft_logits || !labels || !khat || !dev_err) return SIMSD_ERR_INVALID_ARG;
  if ((size_t)batch * B * (size_t)V >= ((size_t)1 << 40)) return SIMSD_ERR_UNSUPPORTED;
  cudaStream_t s = (cudaStream_t)stream;
  if (logit_dtype == SIMSD_DTYPE_BF16)
    return expected_prefix_impl<__nv_bfloat16>((const __nv_bfloat16*)draft_logits, labels, batch, B, gamma, V,
                                               temperature, (int)mode, tau_margin, beta, khat, alpha,
                                               workspace, workspace_bytes, dev_err, s);
  return expected_prefix_impl<float>((const float*)draft_logits, labels, batch, B, gamma, V, temperature,
                                     (int)mode, tau_margin, beta, khat, alpha, workspace, workspace_bytes,
                                     dev_err, s);
}
