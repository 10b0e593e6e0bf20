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
//   K3b accept_finish   : one wave of CTAs, each an equal range of the batch's (request,
//                         group of 4 entries) pairs; per request touched, a CTA merges the chunk
//                         pairs, re-derives the accept decisions (cheap), and if a step was
//                         rejected runs the race over its groups of the rejected slot's rows;
//                         winners meet in a 64-bit atomicMax; the last CTA of the request
//                         (atomic ticket, no waiting) writes the outputs. K3a zeroes the
//                         winners and tickets at the start of every call.
#include <cudaTypedefs.h>
#include <float.h>

#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "logits.cuh"
#include "tc_ptx.cuh"

namespace simsd {

namespace {

constexpr int kStatThreads = 256;
constexpr int kFinishThreads = 256;

struct AcceptWs {
  float2* stats;                // [batch][gamma][2][nchunk]  (max, sum exp) per chunk
  unsigned long long* winners;  // [batch][2]  race winners: residual, target (0: no positive residual)
  unsigned* ticket;             // [batch]     CTAs of K3b finished
  long long n_stats;            // entries of `stats` (checked build)
  uint32_t* err;                // the call's error word
};

struct AcceptPlan {
  int nchunk_a, chunk_a;  // K3a: chunks per row, elements per chunk (multiple of 8)
  // K3b: CTAs, each a range of the (request, group of 4 entries) pairs: nb_b > 0, request r
  // takes CTAs r nb_b .. r nb_b + nb_b - 1, cg_b groups each (the last fewer); nb_b = 0,
  // equal ranges across request boundaries (stream-K)
  int ctas_b, nb_b, cg_b;
  size_t off_stats, off_winners, off_ticket, bytes;
};

// Warps of the stats kernel and CTAs of the finish kernel resident at once on the current
// device (occupancy query, cached per device).
int resident_stat_warps();
int resident_finish_ctas();

// K3a cuts every verified row into nchunk_a equal chunks, one work item per (row, chunk),
// and the items are dealt to the resident warps round-robin. nchunk_a is the smallest count
// whose items fill the warps' last round to at least 97 % (the kernel's time is set by the
// warps that take the most items), else the best fill; chunks stay at least 512 entries.
// K3b takes one wave of CTAs over the batch's (request, group of 4 entries) pairs, at least
// 256 groups each, so no CTA's range is empty and each request's CTAs are consecutive. When
// a whole number of CTAs per request fills at least 90 % of the resident slots, each CTA stays
// within one request; otherwise (e.g. batch 256 on 304 slots: one CTA each, 84 %) the ranges
// are equal and cross request boundaries, and a CTA that holds the end of one request and
// the start of the next sets both up in turn (the statistics merge of 2 gamma rows).
// `models` = 2 (target and draft rows: sampling) or 1 (target rows only: greedy).
AcceptPlan make_plan(int batch, int gamma, int V, int models = 2) {
  AcceptPlan p;
  const long rows = (long)batch * gamma * models;
  const long W = std::max(1, resident_stat_warps());
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
  p.chunk_a = (int)(((V + best_nc - 1) / best_nc + 7) / 8 * 8);  // 16-byte loads of bf16
  p.nchunk_a = (V + p.chunk_a - 1) / p.chunk_a;
  const long long ng = (V + 3) / 4, groups = (long long)batch * ng;
  const long long slots = std::max(1, resident_finish_ctas());
  const long long nb = batch > 0 ? std::min<long long>(slots / batch, (V + 1023) / 1024) : 0;
  if (nb >= 1 && 10 * batch * nb >= 9 * slots) {
    p.nb_b = (int)nb;
    p.cg_b = (int)((ng + nb - 1) / nb);
    p.ctas_b = (int)(batch * nb);
  } else {
    p.nb_b = 0;
    p.cg_b = 0;
    p.ctas_b = (int)std::max<long long>(1, std::min<long long>(slots, groups / 256));
  }
  size_t off = 0;
  p.off_stats = off;
  off = align_up(off + (size_t)batch * gamma * models * p.nchunk_a * sizeof(float2), 256);
  p.off_winners = off;
  off = align_up(off + (size_t)batch * 2 * sizeof(unsigned long long), 256);
  p.off_ticket = off;
  off = align_up(off + (size_t)batch * sizeof(unsigned), 256);
  p.bytes = off;
  return p;
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

// ----------------------------------------------------------------------------- K3a
// One warp per (row, chunk) work item; a persistent grid of warps strides over the items,
// so there is no block-level synchronisation. A lane streams its share of the chunk in
// batches of kPer 16-byte loads in flight, keeping a running (max, sum exp) across batches.
// exp is evaluated as 2^((x - m) * log2 e) with the ex2 instruction (about 2 ulp; the
// acceptance decisions use the accurate exp on single values).
constexpr int kPer = 16;  // 16-byte loads in flight per lane


template <typename LT>
// Two CTAs per SM: each lane holds 16 16-byte loads in flight (64 registers), and a third
// CTA would force spills.
__global__ void __launch_bounds__(kStatThreads, 2) accept_stats_kernel(
    const LT* __restrict__ target, const LT* __restrict__ draft,
    const uint8_t* __restrict__ labels, int batch, int B, int gamma, int V, float T,
    AcceptPlan plan, AcceptWs ws) {
  // K3b may be scheduled as SMs free up; it waits for this grid before it reads anything
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int lane = threadIdx.x & 31;
  const long warp_global = (long)blockIdx.x * (kStatThreads / 32) + (threadIdx.x >> 5);
  const long nwarps = (long)gridDim.x * (kStatThreads / 32);
  const int nchunk = plan.nchunk_a;
  const long items = (long)batch * gamma * 2 * nchunk;
  if (blockIdx.x == 0) {  // scratch of K3b starts at zero on every call
    for (int i = threadIdx.x; i < batch; i += blockDim.x) {
      if (!chk(2LL * i, 2, 2LL * batch, ws.err)) continue;
      ws.winners[2 * i] = 0ull;
      ws.winners[2 * i + 1] = 0ull;
      ws.ticket[i] = 0u;
    }
  }
  const bool unit_T = (T == 1.f);
  const bool vec_ok = stream_ok(V, target, draft);
  constexpr int E = LogitIO<LT>::kVec;
  const uint4 neg_inf = make_uint4(LogitIO<LT>::kNegInfWord, LogitIO<LT>::kNegInfWord,
                                   LogitIO<LT>::kNegInfWord, LogitIO<LT>::kNegInfWord);
  for (long item = warp_global; item < items; item += nwarps) {
    const int chunk = (int)(item % nchunk);
    const long row = item / nchunk;
    const int model = (int)(row & 1);
    const int step = (int)((row >> 1) % gamma);
    const int r = (int)((row >> 1) / gamma);
    const bool lab_ok = chk((long long)r * 2 * B, 2 * B, (long long)batch * 2 * B, ws.err);
    const uint8_t lb = lane < B && lab_ok ? labels[(size_t)r * 2 * B + lane] : (uint8_t)0;
    const unsigned hit = __ballot_sync(0xffffffffu, lane < B && !(lb & kSegMask) && (lb & 0x7F) == step + 1);
    float m = -INFINITY, sum = 0.f;
    const int c0 = chunk * plan.chunk_a;
    const int len = min(plan.chunk_a, V - c0);
    if (hit && len > 0 &&
        chk(((long long)r * B + (__ffs(hit) - 1)) * V + c0, len, (long long)batch * B * V, ws.err)) {
      const int k = __ffs(hit) - 1;
      const LT* rowp = (model ? draft : target) + ((size_t)r * B + k) * (size_t)V;
      if (vec_ok) {  // c0 is a multiple of 8: every 16-byte load is aligned
        const LT* src = rowp + c0;
        const int nv = len / E;
        // one batch of loads: its maximum first (x / T rounded is monotone in x, so the
        // batch maximum is scaled once), then one ex2 per entry against the running maximum
        auto reduce = [&](const auto& x, int K) {
          typename LogitIO<LT>::MaxAcc acc = LogitIO<LT>::max_init();
#pragma unroll
          for (int u = 0; u < K; ++u) acc = LogitIO<LT>::max_acc(acc, x[u]);
          const float mb = scale_logit(LogitIO<LT>::max_value(acc), T, unit_T);
          if (mb > m) {  // rescale what was summed so far to the new maximum
            sum = (m == -INFINITY) ? 0.f : sum * exp_shifted(m, mb);
            m = mb;
          }
          if (m != -INFINITY) {
            float s0 = 0.f, s1 = 0.f;
#pragma unroll
            for (int u = 0; u < K; ++u)
#pragma unroll
              for (int j = 0; j < E; j += 2) {
                s0 += exp_shifted(scale_logit(LogitIO<LT>::entry(x[u], j), T, unit_T), m);
                s1 += exp_shifted(scale_logit(LogitIO<LT>::entry(x[u], j + 1), T, unit_T), m);
              }
            sum += s0 + s1;
          }
        };
        if constexpr (sizeof(LT) == 2) {
          // bf16 (8 entries per load, twice the arithmetic per byte): two halves of kPer / 2
          // loads, one in flight while the other is reduced
          constexpr int H = kPer / 2, step = 32 * H;
          uint4 xa[H], xb[H];
          auto load = [&](uint4 (&x)[H], int base) {
#pragma unroll
            for (int u = 0; u < H; ++u) {
              const int i = base + lane + 32 * u;
              x[u] = i < nv ? ld_stream16(src + (size_t)E * i) : neg_inf;
            }
          };
          load(xa, 0);
          for (int base = 0; base < nv; base += 2 * step) {
            if (base + step < nv) load(xb, base + step);
            reduce(xa, H);
            if (base + step >= nv) break;
            if (base + 2 * step < nv) load(xa, base + 2 * step);
            reduce(xb, H);
          }
        } else {  // fp32: batches of kPer loads per lane in flight
          for (int base = 0; base < nv; base += 32 * kPer) {
            uint4 x[kPer];
#pragma unroll
            for (int u = 0; u < kPer; ++u) {
              const int i = base + lane + 32 * u;
              x[u] = i < nv ? ld_stream16(src + (size_t)E * i) : neg_inf;
            }
            reduce(x, kPer);
          }
        }
      } else {
        for (int v = lane; v < len; v += 32) {
          const float z = scale_logit(LogitIO<LT>::ld1(rowp + c0 + v), T, unit_T);
          if (z > m) {
            sum = (m == -INFINITY) ? 0.f : sum * exp_shifted(m, z);
            m = z;
          }
          sum += exp_shifted(z, m);
        }
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
      const float s2 = __shfl_xor_sync(0xffffffffu, sum, o);
      lse_merge(m, sum, m2, s2);
    }
    if (lane == 0 && chk(item, 1, ws.n_stats, ws.err))
      ws.stats[item] = make_float2(m, sum);  // items enumerate [row][chunk]
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

// -ln(u) for u in (0, 1) to a few ulp relative. The race winners sit where u is close to 1
// and -ln(u) tiny, where the lg2 instruction's absolute error (about 2^-22) would be a large
// relative one; there (u >= 1/2) the identity -ln(u) = 2 atanh(s), s = (1 - u) / (1 + u) in
// (0, 1/3], is summed as an odd series up to s^13 (truncation below 2e-8 relative; 1 - u is
// exact). Below 1/2 the result is at least ln 2 and lg2's absolute error is harmless.
__device__ __forceinline__ float neg_log_uniform(float u) {
  float y;  // both forms, then a select: no divergence between the lanes of a warp
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(u));
  const float below = y * -0.6931471805599453f;
  const float sv = __fdividef(1.f - u, 1.f + u);
  const float s2 = sv * sv;
  float poly = 2.f / 13.f;
  poly = fmaf(poly, s2, 2.f / 11.f);
  poly = fmaf(poly, s2, 2.f / 9.f);
  poly = fmaf(poly, s2, 2.f / 7.f);
  poly = fmaf(poly, s2, 2.f / 5.f);
  poly = fmaf(poly, s2, 2.f / 3.f);
  poly = fmaf(poly, s2, 2.f);
  return u < 0.5f ? below : sv * poly;
}

// Race keys of the 4 entries of counter group g (entries 4g .. 4g + 3 below `end`) on the
// residual max(0, p - q), or on p when `on_p`. p and q use the ex2 instruction (a few ulp),
// which moves a key by about 1e-6 relative: only a race whose two best keys are that close
// can change winner.
__device__ __forceinline__ void race_group(int g, int end, const float (&t)[4], const float (&d)[4],
                                           float T, bool unit_T, float mt, float inv_st, float md,
                                           float inv_sd, bool on_p, uint32_t r, uint32_t off_lo,
                                           uint32_t off_hi, uint32_t key0, uint32_t key1,
                                           unsigned long long& best) {
  float key[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    // p and q rounded on their own (no fused multiply-add into p - q): where the two agree
    // in fp32 the residual is exactly 0, not the rounding error of q
    const float p = __fmul_rn(exp_shifted(scale_logit(t[j], T, unit_T), mt), inv_st);
    if (on_p) {
      key[j] = p;
    } else {
      const float q = __fmul_rn(exp_shifted(scale_logit(d[j], T, unit_T), md), inv_sd);
      key[j] = __fsub_rn(p, q);
    }
    if (4 * g + j >= end) key[j] = on_p ? -1.f : 0.f;
  }
  // no branch around the counter block: the groups of a batch then run their Philox
  // rounds side by side (the few groups without a positive key are drawn for nothing)
  Philox4 c4 = {r, off_lo, off_hi, kResampleTag | (uint32_t)g};
  const Philox4 rnd = philox4x32_10(c4, key0, key1);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float E = neg_log_uniform(word_to_uniform(philox_word(rnd, j)));
    const unsigned long long kr = pack_key(__fdividef(key[j], E), 4 * g + j);
    const bool take = key[j] > 0.f || (on_p && key[j] >= 0.f);
    best = (take && kr > best) ? kr : best;
  }
}

// Race over entries [c0, c1) (c0 a multiple of 4) of one target row (and draft row unless
// `on_p`), by `nthreads` threads with thread index `t`: four counter groups' loads in
// flight per thread at a time.
template <typename LT>
__device__ __forceinline__ void race_range(const LT* __restrict__ trow, const LT* __restrict__ drow,
                                           int c0, int c1, int t, int nthreads, bool vec_ok,
                                           float T, bool unit_T, float mt, float inv_st, float md,
                                           float inv_sd, bool on_p, uint32_t r, uint32_t off_lo,
                                           uint32_t off_hi, uint32_t key0, uint32_t key1,
                                           unsigned long long& best) {
  using IO = LogitIO<LT>;
  const int g0 = c0 / 4, g1 = c0 < c1 ? (c1 + 3) / 4 : g0;
  for (int gb = g0 + t; gb < g1; gb += 4 * nthreads) {
    // entries as loaded (aligned rows: one load per row and group; unaligned rows: one per
    // entry), widened only where they are used, after every load of the batch is issued
    typename IO::Raw4 rt[4], rd[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int g = gb + u * nthreads;
      if (g < g1) {
        rt[u] = vec_ok ? IO::ldraw4(trow, g) : IO::ldraw4_each(trow, g, c1);
        if (!on_p) rd[u] = vec_ok ? IO::ldraw4(drow, g) : IO::ldraw4_each(drow, g, c1);
      }
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int g = gb + u * nthreads;
      if (g < g1) {
        const float4 a = IO::widen4(rt[u]);
        const float4 b = on_p ? a : IO::widen4(rd[u]);
        const float tv[4] = {a.x, a.y, a.z, a.w}, dv[4] = {b.x, b.y, b.z, b.w};
        race_group(g, c1, tv, dv, T, unit_T, mt, inv_st, md, inv_sd, on_p, r, off_lo, off_hi,
                   key0, key1, best);
      }
    }
  }
}

// Two CTAs per SM (the grid is one wave of them). The (request, counter group) pairs,
// request-major, are cut into one contiguous range per CTA (the plan: a whole number of CTAs
// per request, or equal ranges across request boundaries, stream-K style, where whole CTAs
// would leave slots idle). A CTA takes the requests its range touches in turn: for each it
// re-derives the decisions and races its groups of the rejected slot; the CTAs touching a
// request count themselves on its ticket, and the last one writes its outputs.
template <typename LT>
__global__ void __launch_bounds__(kFinishThreads, 2) accept_finish_kernel(
    const LT* __restrict__ target, const LT* __restrict__ draft,
    const int32_t* __restrict__ tokens, const uint8_t* __restrict__ labels, int batch, int B,
    int gamma, int V, float T, uint32_t key0, uint32_t key1, uint32_t off_lo, uint32_t off_hi,
    AcceptPlan plan, AcceptWs ws, int32_t* __restrict__ accepted_len,
    int32_t* __restrict__ out_tokens, int32_t* __restrict__ out_pos,
    int32_t* __restrict__ n_commit, uint32_t* __restrict__ dev_err) {
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const bool unit_T = (T == 1.f);
  const int ng = (V + 3) / 4;  // counter groups of a row
  // this CTA's range [f0, f1) of the flattened groups r * ng + g and the requests it touches,
  // [r_lo, r_hi] (whole CTAs per request: one, found without a 64-bit division)
  long long f0, f1;
  int r_lo, r_hi;
  if (plan.nb_b > 0) {
    const int rq = blockIdx.x / plan.nb_b, ch = blockIdx.x - rq * plan.nb_b;
    f0 = (long long)rq * ng + (long long)ch * plan.cg_b;
    f1 = (long long)rq * ng + min((long long)ng, (long long)(ch + 1) * plan.cg_b);
    r_lo = r_hi = rq;
  } else {
    const long long F = (long long)batch * ng;
    f0 = (long long)blockIdx.x * F / gridDim.x;
    f1 = ((long long)blockIdx.x + 1) * F / gridDim.x;
    r_lo = (int)(f0 / ng);
    r_hi = f1 > f0 ? (int)((f1 - 1) / ng) : r_lo - 1;
  }
  // CTAs whose ranges touch request r, less one (stream-K: the CTA holding flattened group f
  // is the largest c with c F / C <= f)
  auto others = [&](int r) -> unsigned {
    if (plan.nb_b > 0) return (unsigned)(plan.nb_b - 1);
    const long long F = (long long)batch * ng;
    auto cta_of = [&](long long f) { return ((f + 1) * gridDim.x + F - 1) / F - 1; };
    return (unsigned)(cta_of((long long)r * ng + ng - 1) - cta_of((long long)r * ng));
  };

  __shared__ int s_order[kMaxB];
  __shared__ int s_a, s_bad, s_gr;
  __shared__ float s_mt, s_st, s_md, s_sd;
  __shared__ float2 s_rowstat[2 * kMaxB];  // merged (max, sum exp) per (step, model)
  __shared__ bool s_last;
  __shared__ unsigned long long s_win;

  bool waited = false;
  for (int r = r_lo; r <= r_hi && r < batch; ++r) {
    const long long rbase = (long long)r * ng;
    const int g_lo = (int)(max(f0, rbase) - rbase), g_hi = (int)(min(f1, rbase + ng) - rbase);
    if (waited) __syncthreads();  // the previous request's shared state has been read
    // checked build: the request's labels, tokens, outputs, scratch and chunk statistics lie
    // inside their arrays (block-uniform; else the request is skipped)
    const bool req_ok =
        chk(r, 1, batch, dev_err) && chk((long long)r * 2 * B, 2 * B, (long long)batch * 2 * B, dev_err) &&
        chk((long long)r * B, B, (long long)batch * B, dev_err) &&
        chk((long long)r * gamma * 2 * plan.nchunk_a, (long long)gamma * 2 * plan.nchunk_a, ws.n_stats, dev_err);
    const uint8_t* lab = labels + (size_t)r * 2 * B;

    // Everything that does not read K3a's results comes before the grid dependency wait, so
    // it overlaps K3a's last items: warp 0 checks the step labels, orders the steps, and loads
    // each verified step's draft token, the two logits at that token and its uniform.
    int bad_w = 0, k_w = 0, x_w = 0;  // warp 0: error bits, slot and token of step `lane`
    int gr_w = gamma;                 // warp 0: steps verified, min(gamma, R)
    float tx = 0.f, dx = 0.f, u = 0.f;
    if (w == 0 && req_ok) {
      // step labels of the data half -> order o_t; validity of the permutation
      // labels 1..R of the open slots (0: committed in an earlier round) -> order o_t
      const uint8_t lb = lane < B ? lab[lane] : 0;
      const int tau = lb & 0x7F;
      const bool ok_lane = lane >= B || (lb != kLabelInvalid && !(lb & kSegMask) && tau <= B);
      const int R = __popc(__ballot_sync(0xffffffffu, lane < B && tau != 0));
      const unsigned bit = (lane < B && tau >= 1 && tau <= B) ? (1u << (tau - 1)) : 0u;
      const unsigned cover = __reduce_or_sync(0xffffffffu, bit);
      const unsigned full = R == 32 ? 0xffffffffu : ((1u << R) - 1u);
      const bool perm = __all_sync(0xffffffffu, ok_lane) && cover == full;
      if (perm && lane < B && tau != 0) s_order[tau - 1] = lane;
      __syncwarp();
      bad_w = perm ? 0 : (int)SIMSD_DEVERR_TAU;
      gr_w = min(gamma, R);
      if (perm && lane < gr_w) {
        k_w = s_order[lane];
        x_w = tokens[(size_t)r * B + k_w];
      }
      const bool tok_bad = perm && lane < gr_w && (x_w < 0 || x_w >= V);
      if (__any_sync(0xffffffffu, tok_bad)) bad_w |= (int)SIMSD_DEVERR_TOKEN;
      if (!bad_w && lane < gr_w && chk(((long long)r * B + k_w) * V + x_w, 1, (long long)batch * B * V, dev_err)) {
        const size_t rowoff = ((size_t)r * B + k_w) * (size_t)V + x_w;
        tx = scale_logit(LogitIO<LT>::ld1(target + rowoff), T, unit_T);
        dx = scale_logit(LogitIO<LT>::ld1(draft + rowoff), T, unit_T);
        Philox4 c4 = {(uint32_t)r, off_lo, off_hi, (uint32_t)(lane >> 2)};
        const Philox4 rnd = philox4x32_10(c4, key0, key1);
        u = word_to_uniform(philox_word(rnd, lane & 3));
      }
    }

    // launched as a programmatic dependent of K3a: wait for K3a's results before reading them
    if (!waited) asm volatile("griddepcontrol.wait;" ::: "memory");
    waited = true;
    if (!req_ok) continue;

    // merge the chunk partials of every verified (step, model) row: warp w takes rows
    // w, w + 8, ...; all of a warp's loads are issued before any is reduced
    constexpr int kWarps = kFinishThreads / 32;
    constexpr int kRowsPerWarp = (2 * kMaxB + kWarps - 1) / kWarps;
    const float2* rstats = ws.stats + (size_t)r * gamma * 2 * plan.nchunk_a;
    for (int c0 = 0; c0 < plan.nchunk_a; c0 += 32) {
      float2 v[kRowsPerWarp];
#pragma unroll
      for (int i = 0; i < kRowsPerWarp; ++i) {
        const int row = w + kWarps * i, c = c0 + lane;
        v[i] = (row < 2 * gamma && c < plan.nchunk_a) ? rstats[(size_t)row * plan.nchunk_a + c]
                                                     : make_float2(-INFINITY, 0.f);
      }
#pragma unroll
      for (int i = 0; i < kRowsPerWarp; ++i) {
        const int row = w + kWarps * i;
        if (row >= 2 * gamma) break;  // warp-uniform
        float m = v[i].x, sum = v[i].y;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
          const float s2 = __shfl_xor_sync(0xffffffffu, sum, o);
          lse_merge(m, sum, m2, s2);
        }
        if (lane == 0) {
          if (c0 == 0) {
            s_rowstat[row] = make_float2(m, sum);
          } else {  // more than 32 chunks: fold into the earlier ones
            float mm = s_rowstat[row].x, ss = s_rowstat[row].y;
            lse_merge(mm, ss, m, sum);
            s_rowstat[row] = make_float2(mm, ss);
          }
        }
      }
    }
    __syncthreads();

    if (w == 0) {
      int a = gr_w;
      if (!bad_w) {
        bool acc = true;
        float mt = 0.f, st = 0.f, md = 0.f, sd = 0.f;
        if (lane < gr_w) {
          const float2 rt = s_rowstat[2 * lane], rd = s_rowstat[2 * lane + 1];
          mt = rt.x;
          st = rt.y;
          md = rd.x;
          sd = rd.y;
          const float px = __fdiv_rn(expf(tx - mt), st);
          const float qx = __fdiv_rn(expf(dx - md), sd);
          acc = (px >= qx) || (u * qx < px);
        }
        const unsigned rej = __ballot_sync(0xffffffffu, lane < gr_w && !acc);
        a = rej ? (__ffs(rej) - 1) : gr_w;
        if (a < gr_w && lane == a) {
          s_mt = mt;
          s_st = st;
          s_md = md;
          s_sd = sd;
        }
      }
      if (lane == 0) {
        s_a = a;
        s_bad = bad_w;
        s_gr = gr_w;
      }
    }
    __syncthreads();
    const int a = s_a;
    const int bad = s_bad;
    const int gr = s_gr;  // steps this request verifies
    if (bad) {  // sentinel outputs, by the CTA holding the request's first group
      if (g_lo == 0) {
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
      continue;
    }

    if (a < gr) {
      // exponential race over this CTA's groups of the rejected slot's vocabulary
      const int k = s_order[a];
      const float mt = s_mt, st = s_st, md = s_md, sd = s_sd;
      const LT* trow = target + ((size_t)r * B + k) * (size_t)V;
      const LT* drow = draft + ((size_t)r * B + k) * (size_t)V;
      const int c0 = 4 * g_lo;
      const int c1 = min(V, 4 * g_hi);
      unsigned long long best_res = 0ull;
      const bool vec_ok = (V & 3) == 0 && ((((uintptr_t)target) | ((uintptr_t)draft)) & (LogitIO<LT>::kAlign - 1)) == 0;
      if (chk(((long long)r * B + k) * V + min(c0, V), c1 - min(c0, V), (long long)batch * B * V, dev_err))
        race_range(trow, drow, min(c0, V), c1, tid, blockDim.x, vec_ok, T, unit_T, mt, 1.f / st, md,
                   1.f / sd, false, (uint32_t)r, off_lo, off_hi, key0, key1, best_res);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const unsigned long long b1 = __shfl_xor_sync(0xffffffffu, best_res, o);
        best_res = b1 > best_res ? b1 : best_res;
      }
      // a residual entry is taken only where it is positive, and its packed key is then
      // nonzero: a winner word still 0 at the end means the residual vanished everywhere
      if (lane == 0 && best_res != 0ull) atomicMax(&ws.winners[2 * r], best_res);
    }
    // last CTA of this request writes the outputs
    __syncthreads();
    if (tid == 0) {
      __threadfence();
      const unsigned done = atomicAdd(&ws.ticket[r], 1u);
      s_last = (done == others(r));
    }
    __syncthreads();
    if (!s_last) continue;
    __threadfence();
    if (tid == 0) s_win = atomicAdd(&ws.winners[2 * r], 0ull);
    __syncthreads();
    if (a < gr && s_win == 0ull) {
      // the residual vanished in fp32 everywhere (p equal to q up to rounding): race on p
      // over the whole row, done here by the last CTA (never on typical inputs)
      const int k = s_order[a];
      const LT* trow = target + ((size_t)r * B + k) * (size_t)V;
      unsigned long long best = 0ull;
      const bool vec_ok = (V & 3) == 0 && ((((uintptr_t)target) | ((uintptr_t)draft)) & (LogitIO<LT>::kAlign - 1)) == 0;
      if (chk(((long long)r * B + k) * V, V, (long long)batch * B * V, dev_err))
        race_range(trow, trow, 0, V, tid, blockDim.x, vec_ok, T, unit_T, s_mt, 1.f / s_st, s_md,
                   1.f / s_sd, true, (uint32_t)r, off_lo, off_hi, key0, key1, best);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const unsigned long long b1 = __shfl_xor_sync(0xffffffffu, best, o);
        best = b1 > best ? b1 : best;
      }
      if (lane == 0) atomicMax(&s_win, best);
      __syncthreads();
    }
    if (tid < B) {
      int tok = -1, pos = -1;
      if (tid < a) {
        pos = s_order[tid];
        tok = tokens[(size_t)r * B + pos];
      } else if (tid == a && a < gr) {
        pos = s_order[a];
        tok = unpack_token(s_win);
      }
      out_tokens[(size_t)r * B + tid] = tok;
      out_pos[(size_t)r * B + tid] = pos;
    }
    if (tid == 0) {
      accepted_len[r] = a;
      n_commit[r] = a + (a < gr ? 1 : 0);
    }
  }
}

// ------------------------------------------------------------------ greedy (T = 0)
// Greedy verification (SPOT page, Algorithm 2, verification at T = 0): the target's own
// choice at a slot is its first largest logit; a step is accepted iff the draft token is
// that choice, and at the first mismatch the choice is committed. Two launches: an argmax
// pass over the verified target rows (one warp per (row, chunk) item, (max, first index)
// per chunk) and a finish kernel with one warp per request.
constexpr int kArgmaxThreads = 256;
constexpr int kNoIndex = 0x7fffffff;

// (value, index) of the first maximum: a larger value wins, an equal one the smaller index.
__device__ __forceinline__ void argmax_merge(float& m, int& i, float m2, int i2) {
  if (i2 == kNoIndex) return;
  if (i == kNoIndex || m2 > m || (m2 == m && i2 < i)) {
    m = m2;
    i = i2;
  }
}

// Key of entry v: the logit at T = 0 (greedy); with `noise`, the coupled-noise key
// logit / T + G_{a,v}, G = -ln(-ln u) with u from the counter (request, absolute position
// a, offset lo, kNoiseTag | v/4), word v % 4 (SPOT page, Gumbel-max and coupling section).
struct NoiseKey {
  bool on;
  float inv_T;  // 1 / T
  uint32_t key0, key1, off_lo;
};

// logit / T - ln(E), E = -ln(u): -ln(u) to a few ulp relative (the winners sit at u near
// 1, E small), its logarithm and the 1 / T scaling to about 1e-6 absolute; keys closer
// than that are near-ties.
__device__ __forceinline__ float noise_key(float logit, float inv_T, uint32_t word) {
  const float E = neg_log_uniform(word_to_uniform(word));
  return fmaf(logit, inv_T, -__logf(E));
}

template <typename LT>
__global__ void __launch_bounds__(kArgmaxThreads) accept_argmax_kernel(
    const LT* __restrict__ target, const uint8_t* __restrict__ labels,
    const int32_t* __restrict__ pos_ids, int batch, int B, int gamma, int V, AcceptPlan plan,
    AcceptWs ws, NoiseKey nk) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int lane = threadIdx.x & 31;
  const long warp_global = (long)blockIdx.x * (kArgmaxThreads / 32) + (threadIdx.x >> 5);
  const long nwarps = (long)gridDim.x * (kArgmaxThreads / 32);
  const int nchunk = plan.nchunk_a;
  const long items = (long)batch * gamma * nchunk;
  const bool vec_ok = stream_ok(V, target, target);
  constexpr int E = LogitIO<LT>::kVec;
  const uint4 neg_inf = make_uint4(LogitIO<LT>::kNegInfWord, LogitIO<LT>::kNegInfWord,
                                   LogitIO<LT>::kNegInfWord, LogitIO<LT>::kNegInfWord);
  for (long item = warp_global; item < items; item += nwarps) {
    const int chunk = (int)(item % nchunk);
    const long row = item / nchunk;
    const int step = (int)(row % gamma);
    const int r = (int)(row / gamma);
    const bool lab_ok = chk((long long)r * 2 * B, 2 * B, (long long)batch * 2 * B, ws.err);
    const uint8_t lb = lane < B && lab_ok ? labels[(size_t)r * 2 * B + lane] : (uint8_t)0;
    const unsigned hit = __ballot_sync(0xffffffffu, lane < B && !(lb & kSegMask) && (lb & 0x7F) == step + 1);
    float m = -INFINITY;
    int mi = kNoIndex;
    const int c0 = chunk * plan.chunk_a;
    const int len = min(plan.chunk_a, V - c0);
    if (hit && len > 0 &&
        chk(((long long)r * B + (__ffs(hit) - 1)) * V + c0, len, (long long)batch * B * V, ws.err)) {
      const int slot = __ffs(hit) - 1;
      const LT* rowp = target + ((size_t)r * B + slot) * (size_t)V + c0;
      const uint32_t apos = nk.on ? (uint32_t)pos_ids[(size_t)r * 2 * B + slot] : 0u;
      // a lane visits its entries in increasing index, so a strict '>' keeps the first
      // maximum (the first non-NaN entry starts the scan, even at -inf)
      if (vec_ok) {  // batches of 16 16-byte loads per lane in flight (c0 is a multiple of 8)
        constexpr int kPerA = 16;
        const int nv = len / E;
        for (int base = 0; base < nv; base += 32 * kPerA) {
          uint4 x[kPerA];
#pragma unroll
          for (int u = 0; u < kPerA; ++u) {
            const int i = base + lane + 32 * u;
            x[u] = i < nv ? ld_stream16(rowp + (size_t)E * i) : neg_inf;
          }
          if (!nk.on) {
            // greedy keys: the batch maximum first (padding is -inf); the first index of it
            // is looked up only when it raises the running maximum (or starts the scan),
            // which keeps the first maximum as the per-entry scan does
            typename LogitIO<LT>::MaxAcc acc = LogitIO<LT>::max_init();
#pragma unroll
            for (int u = 0; u < kPerA; ++u) acc = LogitIO<LT>::max_acc(acc, x[u]);
            const float mb = LogitIO<LT>::max_value(acc);
            if (mb > m || (mi == kNoIndex && mb == mb)) {
              int first = kNoIndex;
#pragma unroll
              for (int u = kPerA - 1; u >= 0; --u) {  // backwards: the last hit is the first index
                const int i = base + lane + 32 * u;
#pragma unroll
                for (int j = E - 1; j >= 0; --j)
                  if (i < nv && LogitIO<LT>::entry(x[u], j) == mb) first = c0 + E * i + j;
              }
              if (first != kNoIndex) {
                m = mb;
                mi = first;
              }
            }
            continue;
          }
#pragma unroll
          for (int u = 0; u < kPerA; ++u) {
            const int i = base + lane + 32 * u;
            if (i >= nv) break;
#pragma unroll
            for (int g = 0; g < E / 4; ++g) {  // groups of 4 entries: one counter block each
              const int v0 = c0 + E * i + 4 * g;
              float xv[4];
#pragma unroll
              for (int j = 0; j < 4; ++j) xv[j] = LogitIO<LT>::entry(x[u], 4 * g + j);
              if (nk.on) {
                Philox4 c4 = {(uint32_t)r, apos, nk.off_lo, kNoiseTag | (uint32_t)(v0 >> 2)};
                const Philox4 rnd = philox4x32_10(c4, nk.key0, nk.key1);
#pragma unroll
                for (int j = 0; j < 4; ++j) xv[j] = noise_key(xv[j], nk.inv_T, philox_word(rnd, j));
              }
#pragma unroll
              for (int j = 0; j < 4; ++j)
                if (xv[j] > m || (mi == kNoIndex && xv[j] == xv[j])) {
                  m = xv[j];
                  mi = v0 + j;
                }
            }
          }
        }
      } else {
        for (int v = lane; v < len; v += 32) {
          float x = LogitIO<LT>::ld1(rowp + v);
          if (nk.on) {
            const int gv = c0 + v;
            Philox4 c4 = {(uint32_t)r, apos, nk.off_lo, kNoiseTag | (uint32_t)(gv >> 2)};
            x = noise_key(x, nk.inv_T, philox_word(philox4x32_10(c4, nk.key0, nk.key1), gv & 3));
          }
          if (x > m || (mi == kNoIndex && x == x)) {
            m = x;
            mi = c0 + v;
          }
        }
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
      const int i2 = __shfl_xor_sync(0xffffffffu, mi, o);
      argmax_merge(m, mi, m2, i2);
    }
    if (lane == 0 && chk(item, 1, ws.n_stats, ws.err)) ws.stats[item] = make_float2(m, __int_as_float(mi));
  }
}

// One warp per request; launched as a programmatic dependent of the argmax pass.
__global__ void __launch_bounds__(256) accept_greedy_finish_kernel(
    const int32_t* __restrict__ tokens, const uint8_t* __restrict__ labels, int batch, int B,
    int gamma, int V, AcceptPlan plan, AcceptWs ws, int32_t* __restrict__ accepted_len,
    int32_t* __restrict__ out_tokens, int32_t* __restrict__ out_pos,
    int32_t* __restrict__ n_commit, uint32_t* __restrict__ dev_err) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int r = blockIdx.x * 8 + w;
  __shared__ int s_order[8][kMaxB];
  // labels, order and draft tokens before the grid dependency wait (they are not the
  // argmax pass's results)
  int bad = 0, k = 0, x = 0, gr = gamma;  // gr: steps verified, min(gamma, R)
  // checked build: the request's labels, tokens, outputs and chunk results lie inside their
  // arrays (warp-uniform; else the warp does nothing)
  const bool rows_ok = r >= batch ||
                       (chk((long long)r * 2 * B, 2 * B, (long long)batch * 2 * B, dev_err) &&
                        chk((long long)r * B, B, (long long)batch * B, dev_err) &&
                        chk((long long)r * gamma * plan.nchunk_a, (long long)gamma * plan.nchunk_a, ws.n_stats, dev_err));
  if (r < batch && rows_ok) {
    // labels 1..R of the open slots (0: committed in an earlier round) -> order o_t
    const uint8_t lb = lane < B ? labels[(size_t)r * 2 * B + lane] : 0;
    const int tau = lb & 0x7F;
    const bool ok_lane = lane >= B || (lb != kLabelInvalid && !(lb & kSegMask) && tau <= B);
    const int R = __popc(__ballot_sync(0xffffffffu, lane < B && tau != 0));
    const unsigned bit = (lane < B && tau >= 1 && tau <= B) ? (1u << (tau - 1)) : 0u;
    const unsigned cover = __reduce_or_sync(0xffffffffu, bit);
    const unsigned full = R == 32 ? 0xffffffffu : ((1u << R) - 1u);
    const bool perm = __all_sync(0xffffffffu, ok_lane) && cover == full;
    if (perm && lane < B && tau != 0) s_order[w][tau - 1] = lane;
    __syncwarp();
    bad = perm ? 0 : (int)SIMSD_DEVERR_TAU;
    gr = min(gamma, R);
    if (perm && lane < gr) {
      k = s_order[w][lane];
      x = tokens[(size_t)r * B + k];
    }
    if (__any_sync(0xffffffffu, perm && lane < gr && (x < 0 || x >= V))) bad |= (int)SIMSD_DEVERR_TOKEN;
  }
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (r >= batch || !rows_ok) return;  // warp-uniform
  if (bad) {
    if (lane == 0) {
      atomicOr(dev_err, (uint32_t)bad);
      accepted_len[r] = -1;
      n_commit[r] = 0;
    }
    if (lane < B) {
      out_tokens[(size_t)r * B + lane] = -1;
      out_pos[(size_t)r * B + lane] = -1;
    }
    return;
  }
  // lane t < gamma: the target's choice at step t, merged over the row's chunks
  float m = -INFINITY;
  int choice = kNoIndex;
  if (lane < gr) {
    const float2* src = ws.stats + ((size_t)r * gamma + lane) * plan.nchunk_a;
    for (int c = 0; c < plan.nchunk_a; ++c) {
      const float2 v = src[c];
      argmax_merge(m, choice, v.x, __float_as_int(v.y));
    }
    if (choice == kNoIndex) choice = 0;  // a row of NaNs only
  }
  const unsigned rej = __ballot_sync(0xffffffffu, lane < gr && x != choice);
  const int a = rej ? (__ffs(rej) - 1) : gr;
  const int choice_a = __shfl_sync(0xffffffffu, choice, a < gr ? a : 0);
  if (lane < B) {
    int tok = -1, pos = -1;
    if (lane < a) {
      pos = s_order[w][lane];
      tok = tokens[(size_t)r * B + pos];
    } else if (lane == a && a < gr) {
      pos = s_order[w][a];
      tok = choice_a;
    }
    out_tokens[(size_t)r * B + lane] = tok;
    out_pos[(size_t)r * B + lane] = pos;
  }
  if (lane == 0) {
    accepted_len[r] = a;
    n_commit[r] = a + (a < gr ? 1 : 0);
  }
}


// The work split (and so the workspace size) does not depend on the logit type: both
// instantiations of a kernel are counted and the smaller residency is taken.
int resident_stat_warps() {
  static int cache_f[64], cache_h[64];
  return std::min(resident_blocks(accept_stats_kernel<float>, kStatThreads, cache_f),
                  resident_blocks(accept_stats_kernel<__nv_bfloat16>, kStatThreads, cache_h)) *
         (kStatThreads / 32);
}

int resident_argmax_ctas() {
  static int cache_f[64], cache_h[64];
  return std::min(resident_blocks(accept_argmax_kernel<float>, kArgmaxThreads, cache_f),
                  resident_blocks(accept_argmax_kernel<__nv_bfloat16>, kArgmaxThreads, cache_h));
}

int resident_finish_ctas() {
  static int cache_f[64], cache_h[64];
  return std::min(resident_blocks(accept_finish_kernel<float>, kFinishThreads, cache_f),
                  resident_blocks(accept_finish_kernel<__nv_bfloat16>, kFinishThreads, cache_h));
}

// Argmax pass (greedy keys, or coupled-noise keys with nk.on) over the verified target
// rows, then the one-warp-per-request finish kernel as its programmatic dependent.
template <typename LT>
simsd_status launch_argmax_verify(const LT* target_logits, const int32_t* draft_tokens,
                                  const uint8_t* labels, const int32_t* pos_ids, int batch, int B,
                                  int gamma, int V, const AcceptPlan& plan, const AcceptWs& ws,
                                  const NoiseKey& nk, int32_t* accepted_len, int32_t* out_tokens,
                                  int32_t* out_pos, int32_t* n_commit, uint32_t* dev_err,
                                  cudaStream_t s) {
  const long warps_g = (long)batch * gamma * plan.nchunk_a;
  const long max_g = std::max(1, resident_argmax_ctas());
  const long grid_g = std::max<long>(1, std::min<long>((warps_g + kArgmaxThreads / 32 - 1) / (kArgmaxThreads / 32), max_g));
  accept_argmax_kernel<LT><<<(unsigned)grid_g, kArgmaxThreads, 0, s>>>(target_logits, labels, pos_ids, batch, B,
                                                                   gamma, V, plan, ws, nk);
  simsd_status st = last_launch_status();
  if (st != SIMSD_OK) return st;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3((unsigned)((batch + 7) / 8));
  cfg.blockDim = dim3(256);
  cfg.stream = s;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, accept_greedy_finish_kernel, draft_tokens, labels, batch, B,
                                           gamma, V, plan, ws, accepted_len, out_tokens, out_pos, n_commit,
                                           dev_err);
  if (e != cudaSuccess) {
    record_cuda_error("cudaLaunchKernelEx(accept_greedy_finish_kernel)", e);
    return SIMSD_ERR_CUDA;
  }
  return last_launch_status();
}

}  // namespace

}  // namespace simsd

SIMSD_API size_t simsd_accept_workspace(int batch, int B, int gamma, int V) {
  if (batch < 0 || B < 1 || gamma < 1 || gamma > B || V < 1) return 0;
  // enough for both the sampling path and the greedy one
  return std::max(simsd::make_plan(batch, gamma, V, 2).bytes, simsd::make_plan(batch, gamma, V, 1).bytes);
}

namespace simsd {
namespace {

template <typename LT>
simsd_status accept_impl(const LT* target_logits, const LT* draft_logits, const int32_t* draft_tokens,
                         const uint8_t* labels, int batch, int B, int gamma, int V, float temperature,
                         uint64_t seed, uint64_t offset, int32_t* accepted_len, int32_t* out_tokens,
                         int32_t* out_pos, int32_t* n_commit, void* workspace, size_t workspace_bytes,
                         uint32_t* dev_err, cudaStream_t s) {
  const bool greedy = temperature == 0.f;
  const AcceptPlan plan = make_plan(batch, gamma, V, greedy ? 1 : 2);
  if (!workspace || workspace_bytes < plan.bytes || (((uintptr_t)workspace) & 255))
    return SIMSD_ERR_WORKSPACE;
  char* base = (char*)workspace;
  AcceptWs ws;
  ws.stats = (float2*)(base + plan.off_stats);
  ws.winners = (unsigned long long*)(base + plan.off_winners);
  ws.ticket = (unsigned*)(base + plan.off_ticket);
  ws.n_stats = (long long)batch * gamma * (greedy ? 1 : 2) * plan.nchunk_a;
  ws.err = dev_err;
  const long grid_a = (long)batch * gamma * 2 * plan.nchunk_a;
  const long grid_b = plan.ctas_b;
  if (grid_a > 0x7fffffffL || grid_b > 0x7fffffffL) return SIMSD_ERR_UNSUPPORTED;
  if (greedy) {  // argmax pass over the verified target rows, then one warp per request
    const NoiseKey nk = {false, 0.f, 0u, 0u, 0u};
    return launch_argmax_verify<LT>(target_logits, draft_tokens, labels, nullptr, batch, B, gamma, V,
                                    plan, ws, nk, accepted_len, out_tokens, out_pos, n_commit, dev_err, s);
  }
  // persistent grid: as many stats CTAs as can be resident at once (fewer if the items are
  // fewer than the resident warps)
  const long max_ctas = std::max(1, resident_stat_warps() / (kStatThreads / 32));
  const long warps_needed = (long)batch * gamma * 2 * plan.nchunk_a;
  const long grid_stats = std::max<long>(1, std::min<long>((warps_needed + kStatThreads / 32 - 1) / (kStatThreads / 32),
                                                           max_ctas));
  accept_stats_kernel<LT><<<(unsigned)grid_stats, kStatThreads, 0, s>>>(
      target_logits, draft_logits, labels, batch, B, gamma, V, temperature, plan, ws);
  simsd_status st = last_launch_status();
  if (st != SIMSD_OK) return st;
  // K3b as a programmatic dependent of K3a: scheduled while K3a drains
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3((unsigned)grid_b);
  cfg.blockDim = dim3(kFinishThreads);
  cfg.stream = s;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(
      &cfg, accept_finish_kernel<LT>, target_logits, draft_logits, draft_tokens, labels, batch, B,
      gamma, V, temperature, (uint32_t)(seed & 0xffffffffu), (uint32_t)(seed >> 32),
      (uint32_t)(offset & 0xffffffffu), (uint32_t)(offset >> 32), plan, ws, accepted_len,
      out_tokens, out_pos, n_commit, dev_err);
  if (e != cudaSuccess) {
    record_cuda_error("cudaLaunchKernelEx(accept_finish_kernel)", e);
    return SIMSD_ERR_CUDA;
  }
  return last_launch_status();
}

template <typename LT>
simsd_status accept_coupled_impl(const LT* target_logits, const int32_t* draft_tokens, const uint8_t* labels,
                                 const int32_t* pos_ids, int batch, int B, int gamma, int V,
                                 float temperature, uint64_t seed, uint64_t offset, int32_t* accepted_len,
                                 int32_t* out_tokens, int32_t* out_pos, int32_t* n_commit, void* workspace,
                                 size_t workspace_bytes, uint32_t* dev_err, cudaStream_t s) {
  const AcceptPlan plan = make_plan(batch, gamma, V, 1);
  if (!workspace || workspace_bytes < plan.bytes || (((uintptr_t)workspace) & 255))
    return SIMSD_ERR_WORKSPACE;
  if ((long)batch * gamma * plan.nchunk_a > 0x7fffffffL) return SIMSD_ERR_UNSUPPORTED;
  char* base = (char*)workspace;
  AcceptWs ws;
  ws.stats = (float2*)(base + plan.off_stats);
  ws.winners = (unsigned long long*)(base + plan.off_winners);
  ws.ticket = (unsigned*)(base + plan.off_ticket);
  ws.n_stats = (long long)batch * gamma * plan.nchunk_a;
  ws.err = dev_err;
  const NoiseKey nk = {temperature > 0.f, temperature > 0.f ? 1.f / temperature : 0.f,
                       (uint32_t)(seed & 0xffffffffu), (uint32_t)(seed >> 32), (uint32_t)(offset & 0xffffffffu)};
  return launch_argmax_verify<LT>(target_logits, draft_tokens, labels, pos_ids, batch, B, gamma, V, plan, ws,
                                  nk, accepted_len, out_tokens, out_pos, n_commit, dev_err, s);
}

}  // namespace
}  // namespace simsd

SIMSD_API simsd_status simsd_accept_ex(const void* target_logits, const void* draft_logits,
                                       simsd_dtype logit_dtype, const int32_t* draft_tokens,
                                       const uint8_t* labels, int batch, int B, int gamma, int V,
                                       float temperature, uint64_t seed, uint64_t offset,
                                       int32_t* accepted_len, int32_t* out_tokens, int32_t* out_pos,
                                       int32_t* n_commit, void* workspace, size_t workspace_bytes,
                                       uint32_t* dev_err, simsd_stream_t stream) {
  SIMSD_NVTX_RANGE("simsd_accept_ex");
  using namespace simsd;
  if (batch < 0 || B < 1 || B > kMaxB || gamma < 1 || gamma > B || V < 1)
    return SIMSD_ERR_INVALID_ARG;
  if (!(temperature >= 0.f)) return SIMSD_ERR_INVALID_ARG;
  if (logit_dtype != SIMSD_DTYPE_FP32 && logit_dtype != SIMSD_DTYPE_BF16) return SIMSD_ERR_INVALID_ARG;
  if (batch == 0) return SIMSD_OK;
  if (!target_logits || !draft_logits || !draft_tokens || !labels || !accepted_len ||
      !out_tokens || !out_pos || !n_commit || !dev_err)
    return SIMSD_ERR_INVALID_ARG;
  if ((size_t)batch * B * (size_t)V >= ((size_t)1 << 40)) return SIMSD_ERR_UNSUPPORTED;
  cudaStream_t s = (cudaStream_t)stream;
  if (logit_dtype == SIMSD_DTYPE_BF16)
    return accept_impl<__nv_bfloat16>((const __nv_bfloat16*)target_logits, (const __nv_bfloat16*)draft_logits,
                                      draft_tokens, labels, batch, B, gamma, V, temperature, seed, offset,
                                      accepted_len, out_tokens, out_pos, n_commit, workspace,
                                      workspace_bytes, dev_err, s);
  return accept_impl<float>((const float*)target_logits, (const float*)draft_logits, draft_tokens, labels,
                            batch, B, gamma, V, temperature, seed, offset, accepted_len, out_tokens,
                            out_pos, n_commit, workspace, workspace_bytes, dev_err, s);
}

SIMSD_API simsd_status simsd_accept(const float* target_logits, const float* draft_logits,
                                    const int32_t* draft_tokens, const uint8_t* labels,
                                    int batch, int B, int gamma, int V, float temperature,
                                    uint64_t seed, uint64_t offset, int32_t* accepted_len,
                                    int32_t* out_tokens, int32_t* out_pos, int32_t* n_commit,
                                    void* workspace, size_t workspace_bytes, uint32_t* dev_err,
                                    simsd_stream_t stream) {
  return simsd_accept_ex(target_logits, draft_logits, SIMSD_DTYPE_FP32, draft_tokens, labels, batch, B,
                         gamma, V, temperature, seed, offset, accepted_len, out_tokens, out_pos,
                         n_commit, workspace, workspace_bytes, dev_err, stream);
}

SIMSD_API simsd_status simsd_accept_coupled_ex(const void* target_logits, simsd_dtype logit_dtype,
                                               const int32_t* draft_tokens, const uint8_t* labels,
                                               const int32_t* pos_ids, int batch, int B, int gamma, int V,
                                               float temperature, uint64_t seed, uint64_t offset,
                                               int32_t* accepted_len, int32_t* out_tokens,
                                               int32_t* out_pos, int32_t* n_commit, void* workspace,
                                               size_t workspace_bytes, uint32_t* dev_err,
                                               simsd_stream_t stream) {
  SIMSD_NVTX_RANGE("simsd_accept_coupled_ex");
  using namespace simsd;
  if (batch < 0 || B < 1 || B > kMaxB || gamma < 1 || gamma > B || V < 1)
    return SIMSD_ERR_INVALID_ARG;
  if (!(temperature >= 0.f)) return SIMSD_ERR_INVALID_ARG;
  if (logit_dtype != SIMSD_DTYPE_FP32 && logit_dtype != SIMSD_DTYPE_BF16) return SIMSD_ERR_INVALID_ARG;
  if (batch == 0) return SIMSD_OK;
  if (!target_logits || !draft_tokens || !labels || !pos_ids || !accepted_len || !out_tokens ||
      !out_pos || !n_commit || !dev_err)
    return SIMSD_ERR_INVALID_ARG;
  if ((size_t)batch * B * (size_t)V >= ((size_t)1 << 40)) return SIMSD_ERR_UNSUPPORTED;
  cudaStream_t s = (cudaStream_t)stream;
  if (logit_dtype == SIMSD_DTYPE_BF16)
    return accept_coupled_impl<__nv_bfloat16>((const __nv_bfloat16*)target_logits, draft_tokens, labels, pos_ids,
                                              batch, B, gamma, V, temperature, seed, offset, accepted_len,
                                              out_tokens, out_pos, n_commit, workspace, workspace_bytes,
                                              dev_err, s);
  return accept_coupled_impl<float>((const float*)target_logits, draft_tokens, labels, pos_ids, batch, B,
                                    gamma, V, temperature, seed, offset, accepted_len, out_tokens, out_pos,
                                    n_commit, workspace, workspace_bytes, dev_err, s);
}

SIMSD_API simsd_status simsd_accept_coupled(const float* target_logits, const int32_t* draft_tokens,
                                            const uint8_t* labels, const int32_t* pos_ids, int batch,
                                            int B, int gamma, int V, float temperature, uint64_t seed,
                                            uint64_t offset, int32_t* accepted_len, int32_t* out_tokens,
                                            int32_t* out_pos, int32_t* n_commit, void* workspace,
                                            size_t workspace_bytes, uint32_t* dev_err,
                                            simsd_stream_t stream) {
  return simsd_accept_coupled_ex(target_logits, SIMSD_DTYPE_FP32, draft_tokens, labels, pos_ids, batch, B,
                                 gamma, V, temperature, seed, offset, accepted_len, out_tokens, out_pos,
                                 n_commit, workspace, workspace_bytes, dev_err, stream);
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

// Identity of the calling thread's current CUDA context (driver entry points resolved once
// through the runtime). A device reset destroys the context and the next one loads the
// library's device code again, possibly at another address; the identity tells the two apart.
bool current_context_id(unsigned long long* id) {
  static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
  static PFN_cuCtxGetId_v12000 get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_current = (PFN_cuCtxGetCurrent_v4000)p;
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_id = (PFN_cuCtxGetId_v12000)p;
  });
  CUcontext ctx = nullptr;
  if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx) return false;
  return get_id(ctx, id) == CUDA_SUCCESS;
}

struct ScratchAddr {
  unsigned long long ctx;  // context the address belongs to
  void* ptr;
  bool valid;
};
std::mutex g_scratch_mutex;
ScratchAddr g_scratch_addr[kMaxDevices];

// Device address of g_accept_scratch on the current device. Resolved (with that device
// current) on the first call per device and again whenever the device's context has been
// replaced (after a device reset); the host-side symbol itself is not a device address and
// is never passed to a kernel. Where the context identity cannot be read, the address is
// looked up on every call (a runtime query; it allocates nothing).
simsd_status noalloc_scratch(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    record_cuda_error("cudaGetDevice", e);
    return SIMSD_ERR_CUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) return SIMSD_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  ScratchAddr& c = g_scratch_addr[dev];
  unsigned long long ctx = 0;
  bool have_ctx = current_context_id(&ctx);
  if (have_ctx && c.valid && c.ctx == ctx) {
    *out = c.ptr;
    return SIMSD_OK;
  }
  void* ptr = nullptr;
  e = cudaGetSymbolAddress(&ptr, g_accept_scratch);
  if (e != cudaSuccess || !ptr) {
    record_cuda_error("cudaGetSymbolAddress", e != cudaSuccess ? e : cudaErrorInvalidSymbol);
    return SIMSD_ERR_CUDA;
  }
  if (!have_ctx) have_ctx = current_context_id(&ctx);  // the lookup made the context current
  c.ctx = ctx;
  c.ptr = ptr;
  c.valid = have_ctx;
  *out = ptr;
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
  SIMSD_NVTX_RANGE("simsd_accept_noalloc");
  using namespace simsd;
  // the argument checks of simsd_accept come first, so both return the same status
  if (batch < 0 || B < 1 || B > kMaxB || gamma < 1 || gamma > B || V < 1)
    return SIMSD_ERR_INVALID_ARG;
  if (!(temperature >= 0.f)) return SIMSD_ERR_INVALID_ARG;
  if (batch == 0) return SIMSD_OK;
  if (!target_logits || !draft_logits || !draft_tokens || !labels || !accepted_len ||
      !out_tokens || !out_pos || !n_commit || !dev_err)
    return SIMSD_ERR_INVALID_ARG;
  if ((size_t)batch * B * (size_t)V >= ((size_t)1 << 40)) return SIMSD_ERR_UNSUPPORTED;
  if (make_plan(batch, gamma, V, temperature == 0.f ? 1 : 2).bytes > kNoAllocScratchBytes)
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
