// Tensor-core (tcgen05 / TMEM) verify attention for bf16, head dim 128.
//
// What it computes (SimSD notes, "关键设计" items 2-3): for every response row of a request
// and query head, softmax attention over the request's cached prompt keys plus the
// response keys that the temporal-causal mask A_ij leaves visible, with RoPE applied to
// the response queries/keys at the copied position ids.
//
// Work decomposition. For each (request b, kv head h) the 2B*G query rows (response slot
// s, head g of the group; row = s*G + g) form one or two 128-row blocks; a "pair" is
// (b, h, all row blocks). Each pair is a sequence of 64-key tiles: tile 0 is the response
// tail (the 2B response keys, rotated and masked here), tiles 1.. stream the prompt keys.
// All pairs' tiles are concatenated and cut into equal contiguous ranges, one per
// persistent CTA (stream-K); a CTA therefore sees at most two partial pairs (its first
// and last), whose (O, max, sum) partials are merged by attn_tc_merge_kernel.
//
// Per CTA, warp roles:
//   producer warp  : TMA loads of prompt K and V tiles (128-byte swizzle) into a ring of
//                    shared-memory stages.
//   MMA warp       : one thread issues S = Q K^T (M = 128 rows, N = 64 keys, K = 128) into
//                    one of two TMEM S buffers, then O += P V (M = 128, N = 128, K = 64)
//                    into the TMEM O accumulator; completion is signalled with
//                    tcgen05.commit to mbarriers.
//   softmax warps  : one thread per query row (TMEM lane). Per segment: load + rotate Q
//                    into shared memory (and the response K/V tail tile); per tile: read
//                    S from TMEM, apply the mask, online softmax in the log2 domain with
//                    lazy rescaling of O (only when the running max grows by > 8), write P
//                    (bf16) to shared memory; epilogue: O / l to global memory (or the
//                    partial to the workspace).
// Every wait is bounded in time; on expiry the kernel raises SIMSD_DEVERR_TIMEOUT in the
// error word and unwinds (no trap).
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "attn_common.cuh"
#include "tc_ptx.cuh"

namespace simsd {
namespace tc {

constexpr int kTileKeys = 64;
constexpr int kD = 128;
constexpr int kBlockRows = 128;
constexpr uint32_t kHalfTile = kTileKeys * 128;       // 64 rows x 128 B (one 64-element half)
constexpr uint32_t kKVTile = 2 * kHalfTile;           // 16 KB: one K (or V) tile
constexpr uint32_t kStageBytes = 2 * kKVTile;         // K + V
constexpr uint32_t kQBlock = 2 * kBlockRows * 128;    // 32 KB: 128 rows x 128 dims
constexpr uint32_t kPBlock = kBlockRows * 128;        // 16 KB: 128 rows x 64 keys
constexpr uint64_t kWaitLimitNs = 2000000000ull;      // 2 s: far beyond any legitimate wait

template <int NRB>
struct Cfg {
  static constexpr int kStages = NRB == 1 ? 4 : 2;
  static constexpr int kSoftmaxThreads = 128 * NRB;
  static constexpr int kProducerWarp = 4 * NRB;
  static constexpr int kMmaWarp = 4 * NRB + 1;
  static constexpr int kThreads = kSoftmaxThreads + 64;
  static constexpr uint32_t kTmemCols = 256 * NRB;
  static constexpr uint32_t kOffQ = 0;
  static constexpr uint32_t kOffP = kOffQ + NRB * kQBlock;            // [rb][buf]
  static constexpr uint32_t kOffStages = kOffP + NRB * 2 * kPBlock;
  static constexpr uint32_t kOffTail = kOffStages + kStages * kStageBytes;
  static constexpr uint32_t kOffBar = kOffTail + kStageBytes;
  static constexpr uint32_t kBarBytes = 256;
  static constexpr uint32_t kSmemBytes = kOffBar + kBarBytes + 1024;  // + base alignment
  static constexpr uint32_t tmem_s(int rb, int buf) { return (uint32_t)(rb * 2 + buf) * 64u; }
  static constexpr uint32_t tmem_o(int rb) { return (uint32_t)NRB * 128u + (uint32_t)rb * 128u; }
};

struct TcArgs {
  int batch, B, Hq, Hkv, G, R, nrb, ctas;  // R = 2B*G real rows per pair
  int layout;
  const __nv_bfloat16* q;
  const __nv_bfloat16* k_resp;
  const __nv_bfloat16* v_resp;
  const int64_t* cache_start;
  const int32_t* prompt_len;
  const int32_t* pos_ids;
  const uint8_t* labels;
  float scale_log2;
  __nv_bfloat16* out;
  float* lse;
  uint32_t* dev_err;
  float* ws_o;     // [2 * ctas][nrb * 128][128] partial numerators
  float2* ws_ml;   // [2 * ctas][nrb * 128] partial (max, sum), log2 domain
  RopeTable rope;
};

// ----------------------------------------------------------------------- scheduling
__device__ __forceinline__ bool request_invalid(const TcArgs& a, int b) {
  return a.prompt_len[b] < 0 || a.labels[(size_t)b * 2 * a.B] == kLabelInvalid;
}
__device__ __forceinline__ int tiles_per_pair(const TcArgs& a, int b) {
  if (request_invalid(a, b)) return 1;
  return 1 + (a.prompt_len[b] + kTileKeys - 1) / kTileKeys;
}

// CTA c covers global tiles [c*T/C, (c+1)*T/C).
__device__ __forceinline__ int64_t cta_begin(int64_t T, int C, int c) {
  return (T * (int64_t)c) / C;
}

struct SchedStart {
  int64_t T, t0, t1, Tb;  // total tiles, this CTA's range, first tile of request b
  int b;
};

// One warp: total tile count and the request containing tile `t0` of CTA `c`.
__device__ SchedStart warp_schedule(const TcArgs& a, int c, int C, int lane) {
  const int ppr = a.Hkv;  // pairs per request
  int64_t tot = 0;
  for (int base = 0; base < a.batch; base += 32) {
    const int b = base + lane;
    int64_t v = b < a.batch ? (int64_t)ppr * tiles_per_pair(a, b) : 0;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    tot += v;
  }
  SchedStart s;
  s.T = tot;
  s.t0 = cta_begin(tot, C, c);
  s.t1 = cta_begin(tot, C, c + 1);
  s.b = a.batch;
  s.Tb = tot;
  int64_t cum = 0;
  for (int base = 0; base < a.batch; base += 32) {
    const int b = base + lane;
    const int64_t v = b < a.batch ? (int64_t)ppr * tiles_per_pair(a, b) : 0;
    int64_t incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int64_t n = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += n;
    }
    const unsigned hit = __ballot_sync(0xffffffffu, b < a.batch && cum + incl > s.t0);
    if (hit) {
      const int L = __ffs(hit) - 1;
      const int64_t excl = __shfl_sync(0xffffffffu, incl - v, L);
      s.b = base + L;
      s.Tb = cum + excl;
      break;
    }
    cum += __shfl_sync(0xffffffffu, incl, 31);
  }
  return s;
}

// Walks the segments (pair pieces) of one CTA's tile range.
struct SegIter {
  int64_t t, t1, Tb, t0;
  int b, nt, ppr, batch;
  // current segment
  int h, i0, n;
  bool first, full, has_tail, invalid;

  __device__ void init(const TcArgs& a, const SchedStart& s) {
    t = s.t0;
    t0 = s.t0;
    t1 = s.t1;
    Tb = s.Tb;
    b = s.b;
    ppr = a.Hkv;
    batch = a.batch;
    nt = (b < batch) ? tiles_per_pair(a, b) : 1;
  }
  // Prepares the segment starting at t; false when the range is exhausted.
  __device__ bool next(const TcArgs& a) {
    if (t >= t1 || b >= batch) return false;
    const int64_t rel = t - Tb;
    const int q = (int)(rel / nt);
    i0 = (int)(rel % nt);
    const int64_t pair_start = Tb + (int64_t)q * nt;
    const int64_t pair_end = pair_start + nt;
    const int64_t seg_end = pair_end < t1 ? pair_end : t1;
    n = (int)(seg_end - t);
    h = q;
    first = (t == t0);
    full = (i0 == 0) && (seg_end == pair_end);
    has_tail = (i0 == 0);
    invalid = request_invalid(a, b);
    return true;
  }
  __device__ void advance(const TcArgs& a) {
    t += n;
    if (t >= Tb + (int64_t)ppr * nt) {
      Tb += (int64_t)ppr * nt;
      ++b;
      nt = (b < batch) ? tiles_per_pair(a, b) : 1;
    }
  }
};

// --------------------------------------------------------------------- small helpers
struct Shared {
  uint64_t bars[20];
  uint32_t tmem_base;
  int abort;
  int64_t T, t0, t1, Tb;
  int b;
};

enum BarIdx { kFull0 = 0, kEmpty0 = 4, kSFull0 = 8, kSFree0 = 10, kPFull0 = 12, kPFree0 = 14,
              kQFull = 16, kDrain = 17 };

__device__ __forceinline__ bool wait_bar(Shared* sh, uint32_t bar, uint32_t parity,
                                         uint32_t* dev_err) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t t_start = ptx::globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    if ((it & 63) == 0) {
      if (*(volatile int*)&sh->abort) return false;
      if (ptx::globaltimer_ns() - t_start > kWaitLimitNs) {
        *(volatile int*)&sh->abort = 1;
        atomicOr(dev_err, SIMSD_DEVERR_TIMEOUT);
        return false;
      }
    }
  }
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}
__device__ __forceinline__ float bf16_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }

// Byte offset of 16-byte chunk `c` (0..7) of row `r` in a 128-byte-swizzled tile whose rows
// are 128 bytes apart (rows grouped by 8 into 1024-byte atoms).
__device__ __forceinline__ uint32_t sw128(int r, int c) {
  return (uint32_t)r * 128u + ((uint32_t)(c ^ (r & 7)) << 4);
}

// Rotates the 16 chunks (8 bf16 each) of one 128-element row held in `v` (chunk c pairs
// with chunk c + 8: elements d and d + 64) at position `pos`.
__device__ __forceinline__ void rope_row(uint4 (&v)[16], int pos, const RopeTable& rt) {
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    uint32_t* lo = reinterpret_cast<uint32_t*>(&v[c]);
    uint32_t* hi = reinterpret_cast<uint32_t*>(&v[c + 8]);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int d0 = 8 * c + 2 * e;
      float s0, c0, s1, c1;
      rope_sincos(pos, rt.c_hi[d0], rt.c_lo[d0], &s0, &c0);
      rope_sincos(pos, rt.c_hi[d0 + 1], rt.c_lo[d0 + 1], &s1, &c1);
      const float x0 = bf16_lo(lo[e]), x1 = bf16_hi(lo[e]);
      const float y0 = bf16_lo(hi[e]), y1 = bf16_hi(hi[e]);
      lo[e] = pack_bf16(x0 * c0 - y0 * s0, x1 * c1 - y1 * s1);
      hi[e] = pack_bf16(x0 * s0 + y0 * c0, x1 * s1 + y1 * c1);
    }
  }
}

__device__ __forceinline__ void load_row(uint4 (&v)[16], const __nv_bfloat16* src) {
  const uint4* p = reinterpret_cast<const uint4*>(src);
#pragma unroll
  for (int c = 0; c < 16; ++c) v[c] = __ldg(p + c);
}

// Stores a 128-element row (16 chunks) into a two-half 128B-swizzled tile at row r.
__device__ __forceinline__ void store_row_sw(uint8_t* tile, uint32_t half_bytes, int r,
                                             const uint4 (&v)[16]) {
#pragma unroll
  for (int c = 0; c < 16; ++c)
    *reinterpret_cast<uint4*>(tile + (c >> 3) * half_bytes + sw128(r, c & 7)) = v[c];
}

// ------------------------------------------------------------------------- the kernel
template <int NRB>
__global__ void __launch_bounds__(Cfg<NRB>::kThreads, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                   const __grid_constant__ TcArgs a) {
  using C = Cfg<NRB>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  Shared* sh = reinterpret_cast<Shared*>(smem + C::kOffBar);
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const uint32_t sbase = ptx::smem_u32(smem);
  auto bar = [&](int i) { return ptx::smem_u32(&sh->bars[i]); };

  if (warp == C::kProducerWarp) {
    const SchedStart s = warp_schedule(a, blockIdx.x, a.ctas, lane);
    if (lane == 0) {
      sh->T = s.T;
      sh->t0 = s.t0;
      sh->t1 = s.t1;
      sh->Tb = s.Tb;
      sh->b = s.b;
      sh->abort = 0;
      for (int i = 0; i < C::kStages; ++i) {
        ptx::mbar_init(bar(kFull0 + i), 1);
        ptx::mbar_init(bar(kEmpty0 + i), 1);
      }
      for (int i = 0; i < 2; ++i) {
        ptx::mbar_init(bar(kSFull0 + i), 1);
        ptx::mbar_init(bar(kSFree0 + i), C::kSoftmaxThreads);
        ptx::mbar_init(bar(kPFull0 + i), C::kSoftmaxThreads);
        ptx::mbar_init(bar(kPFree0 + i), 1);
      }
      ptx::mbar_init(bar(kQFull), C::kSoftmaxThreads);
      ptx::mbar_init(bar(kDrain), 1);
      ptx::fence_mbar_init();
      ptx::prefetch_tensormap(&tmk);
      ptx::prefetch_tensormap(&tmv);
    }
  } else if (warp == C::kMmaWarp) {
    ptx::tmem_alloc(ptx::smem_u32(&sh->tmem_base), C::kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();

  SchedStart st;
  st.T = sh->T;
  st.t0 = sh->t0;
  st.t1 = sh->t1;
  st.Tb = sh->Tb;
  st.b = sh->b;
  const uint32_t tmem = sh->tmem_base;
  const int twoB = 2 * a.B;

  if (warp == C::kProducerWarp) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      SegIter it;
      it.init(a, st);
      uint32_t m = 0;
      bool ok = true;
      while (ok && it.next(a)) {
        if (!it.invalid) {
          const int64_t start = a.cache_start[it.b];
          for (int i = it.i0; i < it.i0 + it.n && ok; ++i) {
            if (i == 0) continue;  // response tail: staged by the softmax warps
            const int s = m % C::kStages;
            ok = wait_bar(sh, bar(kEmpty0 + s), ((m / C::kStages) & 1) ^ 1, a.dev_err);
            if (!ok) break;
            ptx::mbar_arrive_expect_tx(bar(kFull0 + s), kStageBytes);
            const int tok = (int)(start + (int64_t)(i - 1) * kTileKeys);
            const uint32_t kdst = sbase + C::kOffStages + s * kStageBytes;
            const uint32_t vdst = kdst + kKVTile;
#pragma unroll
            for (int half = 0; half < 2; ++half) {
              if (a.layout == SIMSD_CACHE_NHD) {
                ptx::tma_load_3d(kdst + half * kHalfTile, &tmk, half * 64, it.h, tok, bar(kFull0 + s));
                ptx::tma_load_3d(vdst + half * kHalfTile, &tmv, half * 64, it.h, tok, bar(kFull0 + s));
              } else {
                ptx::tma_load_3d(kdst + half * kHalfTile, &tmk, half * 64, tok, it.h, bar(kFull0 + s));
                ptx::tma_load_3d(vdst + half * kHalfTile, &tmv, half * 64, tok, it.h, bar(kFull0 + s));
              }
            }
            ++m;
          }
        }
        it.advance(a);
      }
      if (!ok) {  // let the loads already issued land before shared memory goes away
        const uint32_t issued = m;
        for (uint32_t k = issued > (uint32_t)C::kStages ? issued - C::kStages : 0; k < issued; ++k) {
          const uint64_t t_start = ptx::globaltimer_ns();
          while (!ptx::mbar_try_wait(bar(kFull0 + k % C::kStages), (k / C::kStages) & 1) &&
                 ptx::globaltimer_ns() - t_start < 100000000ull) {
          }
        }
      }
    }
  } else if (warp == C::kMmaWarp) {
    // ------------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idS = ptx::idesc_bf16(128, kTileKeys, 0, 0);
      constexpr uint32_t idPV = ptx::idesc_bf16(128, kD, 0, 1);
      SegIter it;
      it.init(a, st);
      uint32_t j = 0, m = 0, nseg = 0;
      bool ok = true;
      // per S/P buffer: where the tile's V lives and which stage to release
      uint32_t vaddr_of[2] = {0, 0};
      int stage_of[2] = {-1, -1};
      auto issue_pv = [&](uint32_t jj, bool first_in_seg) -> bool {
        const int buf = jj & 1;
        if (!wait_bar(sh, bar(kPFull0 + buf), (jj >> 1) & 1, a.dev_err)) return false;
        ptx::tc_fence_after();
#pragma unroll
        for (int rb = 0; rb < NRB; ++rb) {
          const uint32_t pbase = sbase + C::kOffP + (rb * 2 + buf) * kPBlock;
#pragma unroll
          for (int kk = 0; kk < kTileKeys / 16; ++kk) {
            const uint64_t ad = ptx::sdesc_sw128(pbase + kk * 32, 16, 1024);
            const uint64_t bd = ptx::sdesc_sw128(vaddr_of[buf] + kk * 16 * 128, kHalfTile, 1024);
            ptx::mma_f16_ss(tmem + C::tmem_o(rb), ad, bd, idPV, (first_in_seg && kk == 0) ? 0u : 1u);
          }
        }
        ptx::mma_commit(bar(kPFree0 + buf));
        if (stage_of[buf] >= 0) ptx::mma_commit(bar(kEmpty0 + stage_of[buf]));
        return true;
      };
      while (ok && it.next(a)) {
        if (it.invalid) {
          it.advance(a);
          continue;
        }
        ok = wait_bar(sh, bar(kQFull), nseg & 1, a.dev_err);
        if (!ok) break;
        ptx::tc_fence_after();
        const uint32_t jfirst = j;
        for (int i = it.i0; i < it.i0 + it.n; ++i, ++j) {
          const int buf = j & 1;
          uint32_t kaddr;
          if (i == 0) {
            kaddr = sbase + C::kOffTail;
            vaddr_of[buf] = kaddr + kKVTile;
            stage_of[buf] = -1;
          } else {
            const int s = m % C::kStages;
            ok = wait_bar(sh, bar(kFull0 + s), (m / C::kStages) & 1, a.dev_err);
            if (!ok) break;
            kaddr = sbase + C::kOffStages + s * kStageBytes;
            vaddr_of[buf] = kaddr + kKVTile;
            stage_of[buf] = s;
            ++m;
          }
          ok = wait_bar(sh, bar(kSFree0 + buf), ((j >> 1) & 1) ^ 1, a.dev_err);
          if (!ok) break;
          ptx::tc_fence_after();
#pragma unroll
          for (int rb = 0; rb < NRB; ++rb) {
            const uint32_t qbase = sbase + C::kOffQ + rb * kQBlock;
#pragma unroll
            for (int kk = 0; kk < kD / 16; ++kk) {
              const uint32_t koff = (kk >> 2) * (kBlockRows * 128) + (kk & 3) * 32;
              const uint64_t ad = ptx::sdesc_sw128(qbase + koff, 16, 1024);
              const uint64_t bd = ptx::sdesc_sw128(kaddr + (kk >> 2) * kHalfTile + (kk & 3) * 32, 16, 1024);
              ptx::mma_f16_ss(tmem + C::tmem_s(rb, buf), ad, bd, idS, kk > 0 ? 1u : 0u);
            }
          }
          ptx::mma_commit(bar(kSFull0 + buf));
          if (j > jfirst) {
            ok = issue_pv(j - 1, j - 1 == jfirst);
            if (!ok) break;
          }
        }
        if (!ok) break;
        ok = issue_pv(j - 1, j - 1 == jfirst);
        ++nseg;
        it.advance(a);
      }
      // drain: every MMA issued so far has completed before TMEM is released
      ptx::mma_commit(bar(kDrain));
      const uint64_t t_start = ptx::globaltimer_ns();
      while (!ptx::mbar_try_wait(bar(kDrain), 0) &&
             ptx::globaltimer_ns() - t_start < 100000000ull) {
      }
    }
  } else {
    // -------------------------------------------------------------- softmax warps
    const int rb = warp >> 2;                // row block of this warpgroup
    const int lrow = (warp & 3) * 32 + lane;  // TMEM lane = row within the block
    const int row = rb * kBlockRows + lrow;   // row within the pair
    const bool real = row < a.R;
    const int s_slot = real ? row / a.G : 0;
    const int g = real ? row % a.G : 0;
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    uint8_t* qtile = smem + C::kOffQ + rb * kQBlock;
    uint8_t* tailk = smem + C::kOffTail;
    uint8_t* tailv = tailk + kKVTile;
    SegIter it;
    it.init(a, st);
    uint32_t j = 0;
    bool ok = true;
    while (ok && it.next(a)) {
      const int b = it.b, h = it.h;
      const size_t orow = ((size_t)b * twoB + s_slot) * a.Hq + (size_t)h * a.G + g;
      if (it.invalid) {
        if (real) {
          uint4* o = reinterpret_cast<uint4*>(a.out + orow * kD);
#pragma unroll
          for (int c = 0; c < 16; ++c) o[c] = make_uint4(0, 0, 0, 0);
          if (a.lse) a.lse[orow] = -INFINITY;
        }
        if (tid == 0 && h == 0 && a.prompt_len[b] < 0) atomicOr(a.dev_err, SIMSD_DEVERR_PROMPT_LEN);
        it.advance(a);
        continue;
      }
      const int P = a.prompt_len[b];
      // ---- segment prologue: rotated Q rows (and the response tail tile)
      {
        uint4 v[16];
        if (real) {
          load_row(v, a.q + orow * kD);
          rope_row(v, a.pos_ids[(size_t)b * twoB + s_slot], a.rope);
        } else {
#pragma unroll
          for (int c = 0; c < 16; ++c) v[c] = make_uint4(0, 0, 0, 0);
        }
        store_row_sw(qtile, kBlockRows * 128, lrow, v);
        if (it.has_tail && rb == 0) {
          const int key = lrow & 63;
          const bool is_v = lrow >= 64;
          if (key < twoB) {
            const size_t krow = (((size_t)b * twoB + key) * a.Hkv + h) * kD;
            load_row(v, (is_v ? a.v_resp : a.k_resp) + krow);
            if (!is_v) rope_row(v, a.pos_ids[(size_t)b * twoB + key], a.rope);
          } else {
#pragma unroll
            for (int c = 0; c < 16; ++c) v[c] = make_uint4(0, 0, 0, 0);
          }
          store_row_sw(is_v ? tailv : tailk, kHalfTile, key, v);
        }
      }
      ptx::fence_proxy_async_smem();
      ptx::mbar_arrive(bar(kQFull));
      // visibility of the 2B response keys for this row (bit j = key j visible)
      uint64_t vis = 0;
      if (it.has_tail) {
        const uint8_t* lab = a.labels + (size_t)b * twoB;
        if (real) {
          const int t = row_threshold(lab[s_slot]);
          for (int k = 0; k < twoB; ++k)
            if (response_key_visible(lab[k], t)) vis |= 1ull << k;
        } else {
          vis = twoB == 64 ? ~0ull : ((1ull << twoB) - 1);
        }
      }
      float m_used = -INFINITY, l = 0.f;
      const uint32_t jfirst = j;
      for (int i = it.i0; i < it.i0 + it.n; ++i, ++j) {
        const int buf = j & 1;
        ok = __all_sync(0xffffffffu, wait_bar(sh, bar(kSFull0 + buf), (j >> 1) & 1, a.dev_err));
        if (!ok) break;
        ptx::tc_fence_after();
        uint32_t sa[32], sb[32];
        const uint32_t ts = tmem + lane_off + C::tmem_s(rb, buf);
        ptx::tmem_ld32(ts, sa);
        ptx::tmem_ld32(ts + 32, sb);
        ptx::tmem_ld_wait(sa);
        ptx::tmem_ld_wait(sb);
        ptx::tc_fence_before();
        ptx::mbar_arrive(bar(kSFree0 + buf));
        float x[64];
        if (i == 0) {
#pragma unroll
          for (int c = 0; c < 64; ++c) {
            const float sv = __uint_as_float(c < 32 ? sa[c] : sb[c - 32]) * a.scale_log2;
            x[c] = ((vis >> c) & 1ull) ? sv : -INFINITY;
          }
        } else {
          const int nvalid = P - (i - 1) * kTileKeys;
#pragma unroll
          for (int c = 0; c < 64; ++c) {
            const float sv = __uint_as_float(c < 32 ? sa[c] : sb[c - 32]) * a.scale_log2;
            x[c] = c < nvalid ? sv : -INFINITY;
          }
        }
        float mt = x[0];
#pragma unroll
        for (int c = 1; c < 64; ++c) mt = fmaxf(mt, x[c]);
        // lazy rescale: only when some row's max grew by more than 2^8; warp-uniform because
        // TMEM loads/stores are warp-collective
        if (__any_sync(0xffffffffu, mt > m_used + 8.f)) {
          const float m_new = fmaxf(m_used, mt);
          if (j != jfirst) {  // rescale O: the previous P V must have landed
            const uint32_t jp = j - 1;
            ok = __all_sync(0xffffffffu,
                            wait_bar(sh, bar(kPFree0 + (jp & 1)), (jp >> 1) & 1, a.dev_err));
            if (!ok) break;
            ptx::tc_fence_after();
            const float alpha = ptx::ex2(m_used - m_new);
            l *= alpha;
            const uint32_t to = tmem + lane_off + C::tmem_o(rb);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              uint32_t o[32];
              ptx::tmem_ld32(to + 32 * k, o);
              ptx::tmem_ld_wait(o);
#pragma unroll
              for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
              ptx::tmem_st32(to + 32 * k, o);
            }
            ptx::tmem_st_wait();
          }
          m_used = m_new;
        }
        uint32_t pk[32];
        float lsum = 0.f;
#pragma unroll
        for (int c = 0; c < 64; c += 2) {
          const float p0 = ptx::ex2(x[c] - m_used);
          const float p1 = ptx::ex2(x[c + 1] - m_used);
          lsum += p0 + p1;
          pk[c >> 1] = pack_bf16(p0, p1);
        }
        l += lsum;
        // P buffer `buf` is free once the P V that last read it (tile j - 2) completed
        ok = __all_sync(0xffffffffu,
                        wait_bar(sh, bar(kPFree0 + buf), ((j >> 1) & 1) ^ 1, a.dev_err));
        if (!ok) break;
        uint8_t* pt = smem + C::kOffP + (rb * 2 + buf) * kPBlock;
#pragma unroll
        for (int c = 0; c < 8; ++c)
          *reinterpret_cast<uint4*>(pt + sw128(lrow, c)) =
              make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
        ptx::fence_proxy_async_smem();
        ptx::tc_fence_before();
        ptx::mbar_arrive(bar(kPFull0 + buf));
      }
      if (!ok) break;
      // ---- epilogue: wait for the last P V, then O / l (or the partial)
      const uint32_t jl = j - 1;
      ok = __all_sync(0xffffffffu, wait_bar(sh, bar(kPFree0 + (jl & 1)), (jl >> 1) & 1, a.dev_err));
      if (!ok) break;
      ptx::tc_fence_after();
      const uint32_t to = tmem + lane_off + C::tmem_o(rb);
      if (it.full) {
        const float inv = 1.f / l;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          uint32_t o[32];
          ptx::tmem_ld32(to + 32 * k, o);
          ptx::tmem_ld_wait(o);
          if (real) {
            uint4* dst = reinterpret_cast<uint4*>(a.out + orow * kD + 32 * k);
#pragma unroll
            for (int c = 0; c < 4; ++c)
              dst[c] = make_uint4(pack_bf16(__uint_as_float(o[8 * c]) * inv, __uint_as_float(o[8 * c + 1]) * inv),
                                  pack_bf16(__uint_as_float(o[8 * c + 2]) * inv, __uint_as_float(o[8 * c + 3]) * inv),
                                  pack_bf16(__uint_as_float(o[8 * c + 4]) * inv, __uint_as_float(o[8 * c + 5]) * inv),
                                  pack_bf16(__uint_as_float(o[8 * c + 6]) * inv, __uint_as_float(o[8 * c + 7]) * inv));
          }
        }
        if (real && a.lse) a.lse[orow] = (m_used + __log2f(l)) * 0.69314718055994530942f;
      } else {
        const int slot = 2 * blockIdx.x + (it.first ? 0 : 1);
        float* wo = a.ws_o + ((size_t)slot * (NRB * kBlockRows) + row) * kD;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          uint32_t o[32];
          ptx::tmem_ld32(to + 32 * k, o);
          ptx::tmem_ld_wait(o);
          if (real) {
            float4* dst = reinterpret_cast<float4*>(wo + 32 * k);
#pragma unroll
            for (int c = 0; c < 8; ++c)
              dst[c] = make_float4(__uint_as_float(o[4 * c]), __uint_as_float(o[4 * c + 1]),
                                   __uint_as_float(o[4 * c + 2]), __uint_as_float(o[4 * c + 3]));
          }
        }
        if (real) a.ws_ml[(size_t)slot * (NRB * kBlockRows) + row] = make_float2(m_used, l);
      }
      ptx::tc_fence_before();
      it.advance(a);
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (warp == C::kMmaWarp) ptx::tmem_dealloc(tmem, C::kTmemCols);
}

// Merges the partial segments of every pair that was split between CTAs. Block c handles
// the pair containing the last tile of CTA c's range when that pair started inside CTA c's
// range and continues past it (so every split pair is merged exactly once).
template <int NRB>
__global__ void __launch_bounds__(128) attn_tc_merge_kernel(const __grid_constant__ TcArgs a) {
  __shared__ SchedStart s_end;
  __shared__ int64_t s_pair_start, s_pair_end;
  __shared__ int s_b, s_h, s_go;
  const int c = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp == 0) {
    // locate the tile t1(c) - 1 with the same scan the attention kernel uses
    SchedStart s = warp_schedule(a, c + 1, a.ctas, lane);  // s.t0 = t1(c)
    const int64_t T = s.T;
    const int64_t t0c = cta_begin(T, a.ctas, c);
    const int64_t t1c = s.t0;
    int go = 0;
    if (lane == 0 && t1c > t0c && t1c < T) {
      // request containing tile t1c - 1: rescan from s (which contains tile t1c)
      int b = s.b;
      int64_t Tb = s.Tb;
      const int64_t last = t1c - 1;
      while (last < Tb) {  // step back one request at a time (rarely more than one)
        --b;
        Tb -= (int64_t)a.Hkv * tiles_per_pair(a, b);
      }
      const int nt = tiles_per_pair(a, b);
      const int q = (int)((last - Tb) / nt);
      const int64_t ps = Tb + (int64_t)q * nt, pe = ps + nt;
      if (pe > t1c && ps >= t0c) {
        go = 1;
        s_pair_start = ps;
        s_pair_end = pe;
        s_b = b;
        s_h = q;
      }
      s_end.T = T;
    }
    go = __shfl_sync(0xffffffffu, go, 0);
    if (lane == 0) s_go = go;
  }
  __syncthreads();
  if (!s_go) return;
  const int64_t T = s_end.T;
  const int64_t ps = s_pair_start, pe = s_pair_end;
  const int b = s_b, h = s_h;
  const int C = a.ctas;
  // CTAs covering [ps, pe): c .. cta_of(pe - 1)
  const int c_last = (int)(((pe - 1 + 1) * (int64_t)C + T - 1) / T) - 1;
  const int twoB = 2 * a.B;
  const int rows = a.R;
  for (int row = warp; row < rows; row += 4) {
    float mmax = -INFINITY;
    for (int cc = c; cc <= c_last; ++cc) {
      if (cta_begin(T, C, cc) == cta_begin(T, C, cc + 1)) continue;  // empty range: no partial
      const int slot = 2 * cc + ((cc == c && cta_begin(T, C, cc) < ps) ? 1 : 0);
      mmax = fmaxf(mmax, a.ws_ml[(size_t)slot * (NRB * kBlockRows) + row].x);
    }
    float L = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int cc = c; cc <= c_last; ++cc) {
      if (cta_begin(T, C, cc) == cta_begin(T, C, cc + 1)) continue;
      const int slot = 2 * cc + ((cc == c && cta_begin(T, C, cc) < ps) ? 1 : 0);
      const float2 ml = a.ws_ml[(size_t)slot * (NRB * kBlockRows) + row];
      const float w = exp2f(ml.x - mmax);
      L += w * ml.y;
      const float4 o = reinterpret_cast<const float4*>(
          a.ws_o + ((size_t)slot * (NRB * kBlockRows) + row) * kD)[lane];
      acc.x += w * o.x;
      acc.y += w * o.y;
      acc.z += w * o.z;
      acc.w += w * o.w;
    }
    const float inv = 1.f / L;
    const int s_slot = row / a.G, g = row % a.G;
    const size_t orow = ((size_t)b * twoB + s_slot) * a.Hq + (size_t)h * a.G + g;
    uint2 pk;
    pk.x = pack_bf16(acc.x * inv, acc.y * inv);
    pk.y = pack_bf16(acc.z * inv, acc.w * inv);
    reinterpret_cast<uint2*>(a.out + orow * kD)[lane] = pk;
    if (lane == 0 && a.lse) a.lse[orow] = (mmax + log2f(L)) * 0.69314718055994530942f;
  }
}

// ------------------------------------------------------------------------------- host
static PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = (PFN_cuTensorMapEncodeTiled_v12000)p;
  });
  return fn;
}

static bool encode_cache_map(CUtensorMap* map, const void* base, int layout, int64_t tokens,
                             int Hkv) {
  auto enc = get_encode();
  if (!enc) return false;
  cuuint64_t dims[3];
  cuuint64_t strides[2];
  cuuint32_t box[3];
  const cuuint32_t estr[3] = {1, 1, 1};
  if (layout == SIMSD_CACHE_NHD) {  // [tokens][Hkv][D]: dims (D, Hkv, tokens)
    dims[0] = kD;
    dims[1] = (cuuint64_t)Hkv;
    dims[2] = (cuuint64_t)(tokens > 0 ? tokens : 1);
    strides[0] = (cuuint64_t)kD * 2;
    strides[1] = (cuuint64_t)Hkv * kD * 2;
    box[0] = 64;
    box[1] = 1;
    box[2] = kTileKeys;
  } else {  // [Hkv][tokens][D]: dims (D, tokens, Hkv)
    dims[0] = kD;
    dims[1] = (cuuint64_t)(tokens > 0 ? tokens : 1);
    dims[2] = (cuuint64_t)Hkv;
    strides[0] = (cuuint64_t)kD * 2;
    strides[1] = (cuuint64_t)(tokens > 0 ? tokens : 1) * kD * 2;
    box[0] = 64;
    box[1] = kTileKeys;
    box[2] = 1;
  }
  const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims,
                         strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

static int rows_per_pair(const simsd_attn_params* p) { return 2 * p->B * (p->Hq / p->Hkv); }

static int grid_ctas(const simsd_attn_params* p) {
  const int sms = device_sm_count();
  return sms > 0 ? sms : 148;
}

template <int NRB>
static simsd_status launch(const simsd_attn_params* p, void* ws, size_t ws_bytes, cudaStream_t stream) {
  using C = Cfg<NRB>;
  TcArgs a;
  a.batch = p->batch;
  a.B = p->B;
  a.Hq = p->Hq;
  a.Hkv = p->Hkv;
  a.G = p->Hq / p->Hkv;
  a.R = rows_per_pair(p);
  a.nrb = NRB;
  a.ctas = grid_ctas(p);
  a.layout = (int)p->cache_layout;
  a.q = (const __nv_bfloat16*)p->q;
  a.k_resp = (const __nv_bfloat16*)p->k_resp;
  a.v_resp = (const __nv_bfloat16*)p->v_resp;
  a.cache_start = p->cache_start;
  a.prompt_len = p->prompt_len;
  a.pos_ids = p->pos_ids;
  a.labels = p->labels;
  const float scale = p->softmax_scale > 0.f ? p->softmax_scale : (float)(1.0 / sqrt((double)kD));
  a.scale_log2 = scale * 1.4426950408889634f;
  a.out = (__nv_bfloat16*)p->out;
  a.lse = p->lse;
  a.dev_err = p->dev_err;
  const size_t o_bytes = align_up((size_t)2 * a.ctas * NRB * kBlockRows * kD * sizeof(float), 256);
  const size_t ml_bytes = align_up((size_t)2 * a.ctas * NRB * kBlockRows * sizeof(float2), 256);
  if (!ws || ws_bytes < o_bytes + ml_bytes || (((uintptr_t)ws) & 255)) return SIMSD_ERR_WORKSPACE;
  a.ws_o = (float*)ws;
  a.ws_ml = (float2*)((char*)ws + o_bytes);
  make_rope_table(&a.rope, (double)p->rope_theta, kD);

  CUtensorMap tmk, tmv;
  const void* kbase = p->cache_tokens > 0 ? p->k_cache : p->k_resp;  // any valid address
  const void* vbase = p->cache_tokens > 0 ? p->v_cache : p->v_resp;
  if (!encode_cache_map(&tmk, kbase, a.layout, p->cache_tokens, p->Hkv) ||
      !encode_cache_map(&tmv, vbase, a.layout, p->cache_tokens, p->Hkv))
    return SIMSD_ERR_CUDA;

  static int attr_done[64][3];
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_done[dev][NRB]) {
    if (cudaFuncSetAttribute(attn_tc_kernel<NRB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)C::kSmemBytes) != cudaSuccess)
      return SIMSD_ERR_CUDA;
    attr_done[dev][NRB] = 1;
  }
  attn_tc_kernel<NRB><<<a.ctas, C::kThreads, C::kSmemBytes, stream>>>(tmk, tmv, a);
  simsd_status st = last_launch_status();
  if (st != SIMSD_OK) return st;
  attn_tc_merge_kernel<NRB><<<a.ctas, 128, 0, stream>>>(a);
  return last_launch_status();
}

}  // namespace tc

bool attn_tc_supported(const simsd_attn_params* p) {
  if (p->dtype != SIMSD_DTYPE_BF16 || p->D != 128) return false;
  const int R = tc::rows_per_pair(p);
  if (R > 256) return false;
  if (p->cache_tokens >= ((int64_t)1 << 31) - tc::kTileKeys) return false;
  return true;
}

size_t attn_tc_workspace(const simsd_attn_params* p) {
  const int nrb = tc::rows_per_pair(p) > 128 ? 2 : 1;
  const int ctas = tc::grid_ctas(p);
  return align_up((size_t)2 * ctas * nrb * tc::kBlockRows * tc::kD * sizeof(float), 256) +
         align_up((size_t)2 * ctas * nrb * tc::kBlockRows * sizeof(float2), 256);
}

simsd_status launch_attn_tc(const simsd_attn_params* p, void* ws, size_t ws_bytes,
                            cudaStream_t stream) {
  const uintptr_t mask = 15;
  if ((((uintptr_t)p->q) | ((uintptr_t)p->k_resp) | ((uintptr_t)p->v_resp) |
       ((uintptr_t)p->out)) & mask)
    return SIMSD_ERR_UNSUPPORTED;
  if (p->cache_tokens > 0 && ((((uintptr_t)p->k_cache) | ((uintptr_t)p->v_cache)) & mask))
    return SIMSD_ERR_UNSUPPORTED;
  if (tc::rows_per_pair(p) > 128) return tc::launch<2>(p, ws, ws_bytes, stream);
  return tc::launch<1>(p, ws, ws_bytes, stream);
}

}  // namespace simsd
