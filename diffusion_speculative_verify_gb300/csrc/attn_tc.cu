// Tensor-core (tcgen05 / TMEM) verify attention for bf16, head dim 128.
//
// What it computes (SimSD notes, "关键设计" items 2-3): for every response row of a request
// and query head, softmax attention over the request's cached prompt keys plus the
// response keys that the temporal-causal mask A_ij leaves visible, with RoPE applied to
// the response queries/keys at the copied position ids.
//
// Work decomposition. For each (request b, kv head h) the 2B*G query rows (response slot
// s, head g of the group; row = s*G + g) form a "pair". Each pair is a sequence of tiles:
// tile 0 is the response tail (the 2B response keys, rotated and masked here), tiles 1..
// stream the prompt keys, 128 at a time. All pairs' tiles, each pair with a start-up share
// (its prologue and epilogue cost in tile units), are concatenated and cut into equal
// contiguous ranges, one per schedule unit (stream-K); a unit therefore sees at most two
// partial pairs (its first and last). A pair split between units is merged inside the
// kernel: every piece but the first writes its (O, max, sum) partial to the workspace and
// publishes it with a flag; the unit holding the first piece (the last segment of its
// range, so the last piece to finish) waits for those flags and combines the partials with
// its own O, still in TMEM.
//
// A schedule unit is one CTA for pairs of up to 128 rows and, above that, a CTA pair (a
// 2-CTA cluster, rows [0, 128) and [128, 256)) whose MMAs span both CTAs (tcgen05
// cta_group::2, M = 256); each CTA of a pair loads only its half of every prompt tile, so a
// tile crosses from memory once per pair. Per CTA, warp roles:
//   producer warp  : TMA loads of prompt K and V tiles (128-byte swizzle) into a ring of
//                    three 64 KB shared-memory slots (CTA pairs: five 32 KB slots).
//   MMA warp       : one thread issues S = Q K^T (M = 128 rows, N = 128 keys, K = 128; A =
//                    the rotated Q in TMEM) into one of two TMEM S buffers, then O += P V
//                    (M = 128, N = 128 = D, K = 128 keys; A = bf16 P in TMEM) into the TMEM O
//                    accumulator; completion is signalled with tcgen05.commit to mbarriers.
//                    (CTA pairs: the even CTA's thread issues for both; the odd CTA's MMA warp
//                    forwards the completion of its own copies; Q is read from shared memory
//                    and three S buffers rotate in TMEM.)
//   softmax warps  : one thread per query row (TMEM lane). Per segment: load + rotate Q
//                    into TMEM and build the response K/V tail tile; per tile:
//                    read S from TMEM, apply the mask, and write P = 2^(s - m) (bf16) in
//                    place over the S columns just read, in one pass against the running
//                    max m unless some P would reach 2^16 (then m is raised to the tile's max
//                    and O and the P already written are rescaled);
//                    epilogue: O / l to global memory (or the partial to the workspace).
// Every wait is bounded in time (TcArgs::wait_ns). A wait that gives up raises
// SIMSD_DEVERR_TIMEOUT and sets the CTA's abort flag. The softmax warps decide to stop
// together, at the start of a segment (so none waits at a named barrier for one that has
// left); the rows the CTA has not finished are set to NaN; the producer waits for its copies
// in flight and the MMA thread for its MMAs; then the CTA frees TMEM and returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <stdio.h>

#include <atomic>
#include <mutex>

#include "attn_common.cuh"
#include "tc_ptx.cuh"

namespace simsd {
namespace tc {

constexpr int kD = 128;
constexpr int kKeys = 128;                          // prompt keys per tile
constexpr int kBlockRows = 128;
constexpr int kTileKeys = 64;                       // granularity of the host-side grid heuristic
constexpr uint64_t kDefaultWaitNs = 2000000000ull;  // 2 s: far beyond any legitimate wait
constexpr uint64_t kDrainWaitNs = 100000000ull;     // unwinding: copies / MMAs already issued
constexpr int kMaxSlots = 8;                        // ring barriers reserved in shared memory
// Start-up and finish of one pair segment (prologue, epilogue, pipeline refill) in units of
// one prompt tile's time; the schedule charges it to every pair. It grows with the response
// span (the RoPE table, the tail rows and the visibility masks scale with 2B): measured on
// GB300, 2B = 16 costs about 5 tiles and 2B = 64 about 8 to 10.
static int seg_cost_tiles(int twoB) { return 4 + twoB / 16; }
constexpr int kPrefetchAhead = 4;  // tiles before a segment's end at which the next one is prefetched
// Merge of a split pair: partials staged in shared memory two at a time.
constexpr int kMergeBatch = 2;
constexpr uint32_t kMergeO = kBlockRows * kD * 4;   // 64 KB: one piece's O rows (fp32)
constexpr uint32_t kMergeML = kBlockRows * 8;       // 1 KB: its (max, sum) per row

struct TcArgs {
  int batch, B, Hq, Hkv, G, R, ctas;  // R = 2B*G real rows per pair; ctas: schedule units
  int cl;                             // CTAs per schedule unit: 1, or 2 when R > 128
  int seg_cost;                       // virtual units charged per pair for start-up
  int layout;
  int64_t cache_tokens;               // rows of the packed prompt cache
  uint64_t wait_ns;                   // bound of every device-side wait
  const __nv_bfloat16* q;
  const __nv_bfloat16* k_resp;
  const __nv_bfloat16* v_resp;
  const int64_t* cache_start;
  const int32_t* prompt_len;
  const int32_t* pos_ids;
  const uint8_t* labels;
  float scale_log2;  // softmax scale * log2(e), folded into the rotated queries
  __nv_bfloat16* out;
  float* lse;
  uint32_t* dev_err;
  float* ws_o;         // [2 * ctas * cl][128][128] partial numerators
  float2* ws_ml;       // [2 * ctas * cl][128] partial (max, sum), log2 domain
  uint64_t* ws_flag;   // [2 * ctas * cl] partial published (the launch's token) or not
  RopeTable rope;
};

// Workspace slot of a partial: CTA `cta`, piece 0 (its range's first segment) or 1 (its last).
__host__ __device__ __forceinline__ size_t part_slot(int cta, int piece) {
  return (size_t)2 * cta + piece;
}

// ----------------------------------------------------------------------- scheduling
// Pair (b, h) has nt(b) = 1 + ceil(P_b / 128) tiles (1 for an invalid request). Besides its
// tiles it is charged `seg_cost` virtual units for its start-up and finish (prologue,
// epilogue, pipeline refill), so it spans nt(b) + seg_cost units of the virtual sequence
// that is cut into equal contiguous ranges, one per schedule unit. A range that begins inside
// a pair's start-up share starts at the pair's tile 0; one that ends inside it does not take
// the pair.
// (Checked build: a request index outside the batch reads as an invalid request.)
__device__ __forceinline__ int tiles_per_pair(const TcArgs& a, int b) {
  if (!chk(b, 1, a.batch, a.dev_err)) return 1;
  const int P = a.prompt_len[b];
  const uint8_t l0 = a.labels[(size_t)b * 2 * a.B];  // both loads issued together
  if ((P < 0) | (l0 == kLabelInvalid)) return 1;
  return 1 + (P + kKeys - 1) / kKeys;
}
__device__ __forceinline__ bool request_invalid(const TcArgs& a, int b) {
  if (!chk(b, 1, a.batch, a.dev_err)) return true;
  const int P = a.prompt_len[b];
  const uint8_t l0 = a.labels[(size_t)b * 2 * a.B];
  return (P < 0) | (l0 == kLabelInvalid);
}

// Unit c covers virtual positions [c*T/C, (c+1)*T/C).
__device__ __forceinline__ int64_t cta_begin(int64_t T, int C, int c) {
  return (T * (int64_t)c) / C;
}

struct SchedStart {
  int64_t T, t0, t1, Tb;  // virtual total, this unit's range, first position of request b
  int b;
};

// Threads 0..127 (named barrier 1): each sums the virtual lengths of a contiguous run of
// requests, a block scan places the runs, and the thread whose run holds t0 finds the
// request. Writes T, t0, t1, b and Tb to shared memory.
__device__ void block_schedule(const TcArgs& a, int c, int C, int tid, int64_t* wsum,
                               int64_t* out_T, int64_t* out_t0, int64_t* out_t1,
                               int64_t* out_Tb, int* out_b) {
  const int lane = tid & 31, w = tid >> 5;
  const int k = (a.batch + 127) >> 7;
  const int b0 = tid * k;
  int64_t sum = 0;
  for (int i = 0; i < k; ++i) {
    const int b = b0 + i;
    if (b < a.batch) sum += (int64_t)a.Hkv * (tiles_per_pair(a, b) + a.seg_cost);
  }
  int64_t incl = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int64_t n = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += n;
  }
  if (lane == 31) wsum[w] = incl;
  ptx::named_bar_sync(1, 128);
  int64_t T = 0, before = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int64_t v = wsum[i];
    before += i < w ? v : 0;
    T += v;
  }
  const int64_t excl = before + incl - sum;
  const int64_t t0 = cta_begin(T, C, c);
  if (tid == 0) {
    *out_T = T;
    *out_t0 = t0;
    *out_t1 = cta_begin(T, C, c + 1);
    if (t0 >= T) {
      *out_b = a.batch;
      *out_Tb = T;
    }
  }
  if (t0 < T && excl <= t0 && t0 < excl + sum) {  // exactly one thread
    int64_t cum = excl;
    for (int i = 0; i < k; ++i) {
      const int b = b0 + i;
      const int64_t len = (int64_t)a.Hkv * (tiles_per_pair(a, b) + a.seg_cost);
      if (t0 < cum + len) {
        *out_b = b;
        *out_Tb = cum;
        break;
      }
      cum += len;
    }
  }
}

// Walks the segments (the nonempty pieces of pairs) of one unit's virtual range.
struct SegIter {
  int64_t t, t0, t1, Tb;  // virtual: current position, the range, first position of request b
  int64_t pend, send;     // virtual ends of the current segment's pair and of the segment
  int b, nt, ppr, batch, sc;
  // current segment: kv head, first tile and tile count
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
    sc = a.seg_cost;
    nt = (b < batch) ? tiles_per_pair(a, b) : 1;
  }
  // Prepares the next nonempty segment at or after t; false when the range is exhausted.
  __device__ bool next(const TcArgs& a) {
    while (t < t1 && b < batch) {
      const int L = nt + sc;
      const int64_t rel = t - Tb;
      const int q = (int)(rel / L);
      const int64_t pstart = Tb + (int64_t)q * L;
      pend = pstart + L;
      send = pend < t1 ? pend : t1;
      i0 = max((int)(t - pstart) - sc, 0);
      n = max((int)(send - pstart) - sc, 0) - i0;
      if (n > 0) {
        h = q;
        first = (t == t0);
        full = (i0 == 0) && (send == pend);
        has_tail = (i0 == 0);
        invalid = request_invalid(a, b);
        return true;
      }
      advance(a);  // only the pair's start-up share lies in the range
    }
    return false;
  }
  __device__ void advance(const TcArgs& a) {
    t = send;
    const int64_t rend = Tb + (int64_t)ppr * (nt + sc);
    if (t >= rend) {
      Tb = rend;
      ++b;
      nt = (b < batch) ? tiles_per_pair(a, b) : 1;
    }
  }
};

// Yields the prompt tiles (kv head, first cache row) of one unit's range, in order.
struct PromptTiles {
  SegIter it;
  int i;
  bool have;
  __device__ void init(const TcArgs& a, const SchedStart& s) {
    it.init(a, s);
    have = false;
  }
  __device__ bool next(const TcArgs& a, int& h, int& tok) {
    while (true) {
      if (!have) {
        if (!it.next(a)) return false;
        have = true;
        i = it.i0;
      }
      if (!it.invalid) {
        while (i < it.i0 + it.n) {
          const int ii = i++;
          if (ii == 0) continue;
          h = it.h;
          tok = (int)(a.cache_start[it.b] + (int64_t)(ii - 1) * kKeys);  // it.b checked by it.next
          return true;
        }
      }
      it.advance(a);
      have = false;
    }
  }
};

// --------------------------------------------------------------------- small helpers
// Barriers: ring slots (full / empty); per S buffer (two, or three with CTA pairs): S
// written, the P V that read it completed, P written; Q and tail stored; MMA drain; the first
// prologue's loads landed; the partials of a split pair copied in for its merge.
enum BarIdx { kFull0 = 0, kEmpty0 = kMaxSlots, kSFull0 = 2 * kMaxSlots, kSFree0 = kSFull0 + 3,
              kPFull0 = kSFree0 + 3, kQFull = kPFull0 + 3, kDrain = kQFull + 1,
              kLoads = kDrain + 1, kMerge = kLoads + 1, kNumBars = kMerge + 1 };

struct Shared {
  uint64_t bars[kNumBars];
  uint32_t tmem_base;
  int abort;
  uint32_t peer_abort;  // CTA pairs: cluster address of the other CTA's abort flag (else 0)
  int64_t T, t0, t1, Tb;
  int b;
  int64_t wsum[4];          // block scan of the schedule
  uint32_t vis[64][2];      // per response slot: visibility bits of response keys 0-31, 32-63
};

// Sets the CTA's abort flag and, once, the timeout bit of the error word.
// In a CTA pair the other CTA's flag is raised too, so that it unwinds without waiting out
// its own limit.
__device__ __forceinline__ void raise_abort(Shared* sh, uint32_t* dev_err) {
  if (!*(volatile int*)&sh->abort) {
    *(volatile int*)&sh->abort = 1;
    atomicOr(dev_err, SIMSD_DEVERR_TIMEOUT);
    if (sh->peer_abort) ptx::st_cluster_u32(sh->peer_abort, 1u);
  }
}

// One probe of phase `parity` of mbarrier `bar`. A plain try_wait may suspend the thread
// until the phase completes; below kHintedWaitNs the wait limit is passed as the suspend-time
// hint instead, so that so short a limit can run out.
constexpr uint64_t kHintedWaitNs = 1000000ull;
__device__ __forceinline__ bool bar_try(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  return limit_ns < kHintedWaitNs ? ptx::mbar_try_wait_hint(bar, parity, (uint32_t)limit_ns)
                                  : ptx::mbar_try_wait(bar, parity);
}

// Waits for phase `parity` of mbarrier `bar`. False if the CTA is unwinding, or if the wait
// gave up after limit_ns (it then starts the unwinding).
__device__ __forceinline__ bool wait_bar(Shared* sh, uint32_t bar, uint32_t parity,
                                         uint32_t* dev_err, uint64_t limit_ns) {
  if (bar_try(bar, parity, limit_ns)) return true;
  const uint64_t t_start = ptx::globaltimer_ns();
  for (;;) {
    if (bar_try(bar, parity, limit_ns)) return true;
    if (*(volatile int*)&sh->abort) return false;
    if (ptx::globaltimer_ns() - t_start > limit_ns) {
      raise_abort(sh, dev_err);
      return false;
    }
  }
}

// Waits, bounded by kDrainWaitNs and regardless of the abort flag, for a phase that work this
// CTA has already issued completes: used for copies and MMAs in flight before the CTA exits.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
  const uint64_t t_start = ptx::globaltimer_ns();
  while (!ptx::mbar_try_wait(bar, parity) && ptx::globaltimer_ns() - t_start < kDrainWaitNs) {
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
// with chunk c + 8: elements d and d + 64) with the (cos, sin) table `cs` of its position
// (64 float2 entries, one per pair), and multiplies by `scale`.
__device__ __forceinline__ void rope_row(uint4 (&v)[16], const float2* cs, float scale) {
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    uint32_t* lo = reinterpret_cast<uint32_t*>(&v[c]);
    uint32_t* hi = reinterpret_cast<uint32_t*>(&v[c + 8]);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int d0 = 8 * c + 2 * e;
      const float4 t = *reinterpret_cast<const float4*>(cs + d0);  // cos0, sin0, cos1, sin1
      const float x0 = bf16_lo(lo[e]), x1 = bf16_hi(lo[e]);
      const float y0 = bf16_lo(hi[e]), y1 = bf16_hi(hi[e]);
      lo[e] = pack_bf16((x0 * t.x - y0 * t.y) * scale, (x1 * t.z - y1 * t.w) * scale);
      hi[e] = pack_bf16((x0 * t.y + y0 * t.x) * scale, (x1 * t.w + y1 * t.z) * scale);
    }
  }
}

// sin / cos of the RoPE angle pos * omega_d: the fraction of a turn is formed exactly as
// in rope_sincos, then the hardware approximations take it (absolute error about 2^-21 on
// [-pi, pi]). Used where the rotated values are rounded to bf16 (relative step 2^-8).
__device__ __forceinline__ void rope_sincos_fast(int pos, float c_hi, float c_lo, float* s, float* c) {
  const float x = (float)pos;
  const float a = x * c_hi;
  const float e = fmaf(x, c_hi, -a);
  const float f = (a - rintf(a)) + fmaf(x, c_lo, e);
  __sincosf(6.28318530717958647692f * f, s, c);
}

// Max over the valid entries (bit c of vm) of a 32-column chunk of fp32 scores.
__device__ __forceinline__ float chunk_max(const uint32_t (&r)[32], uint32_t vm) {
  float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
  if (vm == 0xffffffffu) {
#pragma unroll
    for (int c = 0; c < 32; ++c) mx[c & 3] = fmaxf(mx[c & 3], __uint_as_float(r[c]));
  } else {
#pragma unroll
    for (int c = 0; c < 32; ++c)
      if ((vm >> c) & 1u) mx[c & 3] = fmaxf(mx[c & 3], __uint_as_float(r[c]));
  }
  return fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
}

// p = 2^(s - m) on the valid entries (0 elsewhere) of a 32-column chunk, packed as bf16
// pairs (lower column in the low half); returns the sum of the fp32 p.
__device__ __forceinline__ float chunk_exp(const uint32_t (&r)[32], uint32_t vm, float m,
                                           uint32_t (&pk)[16]) {
  float s0 = 0.f, s1 = 0.f;
  if (vm == 0xffffffffu) {
#pragma unroll
    for (int c = 0; c < 32; c += 2) {
      const float p0 = ptx::ex2(__uint_as_float(r[c]) - m);
      const float p1 = ptx::ex2(__uint_as_float(r[c + 1]) - m);
      s0 += p0;
      s1 += p1;
      pk[c >> 1] = pack_bf16(p0, p1);
    }
  } else {
#pragma unroll
    for (int c = 0; c < 32; c += 2) {
      const float p0 = ((vm >> c) & 1u) ? ptx::ex2(__uint_as_float(r[c]) - m) : 0.f;
      const float p1 = ((vm >> (c + 1)) & 1u) ? ptx::ex2(__uint_as_float(r[c + 1]) - m) : 0.f;
      s0 += p0;
      s1 += p1;
      pk[c >> 1] = pack_bf16(p0, p1);
    }
  }
  return s0 + s1;
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

// Which tail row (response K, rotated here, or response V) softmax thread `tid` loads in a
// segment's prologue. When the threads beyond this CTA's rows (tid >= rw) can take all
// 2 * 2B tail rows ("early"), they load them together with the Q rows; otherwise threads
// 0..63 take the K rows and 64..127 the V rows (zero rows beyond 2B) once Q is in TMEM.
struct TailRole {
  int key;
  bool row, k, early;
};
__device__ __forceinline__ TailRole tail_role(int rw, int twoB, int tid, bool has_tail) {
  TailRole t;
  t.early = has_tail && 128 - rw >= 2 * twoB;
  if (t.early) {
    const int e = tid - rw;
    t.row = e >= 0 && e < 2 * twoB;
    t.k = e < twoB;
    t.key = t.k ? e : e - twoB;
  } else {
    t.key = tid & 63;
    t.row = has_tail && t.key < twoB;
    t.k = tid < 64;
  }
  return t;
}

// L2 prefetch of what the prologue of the segment (request nb, kv head nh, with a tail tile
// when ntail) loads: this thread's Q row, its tail K or V row (same thread mapping as the
// prologue) and the labels and position ids.
__device__ __forceinline__ void prefetch_prologue(const TcArgs& a, int nb, int nh, int ntail,
                                                  int twoB, int s_slot, int g, bool real, int rw,
                                                  int tid) {
  if (real) {
    const __nv_bfloat16* qrow = a.q + (((size_t)nb * twoB + s_slot) * a.Hq + (size_t)nh * a.G + g) * kD;
    asm volatile("prefetch.global.L2 [%0];" ::"l"(qrow));
    asm volatile("prefetch.global.L2 [%0];" ::"l"(qrow + 64));
  }
  const TailRole tr = tail_role(rw, twoB, tid, ntail != 0);
  if (tr.row) {
    const __nv_bfloat16* trow =
        (tr.k ? a.k_resp : a.v_resp) + (((size_t)nb * twoB + tr.key) * a.Hkv + nh) * kD;
    asm volatile("prefetch.global.L2 [%0];" ::"l"(trow));
    asm volatile("prefetch.global.L2 [%0];" ::"l"(trow + 64));
  }
  if (tid == 0) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(a.labels + (size_t)nb * twoB));
    asm volatile("prefetch.global.L2 [%0];" ::"l"(a.pos_ids + (size_t)nb * twoB));
  }
}

// A 128-element bf16 row (16 chunks) into 64 TMEM columns of this thread's lane:
// elements (2c, 2c + 1) in column c, the lower index in the low half.
__device__ __forceinline__ void tmem_st_row(uint32_t taddr, const uint4 (&v)[16]) {
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    uint32_t w[32];
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      w[4 * c] = v[8 * half + c].x;
      w[4 * c + 1] = v[8 * half + c].y;
      w[4 * c + 2] = v[8 * half + c].z;
      w[4 * c + 3] = v[8 * half + c].w;
    }
    ptx::tmem_st32(taddr + 32 * half, w);
  }
}

// Flags of published partials: written with release and read with acquire at GPU scope.
__device__ __forceinline__ uint64_t ld_acquire_u64(const uint64_t* p) {
  uint64_t v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_u64(uint64_t* p, uint64_t v) {
  asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
// The value a partial's flag takes in this launch: the grid's launch number, top bit set (so
// never 0, the value every CTA gives its own flags at entry; replays of a CUDA graph reuse
// the number, which is why flags are also cleared once merged).
__device__ __forceinline__ uint64_t launch_token() {
  uint64_t g;
  asm volatile("mov.u64 %0, %%gridid;" : "=l"(g));
  return g | (1ull << 63);
}

// This thread's output row of a segment the CTA did not finish: a whole pair's row (and its
// lse) becomes NaN, and so does a split pair's when this is its first piece (the CTA that
// merges the pair); a later piece gets a NaN partial (published like any partial), which the
// merge carries into the pair's output. Invalid requests get their zero rows as usual.
__device__ __forceinline__ void mark_unfinished(const TcArgs& a, const SegIter& it, bool real,
                                                size_t orow, size_t slot, int row) {
  if (!real) return;
  const int64_t nrows = (int64_t)a.batch * 2 * a.B * a.Hq;
  if (!chk((int64_t)orow, 1, nrows, a.dev_err) ||
      !chk((int64_t)slot * kBlockRows + row, 1, (int64_t)2 * a.ctas * a.cl * kBlockRows, a.dev_err))
    return;
  if (it.invalid) {
    uint4* o = reinterpret_cast<uint4*>(a.out + orow * kD);
#pragma unroll
    for (int c = 0; c < 16; ++c) o[c] = make_uint4(0, 0, 0, 0);
    if (a.lse) a.lse[orow] = -INFINITY;
    return;
  }
  const float qnan = __int_as_float(0x7FC00000);
  if (it.full || it.i0 == 0) {
    const uint32_t nan2 = 0x7FC07FC0u;  // two bf16 quiet NaNs
    uint4* o = reinterpret_cast<uint4*>(a.out + orow * kD);
#pragma unroll
    for (int c = 0; c < 16; ++c) o[c] = make_uint4(nan2, nan2, nan2, nan2);
    if (a.lse) a.lse[orow] = qnan;
  } else {
    a.ws_ml[slot * kBlockRows + row] = make_float2(qnan, qnan);
  }
}

// =========================================================================================
// Both MMAs take A from TMEM and run at N = 128 (measured on GB300: 64 cycles per
// 128 x 128 x 16 instruction, A from TMEM or shared memory alike, and per 256 x 128 x 16
// over a CTA pair; N = 64 runs about 1.4x slower per flop):
//   S_j = Q K_j^T   A = rotated Q (TMEM), B = K tile (smem, K-major), N = 128 keys
//   O  += P_j V_j   A = P_j (TMEM, bf16),  B = V tile (smem, MN-major), N = 128 = D
// TMEM columns: S buffers [0,128) and [128,256), O [256,384), Q [384,448). P_j (bf16 pairs,
// 64 columns) is written in place over the first columns of S_j, which the softmax has
// already read, so P double-buffers with S; an S buffer is released by the commit of the
// P V that read its P.
// CTA pairs take A of S = Q K^T from shared memory instead (this CTA's 128 rotated Q rows,
// 128-byte swizzle, behind a five-slot ring), which frees TMEM for a third S buffer:
// S [0,128), [128,256), [256,384), O [384,512). S_{j+3} then waits for P_j V_j instead of
// S_{j+2}, so the chain last P_j -> P_j V_j -> next S into that buffer has a tile of slack
// against the softmax.
// Warps 0-3: softmax (thread = row = TMEM lane; warps whose 32 rows are all padding skip
// their work), warp 4: TMA producer, warp 5: MMA issuer (non-blocking event loop).
namespace r128 {
constexpr uint32_t kHalf = kKeys * 128;          // 16 KB: one 64-element half of a K or V tile
constexpr uint32_t kKV = 2 * kHalf;              // 32 KB
constexpr uint32_t kStage = 2 * kKV;             // 64 KB: K + V
constexpr int kStages = 3;
constexpr uint32_t kTailHalf = 64 * 128;         // tail tile: 2B <= 64 keys, 64-key layout
constexpr uint32_t kTailKV = 2 * kTailHalf;      // 16 KB
constexpr uint32_t kOffStages = 0;
constexpr uint32_t kOffTail = kOffStages + kStages * kStage;  // tail K (16 KB) then V (16 KB)
constexpr uint32_t kOffBar = kOffTail + 2 * kTailKV;
constexpr uint32_t kSmemBytes = kOffBar + 2048 + 1024;        // barriers + alignment slack
constexpr int kThreads = 192;
constexpr int kProducerWarp = 4, kMmaWarp = 5;
constexpr uint32_t kTmemS0 = 0, kTmemO = 256, kTmemQ = 384, kTmemCols = 512;
static_assert(kStages <= kMaxSlots, "stage barriers");
// CTA pairs (pairs of 129..256 rows): per CTA and prompt tile, K of 64 of the tile's 128 keys
// (CTA r: keys [64 r, 64 r + 64), all dims as two 64-dim halves) then V of all 128 keys for
// 64 of the dims (CTA r: dims [64 r, 64 r + 64)); the tail tile likewise: tail K keys
// [32 r, 32 r + 32), tail V dims [64 r, 64 r + 64) of all 64 tail keys.
constexpr uint32_t kPKHalf = 64 * 128;                    // 8 KB
constexpr uint32_t kPStage = 2 * kPKHalf + kKeys * 128;   // 32 KB
constexpr int kPStages = 5;
constexpr uint32_t kPTailKHalf = 32 * 128;                // 4 KB
constexpr uint32_t kPOffQ = kOffStages + kPStages * kPStage;  // 32 KB: Q as two 64-dim halves
constexpr uint32_t kPTmemO = 384;
static_assert(kPOffQ + 2 * kHalf == kOffTail, "ring + Q of a CTA pair fill the single-CTA ring");
static_assert(kPStages <= kMaxSlots, "stage barriers");
}  // namespace r128

// kPair: the two CTAs of a schedule unit form a cluster and one tcgen05.mma (cta_group::2,
// M = 256) covers both 128-row blocks; each CTA loads only its half of every K and V tile
// (above), so a tile crosses from memory once per pair; the ring holds five tiles, Q sits
// in shared memory and three S buffers rotate in TMEM.
// The even CTA issues every MMA; the odd CTA's MMA warp forwards the completion of its own
// copies to the even CTA's ring barriers.
template <bool kPair>
__global__ void __launch_bounds__(r128::kThreads, 1)
    attn_tc128_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                      const __grid_constant__ TcArgs a) {
  using namespace r128;
  static_assert(sizeof(Shared) <= 2048, "barrier area");
  static_assert(kSmemBytes <= 232448, "shared memory per CTA");
  constexpr uint32_t STG = kPair ? kPStage : kStage;    // bytes of one ring stage
  constexpr int NSTG = kPair ? kPStages : kStages;      // ring stages
  constexpr uint32_t KHALF = kPair ? kPKHalf : kHalf;   // one 64-dim half of a stage's K
  constexpr uint32_t VOFF = 2 * KHALF;                  // V within a stage
  constexpr uint32_t TKHALF = kPair ? kPTailKHalf : kTailHalf;
  constexpr int MROWS = kPair ? 256 : 128;              // rows of one MMA
  constexpr int NSB = kPair ? 3 : 2;                    // S buffers in TMEM
  constexpr uint32_t TMO = kPair ? kPTmemO : kTmemO;    // O accumulator column
  // (No early launch_dependents: a following call on the same workspace must not start
  // while this grid's CTAs still merge split pairs.)
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  Shared* sh = reinterpret_cast<Shared*>(smem + kOffBar);
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const uint32_t sbase = ptx::smem_u32(smem);
  auto bar = [&](int i) { return ptx::smem_u32(&sh->bars[i]); };
  // Pairs of more than 128 rows: two CTAs take each schedule unit, CTA `crank` the rows
  // [128 crank, 128 crank + 128). Without kPair they are independent (each loads the unit's
  // whole prompt tiles) and differ only in their rows; with kPair they are the two halves of
  // one MMA unit (cluster rank = crank).
  const int cl = a.cl;
  const int vcta = blockIdx.x / cl, crank = blockIdx.x - vcta * cl;
  const int row0 = crank * 128;  // first pair row of this CTA
  const uint64_t wait_ns = a.wait_ns;
  // Tile j uses S buffer j % NSB. kPFull0 + b: P of the tile in S buffer b written.
  // kSFree0 + b: the P V that read S buffer b completed; its phase for tile j is j / NSB, and
  // the previous phase (tile j - NSB) is always complete by the time anyone waits for tile j,
  // so a parity wait is unambiguous.
  // With kPair, the ring barriers count this CTA's own copies; the even CTA's full barriers
  // also wait for the odd CTA's forwarded arrival, and its P and Q barriers count one arrival
  // per softmax warp of both CTAs. Every other barrier is arrived at by MMA commits, in both
  // CTAs at once.

  // This CTA's boxes of prompt tile (kv head h, first key tok): K as two 64-dim halves, then
  // V, into the stage at `dst` (counted on `fbar`); !load: into L2 only.
  auto tile_boxes = [&](int h, int tok, bool load, uint32_t dst, uint32_t fbar) {
    auto box = [&](const CUtensorMap* map, int d0, int key0, uint32_t to) {
      const int c1 = a.layout == SIMSD_CACHE_NHD ? h : key0;
      const int c2 = a.layout == SIMSD_CACHE_NHD ? key0 : h;
      if (load)
        ptx::tma_load_3d(to, map, d0, c1, c2, fbar);
      else
        ptx::tma_prefetch_3d(map, d0, c1, c2);
    };
    const int ktok = kPair ? tok + 64 * crank : tok;
#pragma unroll
    for (int half = 0; half < 2; ++half) box(&tmk, half * 64, ktok, dst + half * KHALF);
    if constexpr (kPair) {
      box(&tmv, 64 * crank, tok, dst + VOFF);
    } else {
#pragma unroll
      for (int half = 0; half < 2; ++half) box(&tmv, half * 64, tok, dst + VOFF + half * kHalf);
    }
  };

  if (warp == kProducerWarp) {
    if (lane == 0) {
      // (launched as a programmatic dependent of the layout kernel: no input is read before
      // that grid has completed)
      asm volatile("griddepcontrol.wait;" ::: "memory");
      // When every unit is one pair, this unit's pair is known before the schedule: its
      // first prompt tiles go into L2 now, so that the stream, which starts after the first
      // prologue, finds them there.
      if ((int64_t)a.batch * a.Hkv == (int64_t)a.ctas && chk(vcta / a.Hkv, 1, a.batch, a.dev_err)) {
        const int gb = vcta / a.Hkv, gh = vcta - (vcta / a.Hkv) * a.Hkv;
        const int P = a.prompt_len[gb];
        const int64_t cs = a.cache_start[gb];
        const int n = min(kStages, (max(P, 0) + kKeys - 1) / kKeys);
        for (int i = 0; i < n; ++i) {
          const int tok = (int)(cs + (int64_t)i * kKeys);
          if (!chk(tok, 1, a.cache_tokens, a.dev_err)) break;
          tile_boxes(gh, tok, false, 0u, 0u);
        }
      }
      sh->abort = 0;
      sh->peer_abort = kPair ? ptx::mapa(ptx::smem_u32(&sh->abort), (uint32_t)(crank ^ 1)) : 0u;
      const bool lead = kPair && crank == 0;
      for (int i = 0; i < NSTG; ++i) {
        ptx::mbar_init(bar(kFull0 + i), lead ? 2 : 1);
        ptx::mbar_init(bar(kEmpty0 + i), 1);
      }
      for (int i = 0; i < NSB; ++i) {
        ptx::mbar_init(bar(kSFull0 + i), 1);
        ptx::mbar_init(bar(kSFree0 + i), 1);
        ptx::mbar_init(bar(kPFull0 + i), kPair ? 8 : 128);
      }
      ptx::mbar_init(bar(kQFull), kPair ? 8 : 128);
      ptx::mbar_init(bar(kDrain), 1);
      ptx::mbar_init(bar(kLoads), 128);
      ptx::mbar_init(bar(kMerge), 1);
      ptx::fence_mbar_init();
      ptx::prefetch_tensormap(&tmk);
      ptx::prefetch_tensormap(&tmv);
    }
  } else if (warp == kMmaWarp) {
    if constexpr (kPair) {
      ptx::tmem_alloc_pair(ptx::smem_u32(&sh->tmem_base), kTmemCols);
      ptx::tmem_relinquish_pair();
    } else {
      ptx::tmem_alloc(ptx::smem_u32(&sh->tmem_base), kTmemCols);
      ptx::tmem_relinquish();
    }
  } else {
    {  // Before the schedule is known: this unit's likely first pair (exact when every unit
       // is one whole pair) has its prologue rows prefetched into L2, so that the first
       // prologue's loads hit there instead of paying a cold access after the schedule.
      const int64_t pairs = (int64_t)a.batch * a.Hkv;
      const int64_t gp = pairs > 0 ? ((int64_t)vcta * pairs) / a.ctas : 0;
      const int gb = (int)(gp / a.Hkv), gh = (int)(gp % a.Hkv);
      const int prow = row0 + tid;
      const bool real = prow < a.R;
      const int rw = (min(128, a.R - row0) + 31) & ~31;
      if (gb < a.batch)
        prefetch_prologue(a, gb, gh, 1, 2 * a.B, real ? prow / a.G : 0, real ? prow % a.G : 0,
                          real, rw, tid);
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");  // (the schedule reads the labels)
    block_schedule(a, vcta, a.ctas, tid, sh->wsum, &sh->T, &sh->t0, &sh->t1, &sh->Tb, &sh->b);
  }
  asm volatile("griddepcontrol.wait;" ::: "memory");  // every thread, before its first input read
  ptx::tc_fence_before();
  if constexpr (kPair) {
    ptx::cluster_sync();  // both CTAs' barriers exist before either arrives on the other's
  } else {
    __syncthreads();
  }
  ptx::tc_fence_after();

  SchedStart st;
  st.T = sh->T;
  st.t0 = sh->t0;
  st.t1 = sh->t1;
  st.Tb = sh->Tb;
  st.b = sh->b;
  const uint32_t tmem = sh->tmem_base;
  const int twoB = 2 * a.B;

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      PromptTiles tiles;
      tiles.init(a, st);
      uint32_t p = 0;  // tiles loaded (ring position)
      bool ok = true, first = true;
      int h, tok;
      while (ok && tiles.next(a, h, tok)) {
        // the first prologue's global loads are issued before the prompt stream, so that
        // they are not queued behind it (the first tile the MMA issuer needs is the tail
        // tile, which the prologue builds in shared memory)
        if (first) {
          first = false;
          ok = wait_bar(sh, bar(kLoads), 0, a.dev_err, wait_ns);
          if (!ok) break;
        }
        const int s = p % NSTG;
        ok = wait_bar(sh, bar(kEmpty0 + s), ((p / NSTG) & 1) ^ 1, a.dev_err, wait_ns);
        if (!ok) break;
        // checked build: a tile row outside the cache or a head outside Hkv is not copied
        // (the stage completes without data, the error word records it)
        if (!chk(tok, 1, a.cache_tokens, a.dev_err) || !chk(h, 1, a.Hkv, a.dev_err)) {
          ptx::mbar_arrive(bar(kFull0 + s));
          ++p;
          continue;
        }
        ptx::mbar_arrive_expect_tx(bar(kFull0 + s), STG);
        tile_boxes(h, tok, true, sbase + kOffStages + s * STG, bar(kFull0 + s));
        ++p;
      }
      // Whether the stream ended or the CTA is unwinding, the copies issued last may still be
      // in flight; they land before the CTA can exit (earlier ones have been consumed). (The
      // even CTA of a pair counts the odd CTA's forwarded arrival on the same barriers: if
      // that one never comes, the bounded drain gives up.)
      for (uint32_t k = p > (uint32_t)NSTG ? p - NSTG : 0; k < p; ++k)
        drain_wait(bar(kFull0 + k % NSTG), (k / NSTG) & 1);
    }
  } else if (warp == kMmaWarp) {
    if (kPair && crank != 0 && lane == 0) {
      // ------------------------------------------------- copy completion forwarder (odd CTA)
      // The even CTA issues the MMAs that read this CTA's half of every stage: each stage's
      // completion here becomes one arrival on the even CTA's full barrier of that stage, in
      // ring order (the producer fills stages in that order; a stage is refilled only after
      // the MMAs, which wait for this arrival, have released it).
      PromptTiles tiles;
      tiles.init(a, st);
      int h, tok;
      for (uint32_t p = 0; tiles.next(a, h, tok); ++p) {
        const int s = p % NSTG;
        if (!wait_bar(sh, bar(kFull0 + s), (p / NSTG) & 1, a.dev_err, wait_ns)) break;
        ptx::mbar_arrive_remote(ptx::mapa(bar(kFull0 + s), 0u));
      }
    }
    // ------------------------------------------------------------------- MMA issuer
    if (lane == 0 && (!kPair || crank == 0)) {
      constexpr uint32_t idS = ptx::idesc_bf16(MROWS, kKeys, 0, 0);
      constexpr uint32_t idS_tail = ptx::idesc_bf16(MROWS, 64, 0, 0);
      constexpr uint32_t idPV = ptx::idesc_bf16(MROWS, kD, 0, 1);
      auto mma = [&](uint32_t d, uint32_t at, uint64_t bd, uint32_t id, uint32_t acc) {
        if constexpr (kPair)
          ptx::mma_f16_ts_pair(d, at, bd, id, acc);
        else
          ptx::mma_f16_ts(d, at, bd, id, acc);
      };
      // S = Q K^T, K step kk: A = Q from TMEM, or with kPair from shared memory
      auto mma_s = [&](uint32_t d, int kk, uint64_t bd, uint32_t id, uint32_t acc) {
        if constexpr (kPair)
          ptx::mma_f16_ss_pair(d, ptx::sdesc_sw128(sbase + kPOffQ + (kk >> 2) * kHalf + (kk & 3) * 32, 16, 1024),
                               bd, id, acc);
        else
          ptx::mma_f16_ts(d, tmem + kTmemQ + kk * 8, bd, id, acc);
      };
      auto commit = [&](uint32_t b) {  // with kPair: the barrier of both CTAs
        if constexpr (kPair)
          ptx::mma_commit_pair_both(b);
        else
          ptx::mma_commit(b);
      };
      SegIter it;
      it.init(a, st);
      uint32_t j = 0, m = 0, nseg = 0;
      bool ok = true;
      // Polls (no suspend) until the segment's Q and tail are stored; false once the CTA
      // unwinds or after wait_ns.
      auto poll_qfull = [&]() -> bool {
        const uint64_t t_start = ptx::globaltimer_ns();
        uint32_t spin = 0;
        while (!ptx::mbar_test(bar(kQFull), nseg & 1)) {
          if ((++spin & 255) == 0) {
            if (*(volatile int*)&sh->abort) return false;
            if (ptx::globaltimer_ns() - t_start > wait_ns) {
              raise_abort(sh, a.dev_err);
              return false;
            }
          }
        }
        return true;
      };
      // Called when the issue loop made no progress: true once it has gone wait_ns without
      // any (then the CTA unwinds) or the CTA is unwinding.
      uint32_t spins = 0;
      uint64_t t_idle = 0;
      auto stalled = [&]() -> bool {
        if ((++spins & 63) != 0) return false;
        const uint64_t now = ptx::globaltimer_ns();
        if (spins == 64) t_idle = now;
        if (*(volatile int*)&sh->abort || now - t_idle > wait_ns) {
          raise_abort(sh, a.dev_err);
          return true;
        }
        return false;
      };
      int stage_of[8];  // per tile (ring): slot to release after its P V, -1 = tail tile
      static_assert(NSB + 1 <= 8, "tile ring");
      auto try_issue_s = [&](uint32_t jj, int i) -> bool {
        const int buf = jj % NSB;
        const int s = m % NSTG;
        if (i != 0 && !ptx::mbar_test(bar(kFull0 + s), (m / NSTG) & 1)) return false;
        if (!ptx::mbar_test(bar(kSFree0 + buf), ((jj / NSB) & 1) ^ 1)) return false;
        ptx::tc_fence_after();
        const uint32_t d = tmem + kTmemS0 + buf * 128;
        if (i == 0) {
          const uint32_t kaddr = sbase + kOffTail;
#pragma unroll
          for (int kk = 0; kk < kD / 16; ++kk)
            mma_s(d, kk, ptx::sdesc_sw128(kaddr + (kk >> 2) * TKHALF + (kk & 3) * 32, 16, 1024), idS_tail,
                  kk > 0 ? 1u : 0u);
          stage_of[jj & 7] = -1;
        } else {
          const uint32_t kaddr = sbase + kOffStages + s * STG;
#pragma unroll
          for (int kk = 0; kk < kD / 16; ++kk)
            mma_s(d, kk, ptx::sdesc_sw128(kaddr + (kk >> 2) * KHALF + (kk & 3) * 32, 16, 1024), idS,
                  kk > 0 ? 1u : 0u);
          stage_of[jj & 7] = s;
          ++m;
        }
        commit(bar(kSFull0 + buf));
        return true;
      };
      // V as B is N-major: 16 keys (rows of 128 bytes) per K step; with kPair each CTA holds
      // a single 64-dim column of atoms, so the leading (N) offset is never used.
      auto try_issue_pv = [&](uint32_t jj, bool first_in_seg) -> bool {
        const int buf = jj % NSB;
        if (!ptx::mbar_test(bar(kPFull0 + buf), (jj / NSB) & 1)) return false;
        ptx::tc_fence_after();
        const int s = stage_of[jj & 7];
        const uint32_t vaddr = s < 0 ? sbase + kOffTail + kTailKV : sbase + kOffStages + s * STG + VOFF;
        const uint32_t lbo = s < 0 ? kTailHalf : kHalf;
        const int nk = s < 0 ? 4 : kKeys / 16;
        for (int kk = 0; kk < nk; ++kk)
          mma(tmem + TMO, tmem + kTmemS0 + buf * 128 + kk * 8,
              ptx::sdesc_sw128(vaddr + kk * 16 * 128, lbo, 1024), idPV, (first_in_seg && kk == 0) ? 0u : 1u);
        commit(bar(kSFree0 + buf));
        if (s >= 0) commit(bar(kEmpty0 + s));
        return true;
      };
      while (ok && it.next(a)) {
        if (it.invalid) {
          it.advance(a);
          continue;
        }
        if (!poll_qfull()) {  // the segment cannot start before Q is in TMEM
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t jfirst = j, jend = j + (uint32_t)it.n;
        uint32_t ns = jfirst, npv = jfirst;
        spins = 0;
        while (npv < jend) {
          bool progressed = false;
          if (npv < ns && try_issue_pv(npv, npv == jfirst)) {
            ++npv;
            progressed = true;
          }
          if (ns < jend && ns <= npv + NSB && try_issue_s(ns, it.i0 + (int)(ns - jfirst))) {
            ++ns;
            progressed = true;
          }
          if (progressed) {
            spins = 0;
          } else if (stalled()) {
            ok = false;
            break;
          }
        }
        if (!ok) break;
        j = jend;
        ++nseg;
        it.advance(a);
      }
      // every MMA issued has completed before TMEM is freed
      if constexpr (kPair)
        ptx::mma_commit_pair_own(bar(kDrain));
      else
        ptx::mma_commit(bar(kDrain));
      drain_wait(bar(kDrain), 0);
    }
  } else {
    // -------------------------------------------------------------- softmax warps
    const int row = warp * 32 + lane;  // TMEM lane = row within this CTA's block
    const int prow = row0 + row;       // row within the pair
    const bool real = prow < a.R;
    const bool warp_active = row0 + warp * 32 < a.R;  // warp-uniform: some row of this warp is real
    const int s_slot = real ? prow / a.G : 0;
    const int g = real ? prow % a.G : 0;
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    const uint32_t tmem_o = tmem + lane_off + TMO;
    uint8_t* tailk = smem + kOffTail;
    uint8_t* tailv = tailk + kTailKV;
    const int rw = (min(128, a.R - row0) + 31) & ~31;  // threads below rw own this block's rows
    // Arrival on the Q / P barriers: each thread, or with kPair one per warp on the even
    // CTA's barrier (after every lane's TMEM stores and fences).
    auto arrive_x = [&](int i) {
      if constexpr (kPair) {
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive_remote(ptx::mapa(bar(i), 0u));
      } else {
        ptx::mbar_arrive(bar(i));
      }
    };
    // Split pairs. This CTA's two partial slots (its range's first and last segment) are
    // published by setting their flags to the launch token once every row is written; the
    // flags are cleared here first (and by the merging CTA once consumed), so a flag left
    // over from an earlier launch is gone long before any CTA of this one looks at it.
    const uint64_t token = launch_token();
    const int64_t nslots = (int64_t)2 * a.ctas * a.cl;
    if (tid == 0 && chk((int64_t)2 * blockIdx.x + 1, 1, nslots, a.dev_err)) {
      a.ws_flag[2 * blockIdx.x] = 0;
      a.ws_flag[2 * blockIdx.x + 1] = 0;
    }
    // every softmax thread, once its row of the partial in `pslot` is written
    auto publish = [&](size_t pslot) {
      __threadfence();
      ptx::named_bar_sync(1, 128);
      if (tid == 0 && chk((int64_t)pslot, 1, nslots, a.dev_err)) st_release_u64(a.ws_flag + pslot, token);
    };
    SegIter it;
    it.init(a, st);
    uint32_t j = 0;
    bool aborted = false;
    bool loads_signalled = false;  // each thread arrives on kLoads once
    while (it.next(a)) {
      // Every softmax thread reaches this point once per segment: the decision to unwind is
      // taken here by all of them together (the flag may be raised while they read it, so
      // the barrier reduces what each saw to one answer).
      if (ptx::bar_or(1, 128, *(volatile int*)&sh->abort != 0)) {
        aborted = true;
        break;
      }
      const int b = it.b, h = it.h;
      const size_t orow = ((size_t)b * twoB + s_slot) * a.Hq + (size_t)h * a.G + g;
      const size_t slot = part_slot(blockIdx.x, it.first ? 0 : 1);
      if (it.invalid) {
        mark_unfinished(a, it, real, orow, slot, row);  // zero rows, lse = -inf
        if (tid == 0 && h == 0 && a.prompt_len[b] < 0) atomicOr(a.dev_err, SIMSD_DEVERR_PROMPT_LEN);
        it.advance(a);
        continue;
      }
      bool ok = true;
      float m_used = -INFINITY, l = 0.f;  // running max (log2 domain) and sum of this segment
      do {
        const int P = a.prompt_len[b];
        const bool has_tail = it.has_tail;
        // ---- prologue: rotated + scaled Q rows into TMEM, rotated tail K and plain tail V
        // tiles. Each thread holds at most one row.
        const TailRole tr = tail_role(kPair ? 128 : rw, twoB, tid, has_tail);  // kPair: never early
        // labels and position ids of the 2B response slots: every warp holds slot `lane` and
        // slot 32 + lane, and hands them out by shuffles (no shared-memory round trip). The
        // row loads come after the table and the masks: issued first, their many requests
        // held up every shuffle behind them (measured: 4x slower loops).
        const size_t lrow = (size_t)b * twoB;
        // checked build: the request's labels / positions, this thread's Q row and tail row
        // lie inside their arrays (a row outside is not loaded)
        const bool lab_ok = chk((int64_t)lrow, twoB, (int64_t)a.batch * twoB, a.dev_err);
        const uint32_t lab_lo = lab_ok && lane < twoB ? a.labels[lrow + lane] : 0u;
        const uint32_t lab_hi = lab_ok && lane + 32 < twoB ? a.labels[lrow + 32 + lane] : 0u;
        const int pos_lo = lab_ok && lane < twoB ? a.pos_ids[lrow + lane] : 0;
        const int pos_hi = lab_ok && lane + 32 < twoB ? a.pos_ids[lrow + 32 + lane] : 0;
        uint4 v[16];
        const size_t tidx = (((size_t)b * twoB + (tr.row ? tr.key : 0)) * a.Hkv + h) * kD;
        const __nv_bfloat16* trow = (tr.k ? a.k_resp : a.v_resp) + tidx;
        const bool q_ok = chk((int64_t)orow * kD, kD, (int64_t)a.batch * twoB * a.Hq * kD, a.dev_err);
        const bool t_ok = !tr.row || chk((int64_t)tidx, kD, (int64_t)a.batch * twoB * a.Hkv * kD, a.dev_err);
        if (!tr.early && tr.row) {  // into L2 now, into registers once Q is in TMEM
          asm volatile("prefetch.global.L2 [%0];" ::"l"(trow));
          asm volatile("prefetch.global.L2 [%0];" ::"l"(trow + 64));
        }
        // (cos, sin) of the 2B response positions, over the tail K and V area (2B <= 64:
        // at most 32 KB); the tail rows are stored once every read of the table is done.
        // Rows are 66 float2 apart where that fits (16 bytes of padding: threads reading
        // different positions' rows then hit different banks), else 64. Thread t fills pair
        // t % 64 of the slots t / 64, t / 64 + 2, ... (the slot is warp-uniform).
        float2* rtab = reinterpret_cast<float2*>(tailk);
        const int tstride = twoB * 66 * 8 <= (int)(2 * kTailKV) ? 66 : 64;
        {
          const int d = tid & 63;
          const float c_hi = a.rope.c_hi[d], c_lo = a.rope.c_lo[d];
          for (int sidx = tid >> 6; sidx < twoB; sidx += 2) {
            const int ps = __shfl_sync(0xffffffffu, sidx < 32 ? pos_lo : pos_hi, sidx & 31);
            float sn, cs;
            rope_sincos_fast(ps, c_hi, c_lo, &sn, &cs);
            rtab[sidx * tstride + d] = make_float2(cs, sn);
          }
        }
        // visibility of the 2B response keys from each response slot: one ballot per slot and
        // key half (lane l evaluates keys l and 32 + l); warp w takes slots w, w + 4, ...
        if (has_tail) {
          const int th_lo = row_threshold((uint8_t)lab_lo), th_hi = row_threshold((uint8_t)lab_hi);
          for (int sl = warp; sl < twoB; sl += 4) {
            const int th = __shfl_sync(0xffffffffu, sl < 32 ? th_lo : th_hi, sl & 31);
            const uint32_t b0 = __ballot_sync(0xffffffffu, lane < twoB && response_key_visible((uint8_t)lab_lo, th));
            const uint32_t b1 =
                __ballot_sync(0xffffffffu, lane + 32 < twoB && response_key_visible((uint8_t)lab_hi, th));
            if (lane == 0) {
              sh->vis[sl][0] = b0;
              sh->vis[sl][1] = b1;
            }
          }
        }
        if (warp_active) {
          if (real && q_ok) load_row(v, a.q + orow * kD);
        } else if (tr.early && tr.row && t_ok) {
          load_row(v, trow);
        }
        // The prompt stream may start once every row this prologue loads is in flight (issued
        // first, they are not queued behind it): here, unless the tail rows come after Q.
        auto signal_loads = [&]() {
          if (!loads_signalled) {
            ptx::mbar_arrive(bar(kLoads));
            loads_signalled = true;
          }
        };
        if (tr.early || !has_tail) signal_loads();
        ptx::named_bar_sync(1, 128);
        // this row's visibility bits (bit k of vis0 / vis1 = key k / 32 + k); padding rows see
        // every response key (their scores stay finite)
        uint32_t vis0 = 0, vis1 = 0;
        if (has_tail) {
          if (real) {
            vis0 = sh->vis[s_slot][0];
            vis1 = sh->vis[s_slot][1];
          } else {
            vis0 = twoB >= 32 ? 0xffffffffu : ((1u << twoB) - 1u);
            vis1 = twoB >= 64 ? 0xffffffffu : (twoB > 32 ? ((1u << (twoB - 32)) - 1u) : 0u);
          }
        }
        if (warp_active) {
          if (real) {
            rope_row(v, rtab + s_slot * tstride, a.scale_log2);
          } else {
#pragma unroll
            for (int c = 0; c < 16; ++c) v[c] = make_uint4(0, 0, 0, 0);
          }
          if constexpr (kPair) {
            store_row_sw(smem + kPOffQ, kHalf, row, v);  // A of S, K-major, 128-byte swizzle
          } else {
            // row -> TMEM lane, dims (2c, 2c+1) -> column c (bf16 pair, low half first)
            tmem_st_row(tmem + lane_off + kTmemQ, v);
            ptx::tmem_st_wait();
          }
        } else if (tr.early && tr.row && tr.k) {
          rope_row(v, rtab + tr.key * tstride, 1.f);  // K rotated, V as is
        }
        if constexpr (kPair) {
          // this CTA's part of the tail tile: threads 0..31 tail K rows 32 crank + t (all dims,
          // rotated), threads 64..127 dims [64 crank, 64 crank + 64) of tail V row t - 64;
          // rows at or beyond 2B are zero
          if (has_tail && (tid < 32 || tid >= 64)) {
            const bool isk = tid < 32;
            const int key = isk ? 32 * crank + tid : tid - 64;
            const bool ld = key < twoB;
            const size_t pidx = (((size_t)b * twoB + (ld ? key : 0)) * a.Hkv + h) * kD;
#pragma unroll
            for (int c = 0; c < 16; ++c) v[c] = make_uint4(0, 0, 0, 0);
            if (ld && chk((int64_t)pidx, kD, (int64_t)a.batch * twoB * a.Hkv * kD, a.dev_err)) {
              if (isk) {
                load_row(v, a.k_resp + pidx);
                signal_loads();
                rope_row(v, rtab + key * tstride, 1.f);
              } else {
                const uint4* src = reinterpret_cast<const uint4*>(a.v_resp + pidx + 64 * crank);
#pragma unroll
                for (int c = 0; c < 8; ++c) v[c] = __ldg(src + c);
              }
            }
          }
        } else if (!tr.early && has_tail) {
          if (tr.row && t_ok) {
            load_row(v, trow);
            signal_loads();
            if (tr.k) rope_row(v, rtab + tr.key * tstride, 1.f);  // K rotated, V as is
          } else {
#pragma unroll
            for (int c = 0; c < 16; ++c) v[c] = make_uint4(0, 0, 0, 0);
          }
        }
        signal_loads();  // (threads without a tail row)
        ptx::named_bar_sync(1, 128);  // table reads done
        if constexpr (kPair) {
          if (has_tail) {
            if (tid < 32) {
              store_row_sw(tailk, kPTailKHalf, tid, v);
            } else if (tid >= 64) {
#pragma unroll
              for (int c = 0; c < 8; ++c) *reinterpret_cast<uint4*>(tailv + sw128(tid - 64, c)) = v[c];
            }
          }
        } else if (tr.early) {
          if (tr.row) store_row_sw(tr.k ? tailk : tailv, kTailHalf, tr.key, v);
          // keys 2B .. 63 of both tail tiles are zero (the tail MMAs read 64 keys)
          const uint4 z[16] = {};
          for (int e = tid; e < 2 * (64 - twoB); e += 128) {
            const int zk = twoB + e % (64 - twoB);
            store_row_sw(e < 64 - twoB ? tailk : tailv, kTailHalf, zk, z);
          }
        } else if (has_tail) {
          store_row_sw(tr.k ? tailk : tailv, kTailHalf, tr.key, v);
        }
        ptx::fence_proxy_async_smem();
        ptx::tc_fence_before();
        arrive_x(kQFull);
        const uint32_t jfirst = j;
        // The next segment's Q rows, tail rows and labels go into L2 a few tiles before this
        // segment ends, so that its prologue does not wait behind the K/V stream in flight.
        int pf_b = -1, pf_h = 0;  // next segment: request, kv head | has_tail << 16
        {
          SegIter nx = it;
          nx.advance(a);
          if (nx.next(a) && !nx.invalid) {
            pf_b = nx.b;
            pf_h = nx.h | (nx.has_tail ? 1 << 16 : 0);
          }
        }
        const int pf_at = max(it.i0, it.i0 + it.n - kPrefetchAhead);
        // S buffer j % NSB and its phase (j / NSB) & 1, advanced with j
        int buf = (int)(j % NSB);
        uint32_t ph = (j / NSB) & 1;
        for (int i = it.i0; i < it.i0 + it.n;
             ++i, ++j, buf = (buf + 1 == NSB) ? 0 : buf + 1, ph ^= (buf == 0) ? 1u : 0u) {
          if (pf_b >= 0 && i == pf_at)
            prefetch_prologue(a, pf_b, pf_h & 0xffff, pf_h >> 16, twoB, s_slot, g, real, rw, tid);
          // S is usually complete already: one probe and one vote, else the bounded wait
          if (!__all_sync(0xffffffffu, ptx::mbar_test(bar(kSFull0 + buf), ph)))
            ok = __all_sync(0xffffffffu, wait_bar(sh, bar(kSFull0 + buf), ph, a.dev_err, wait_ns));
          if (!ok) break;
          if (!warp_active) {  // padding rows only: keep the P barrier's count, skip the work
            arrive_x(kPFull0 + buf);
            continue;
          }
          ptx::tc_fence_after();
          const uint32_t ts = tmem + lane_off + kTmemS0 + buf * 128;
          const int nchunks = (i == 0) ? 2 : kKeys / 32;  // warp-uniform
          const int nvalid = (i == 0) ? 0 : P - (i - 1) * kKeys;
          // valid-column bits of 32-column chunk k
          auto chunk_mask = [&](int k) -> uint32_t {
            if (i == 0) return k == 0 ? vis0 : vis1;
            const int n = nvalid - 32 * k;
            return n >= 32 ? 0xffffffffu : (n <= 0 ? 0u : ((1u << n) - 1u));
          };
          // One pass in the common case: chunk k's P = 2^(s - m), m the running max, goes in
          // place over S columns [16k, 16k + 16), which this thread has already read, once the
          // warp has checked that no row's chunk sum reached 2^16 (so every P of the chunk is
          // below 2^16; no max pass is needed for that). Otherwise, and for a row that has no
          // max yet (a segment's first scores), the tile's max is taken over the remaining
          // chunks, O and the P chunks already written are rescaled, and it goes on. With CTA
          // pairs (softmax-bound) chunks go two at a time (nchunks is even): one load wait and
          // one vote per 64 columns; the single-CTA kernel (stream-bound) measured faster with
          // one chunk at a time.
          float lsum = 0.f;
          int k = 0;
          bool grew = __any_sync(0xffffffffu, m_used == -INFINITY);
          if (!grew && !kPair) {
#pragma unroll 1
            for (; k < nchunks; ++k) {
              uint32_t r[32];
              ptx::tmem_ld32(ts + 32 * k, r);
              ptx::tmem_ld_wait(r);
              uint32_t pk[16];
              const float cs = chunk_exp(r, chunk_mask(k), m_used, pk);
              if (__any_sync(0xffffffffu, !(cs < 65536.f))) {  // (a NaN sum takes the slow path)
                grew = true;
                break;
              }
              lsum += cs;
              ptx::tmem_st16(ts + 16 * k, pk);
            }
          } else if (!grew) {
#pragma unroll 1
            for (; k < nchunks; k += 2) {
              uint32_t r[32], r2[32];
              ptx::tmem_ld32(ts + 32 * k, r);
              ptx::tmem_ld32(ts + 32 * k + 32, r2);
              ptx::tmem_ld_wait(r);
              ptx::tmem_ld_wait(r2);
              uint32_t pk[16], pk2[16];
              const float cs = chunk_exp(r, chunk_mask(k), m_used, pk);
              const float cs2 = chunk_exp(r2, chunk_mask(k + 1), m_used, pk2);
              if (__any_sync(0xffffffffu, !(cs < 65536.f) || !(cs2 < 65536.f))) {  // (NaN: slow path)
                grew = true;
                break;
              }
              lsum += cs + cs2;
              ptx::tmem_st16(ts + 16 * k, pk);
              ptx::tmem_st16(ts + 16 * k + 16, pk2);
            }
          }
          if (grew) {
            float mt = -INFINITY;
#pragma unroll 1
            for (int kk = k; kk < nchunks; ++kk) {
              uint32_t r[32];
              ptx::tmem_ld32(ts + 32 * kk, r);
              ptx::tmem_ld_wait(r);
              mt = fmaxf(mt, chunk_max(r, chunk_mask(kk)));
            }
            const float m_new = fmaxf(m_used, mt);
            const float alpha = m_used == -INFINITY ? 0.f : ptx::ex2(m_used - m_new);
            if (j != jfirst) {  // O holds P V of earlier tiles: rescale it once the last P V landed
              const uint32_t jp = j - 1;
              ok = __all_sync(0xffffffffu, wait_bar(sh, bar(kSFree0 + jp % NSB), (jp / NSB) & 1,
                                                    a.dev_err, wait_ns));
              if (!ok) break;
              ptx::tc_fence_after();
              l *= alpha;
#pragma unroll 1
              for (int kk = 0; kk < 4; ++kk) {
                uint32_t o[32];
                ptx::tmem_ld32(tmem_o + 32 * kk, o);
                ptx::tmem_ld_wait(o);
#pragma unroll
                for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                ptx::tmem_st32(tmem_o + 32 * kk, o);
              }
            }
            lsum *= alpha;
#pragma unroll 1
            for (int kk = 0; kk < k; ++kk) {  // P chunks already written with the old max
              uint32_t pk[16];
              ptx::tmem_ld16(ts + 16 * kk, pk);
              ptx::tmem_ld16_wait(pk);
#pragma unroll
              for (int e = 0; e < 16; ++e) pk[e] = pack_bf16(bf16_lo(pk[e]) * alpha, bf16_hi(pk[e]) * alpha);
              ptx::tmem_st16(ts + 16 * kk, pk);
            }
            m_used = m_new;
            const float msafe = m_used == -INFINITY ? 0.f : m_used;
#pragma unroll 1
            for (; k < nchunks; ++k) {
              uint32_t r[32], pk[16];
              ptx::tmem_ld32(ts + 32 * k, r);
              ptx::tmem_ld_wait(r);
              lsum += chunk_exp(r, chunk_mask(k), msafe, pk);
              ptx::tmem_st16(ts + 16 * k, pk);
            }
          }
          l += lsum;
          ptx::tmem_st_wait();
          ptx::tc_fence_before();
          arrive_x(kPFull0 + buf);
        }
        if (!ok) break;
        // ---- epilogue: wait for the last P V, then O / l, or, for a later piece of a split
        // pair, the partial (the pair's first piece keeps O in TMEM for the merge below)
        const uint32_t jl = j - 1;
        ok = __all_sync(0xffffffffu, wait_bar(sh, bar(kSFree0 + jl % NSB), (jl / NSB) & 1, a.dev_err, wait_ns));
        if (!ok) break;
        ptx::tc_fence_after();
        if ((it.full || it.i0 > 0) && warp_active &&
            chk((int64_t)orow * kD, kD, (int64_t)a.batch * twoB * a.Hq * kD, a.dev_err) &&
            chk((int64_t)slot * kBlockRows + row, 1, nslots * kBlockRows, a.dev_err)) {
          const float inv = it.full ? 1.f / l : 1.f;
#pragma unroll 1
          for (int k = 0; k < 4; ++k) {
            uint32_t o[32];
            ptx::tmem_ld32(tmem_o + 32 * k, o);
            ptx::tmem_ld_wait(o);
            if (!real) continue;
            if (it.full) {
              uint4* dst = reinterpret_cast<uint4*>(a.out + orow * kD + 32 * k);
#pragma unroll
              for (int c = 0; c < 4; ++c)
                dst[c] = make_uint4(pack_bf16(__uint_as_float(o[8 * c]) * inv, __uint_as_float(o[8 * c + 1]) * inv),
                                    pack_bf16(__uint_as_float(o[8 * c + 2]) * inv, __uint_as_float(o[8 * c + 3]) * inv),
                                    pack_bf16(__uint_as_float(o[8 * c + 4]) * inv, __uint_as_float(o[8 * c + 5]) * inv),
                                    pack_bf16(__uint_as_float(o[8 * c + 6]) * inv, __uint_as_float(o[8 * c + 7]) * inv));
            } else {
              // 16-byte chunk c of this 32-column group goes to position c ^ (row & 7), so that
              // the merging CTA reads its copy of the rows without bank conflicts
              float4* dst = reinterpret_cast<float4*>(a.ws_o + (slot * kBlockRows + row) * kD + 32 * k);
#pragma unroll
              for (int c = 0; c < 8; ++c)
                dst[c ^ (row & 7)] = make_float4(__uint_as_float(o[4 * c]), __uint_as_float(o[4 * c + 1]),
                                                 __uint_as_float(o[4 * c + 2]), __uint_as_float(o[4 * c + 3]));
            }
          }
          if (real) {
            if (it.full) {
              if (a.lse) a.lse[orow] = (m_used + __log2f(l)) * 0.69314718055994530942f;
            } else {
              a.ws_ml[slot * kBlockRows + row] = make_float2(m_used, l);
            }
          }
        }
        ptx::tc_fence_before();
      } while (false);
      // One answer for the segment: a warp that gave up left the tile loop or the epilogue
      // early and meets the others here.
      ok = !ptx::bar_or(1, 128, !ok);
      if (!ok) {
        mark_unfinished(a, it, real, orow, slot, row);  // this segment stopped part-way
        if (!it.full && it.i0 > 0) publish(slot);
      } else if (!it.full && it.i0 > 0) {
        publish(slot);
      } else if (!it.full) {
        // ---- merge of a split pair, by its first piece (the last segment of this range): the
        // later pieces are the first segment of every non-empty unit up to the one holding
        // the pair's end, in the CTA of this row block (partial slot 0)
        const int64_t T = st.T;
        const int C = a.ctas;
        const int c_last = (int)((it.pend * (int64_t)C + T - 1) / T) - 1;
        bool got = true;
        if (tid == 0) {
          const uint64_t t_start = ptx::globaltimer_ns();
          for (int vc = vcta + 1; vc <= c_last && got; ++vc) {
            if (cta_begin(T, C, vc) == cta_begin(T, C, vc + 1)) continue;
            const int64_t ps = (int64_t)part_slot(vc * a.cl + crank, 0);
            if (!chk(ps, 1, nslots, a.dev_err)) continue;
            while (ld_acquire_u64(a.ws_flag + ps) != token) {
              if (*(volatile int*)&sh->abort) {
                got = false;
                break;
              }
              if (ptx::globaltimer_ns() - t_start > wait_ns) {
                raise_abort(sh, a.dev_err);
                got = false;
                break;
              }
              __nanosleep(64);
            }
          }
          if (got) {  // each slot is published once per launch: consumed, cleared
            for (int vc = vcta + 1; vc <= c_last; ++vc) {
              if (cta_begin(T, C, vc) == cta_begin(T, C, vc + 1)) continue;
              const int64_t ps = (int64_t)part_slot(vc * a.cl + crank, 0);
              if (chk(ps, 1, nslots, a.dev_err)) a.ws_flag[ps] = 0;
            }
          }
        }
        got = !ptx::bar_or(1, 128, !got);
        // The pieces' partials come into shared memory (the ring, idle once this last
        // segment's P V completed), two at a time, one bulk copy each for O (64 KB) and for
        // (max, sum) (1 KB); each is folded into this piece's O in TMEM (online rescale).
        float mt = m_used, L = l;
        int vc = vcta + 1, batch = 0;
        while (got) {
          int ps_b[kMergeBatch], nb = 0;
          for (; vc <= c_last && nb < kMergeBatch; ++vc) {
            if (cta_begin(T, C, vc) == cta_begin(T, C, vc + 1)) continue;
            ps_b[nb++] = (int)part_slot(vc * a.cl + crank, 0);
          }
          if (nb == 0) break;
          if (tid == 0) {
            ptx::fence_proxy_async_smem();  // earlier reads of the staging area are done (barrier)
            ptx::mbar_arrive_expect_tx(bar(kMerge), (uint32_t)nb * (kMergeO + kMergeML));
            for (int q = 0; q < nb; ++q) {
              const int64_t ps = ps_b[q];
              if (!chk(ps, 1, nslots, a.dev_err)) continue;  // (the wait then gives up)
              ptx::bulk_load_g2s(sbase + kOffStages + q * kMergeO, a.ws_o + ps * kBlockRows * kD, kMergeO, bar(kMerge));
              ptx::bulk_load_g2s(sbase + kOffStages + kMergeBatch * kMergeO + q * kMergeML,
                                 a.ws_ml + ps * kBlockRows, kMergeML, bar(kMerge));
            }
          }
          got = !ptx::bar_or(1, 128, !wait_bar(sh, bar(kMerge), batch & 1, a.dev_err, wait_ns));
          if (!got) break;
          if (warp_active) {
            ptx::tc_fence_after();
            for (int q = 0; q < nb; ++q) {
              const float2 ml = reinterpret_cast<const float2*>(smem + kOffStages + kMergeBatch * kMergeO +
                                                                 q * kMergeML)[row];
              const float m_new = fmaxf(mt, ml.x);
              const float a_self = exp2f(mt - m_new), a_p = exp2f(ml.x - m_new);
              L = L * a_self + ml.y * a_p;
              mt = m_new;
              const float4* srow = reinterpret_cast<const float4*>(smem + kOffStages + q * kMergeO) + row * (kD / 4);
#pragma unroll 1
              for (int k = 0; k < 4; ++k) {
                uint32_t o[32];
                ptx::tmem_ld32(tmem_o + 32 * k, o);
                ptx::tmem_ld_wait(o);
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                  const float4 v = srow[8 * k + (c ^ (row & 7))];
                  o[4 * c] = __float_as_uint(fmaf(a_p, v.x, __uint_as_float(o[4 * c]) * a_self));
                  o[4 * c + 1] = __float_as_uint(fmaf(a_p, v.y, __uint_as_float(o[4 * c + 1]) * a_self));
                  o[4 * c + 2] = __float_as_uint(fmaf(a_p, v.z, __uint_as_float(o[4 * c + 2]) * a_self));
                  o[4 * c + 3] = __float_as_uint(fmaf(a_p, v.w, __uint_as_float(o[4 * c + 3]) * a_self));
                }
                ptx::tmem_st32(tmem_o + 32 * k, o);
              }
              ptx::tmem_st_wait();  // the next piece (or the final read) loads these columns
            }
            ptx::tc_fence_before();
          }
          ++batch;
          ptx::named_bar_sync(1, 128);  // the staging area is read before it is refilled
        }
        if (!got) {
          mark_unfinished(a, it, real, orow, slot, row);
        } else if (warp_active) {
          ptx::tc_fence_after();
          const bool rok = real && chk((int64_t)orow * kD, kD, (int64_t)a.batch * twoB * a.Hq * kD, a.dev_err);
          const float inv = 1.f / L;
#pragma unroll 1
          for (int k = 0; k < 4; ++k) {
            uint32_t o[32];
            ptx::tmem_ld32(tmem_o + 32 * k, o);
            ptx::tmem_ld_wait(o);
            if (!rok) continue;
            uint4* dst = reinterpret_cast<uint4*>(a.out + orow * kD + 32 * k);
#pragma unroll
            for (int c = 0; c < 4; ++c)
              dst[c] = make_uint4(pack_bf16(__uint_as_float(o[8 * c]) * inv, __uint_as_float(o[8 * c + 1]) * inv),
                                  pack_bf16(__uint_as_float(o[8 * c + 2]) * inv, __uint_as_float(o[8 * c + 3]) * inv),
                                  pack_bf16(__uint_as_float(o[8 * c + 4]) * inv, __uint_as_float(o[8 * c + 5]) * inv),
                                  pack_bf16(__uint_as_float(o[8 * c + 6]) * inv, __uint_as_float(o[8 * c + 7]) * inv));
          }
          if (rok && a.lse) a.lse[orow] = (mt + log2f(L)) * 0.69314718055994530942f;
          ptx::tc_fence_before();
        }
      }
      it.advance(a);
    }
    if (aborted) {  // the segment reached and every later one of the range are unfinished
      do {
        const size_t orow = ((size_t)it.b * twoB + s_slot) * a.Hq + (size_t)it.h * a.G + g;
        const size_t pslot = part_slot(blockIdx.x, it.first ? 0 : 1);
        mark_unfinished(a, it, real, orow, pslot, row);
        if (!it.full && it.i0 > 0 && !it.invalid) publish(pslot);  // (a NaN partial)
        it.advance(a);
      } while (it.next(a));
    }
    if (!loads_signalled) ptx::mbar_arrive(bar(kLoads));  // no prologue ran: release the producer
  }

  ptx::tc_fence_before();
  if constexpr (kPair) {
    // the even CTA's MMAs read this CTA's shared memory and TMEM until its drain: neither CTA
    // frees TMEM or exits before both are here
    ptx::cluster_sync();
    ptx::tc_fence_after();
    if (warp == kMmaWarp) ptx::tmem_dealloc_pair(tmem, kTmemCols);
  } else {
    __syncthreads();
    ptx::tc_fence_after();
    if (warp == kMmaWarp) ptx::tmem_dealloc(tmem, kTmemCols);
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
                             int Hkv, int box_keys) {
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
    box[2] = (cuuint32_t)box_keys;
  } else {  // [Hkv][tokens][D]: dims (D, tokens, Hkv)
    dims[0] = kD;
    dims[1] = (cuuint64_t)(tokens > 0 ? tokens : 1);
    dims[2] = (cuuint64_t)Hkv;
    strides[0] = (cuuint64_t)kD * 2;
    strides[1] = (cuuint64_t)(tokens > 0 ? tokens : 1) * kD * 2;
    box[0] = 64;
    box[1] = (cuuint32_t)box_keys;
    box[2] = 1;
  }
  const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims,
                         strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// True when `ptr` is device memory of the current device `dev` (or managed memory): the
// tensor maps read the cache through this GPU's own memory system only.
static bool on_device(const void* ptr, int dev) {
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, ptr) != cudaSuccess) {
    cudaGetLastError();  // clear the sticky-free error of an unknown pointer
    return false;
  }
  if (at.type == cudaMemoryTypeManaged) return true;
  return at.type == cudaMemoryTypeDevice && at.device == dev;
}

static int rows_per_pair(const simsd_attn_params* p) { return 2 * p->B * (p->Hq / p->Hkv); }
// CTAs per schedule unit: two for pairs of more than 128 rows (one per 128-row block).
static int ctas_per_unit(const simsd_attn_params* p) { return rows_per_pair(p) > 128 ? 2 : 1; }

// The dynamic shared memory attribute of both kernels is set once per device; for the CTA-pair
// kernel the number of its 2-CTA clusters that fit on the device at once is queried then too.
static std::mutex g_attr_mutex;
static bool g_attr_done[64];
static int g_pair_clusters[64];

static simsd_status set_smem_attr(int dev) {
  std::lock_guard<std::mutex> lock(g_attr_mutex);
  if (dev >= 0 && dev < 64 && g_attr_done[dev]) return SIMSD_OK;
  cudaError_t e = cudaFuncSetAttribute(attn_tc128_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)r128::kSmemBytes);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(attn_tc128_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)r128::kSmemBytes);
  if (e != cudaSuccess) {
    record_cuda_error("cudaFuncSetAttribute", e);
    return SIMSD_ERR_CUDA;
  }
  int sms = device_sm_count();
  if (sms <= 0) sms = 148;
  int n = 0;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = 2;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3((unsigned)(sms & ~1));
  cfg.blockDim = dim3((unsigned)r128::kThreads);
  cfg.dynamicSmemBytes = r128::kSmemBytes;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  if (cudaOccupancyMaxActiveClusters(&n, attn_tc128_kernel<true>, &cfg) != cudaSuccess || n <= 0) {
    cudaGetLastError();
    n = sms / 2;
  }
  if (dev >= 0 && dev < 64) {
    g_pair_clusters[dev] = n;
    g_attr_done[dev] = true;
  }
  return SIMSD_OK;
}

static int pair_clusters_resident() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (set_smem_attr(dev) != SIMSD_OK) return 0;
  std::lock_guard<std::mutex> lock(g_attr_mutex);
  return g_pair_clusters[dev];
}

// Persistent grid: one CTA per SM; when every (request, kv head) pair fits on the SMs and
// prompts are short, one unit per pair instead (no pair is split, nothing to merge).
// (With `cl` = 2 CTAs per unit: at most as many units as 2-CTA clusters fit at once.)
static int grid_units(const simsd_attn_params* p, int cl) {
  int sms = device_sm_count();
  if (sms <= 0) sms = 148;
  sms /= cl;
  if (cl == 2) {
    const int nc = pair_clusters_resident();
    if (nc > 0 && nc < sms) sms = nc;
  }
  const int64_t pairs = (int64_t)p->batch * p->Hkv;
  const int64_t avg_tiles = 1 + (p->batch > 0 ? (p->cache_tokens / p->batch + kTileKeys - 1) / kTileKeys : 0);
  if (pairs > 0 && pairs <= sms && avg_tiles <= 64) return (int)pairs;
  return sms;
}

struct WsLayout {
  size_t o, ml, flag, bytes;
};
static WsLayout ws_layout(int ctas) {
  WsLayout w;
  w.o = 0;
  w.ml = align_up(w.o + (size_t)2 * ctas * kBlockRows * kD * sizeof(float), 256);
  w.flag = align_up(w.ml + (size_t)2 * ctas * kBlockRows * sizeof(float2), 256);
  w.bytes = align_up(w.flag + (size_t)2 * ctas * sizeof(uint64_t), 256);
  return w;
}


static simsd_status launch(const simsd_attn_params* p, void* ws, size_t ws_bytes, cudaStream_t stream) {
  int dev = 0;
  const cudaError_t de = cudaGetDevice(&dev);
  if (de != cudaSuccess) {
    record_cuda_error("cudaGetDevice", de);
    return SIMSD_ERR_CUDA;
  }
  if (p->cache_tokens > 0 && (!on_device(p->k_cache, dev) || !on_device(p->v_cache, dev)))
    return SIMSD_ERR_INVALID_ARG;
  TcArgs a;
  a.batch = p->batch;
  a.B = p->B;
  a.Hq = p->Hq;
  a.Hkv = p->Hkv;
  a.G = p->Hq / p->Hkv;
  a.R = rows_per_pair(p);
  a.cl = ctas_per_unit(p);
  a.seg_cost = seg_cost_tiles(2 * p->B);
  a.ctas = grid_units(p, a.cl);
  a.layout = (int)p->cache_layout;
  a.cache_tokens = p->cache_tokens;
  a.wait_ns = p->wait_limit_ns > 0 ? p->wait_limit_ns : kDefaultWaitNs;
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
  const WsLayout wl = ws_layout(a.ctas * a.cl);
  if (!ws || ws_bytes < wl.bytes || (((uintptr_t)ws) & 255)) return SIMSD_ERR_WORKSPACE;
  a.ws_o = (float*)((char*)ws + wl.o);
  a.ws_ml = (float2*)((char*)ws + wl.ml);
  a.ws_flag = (uint64_t*)((char*)ws + wl.flag);
  make_rope_table(&a.rope, (double)p->rope_theta, kD);

  CUtensorMap tmk, tmv;
  const void* kbase = p->cache_tokens > 0 ? p->k_cache : p->k_resp;  // any valid address
  const void* vbase = p->cache_tokens > 0 ? p->v_cache : p->v_resp;
  // CTA pairs: each CTA's K box is 64 of a tile's keys (V: all 128 keys, 64 dims)
  if (!encode_cache_map(&tmk, kbase, a.layout, p->cache_tokens, p->Hkv, a.cl == 2 ? 64 : kKeys) ||
      !encode_cache_map(&tmv, vbase, a.layout, p->cache_tokens, p->Hkv, kKeys)) {
    record_cuda_error("cuTensorMapEncodeTiled", cudaErrorInvalidValue);
    return SIMSD_ERR_CUDA;
  }
  const simsd_status ast = set_smem_attr(dev);
  if (ast != SIMSD_OK) return ast;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute cat[2];
  // a programmatic dependent of the stream's previous kernel (the layout kernel), and with
  // CTA pairs a 2-CTA cluster
  cat[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  cat[0].val.programmaticStreamSerializationAllowed = 1;
  cat[1].id = cudaLaunchAttributeClusterDimension;
  cat[1].val.clusterDim.x = 2;
  cat[1].val.clusterDim.y = 1;
  cat[1].val.clusterDim.z = 1;
  cfg.gridDim = dim3((unsigned)(a.ctas * a.cl));
  cfg.blockDim = dim3((unsigned)r128::kThreads);
  cfg.dynamicSmemBytes = r128::kSmemBytes;
  cfg.stream = stream;
  cfg.attrs = cat;
  cfg.numAttrs = a.cl == 2 ? 2 : 1;
  const void* kfn = a.cl == 2 ? (const void*)attn_tc128_kernel<true> : (const void*)attn_tc128_kernel<false>;
  cudaError_t le = a.cl == 2 ? cudaLaunchKernelEx(&cfg, attn_tc128_kernel<true>, tmk, tmv, a)
                             : cudaLaunchKernelEx(&cfg, attn_tc128_kernel<false>, tmk, tmv, a);
  if (le == cudaSuccess) le = cudaGetLastError();
  if (le != cudaSuccess) {
    cudaFuncAttributes fa;
    char what[200] = "attention kernel launch";
    if (cudaFuncGetAttributes(&fa, kfn) == cudaSuccess)
      snprintf(what, sizeof(what),
               "attention kernel launch (threads %d, regs %d, max threads %d, dyn smem %u, "
               "max dyn smem %d, static smem %zu, local %zu)",
               r128::kThreads, fa.numRegs, fa.maxThreadsPerBlock, r128::kSmemBytes,
               fa.maxDynamicSharedSizeBytes, fa.sharedSizeBytes, fa.localSizeBytes);
    record_cuda_error(what, le);
    return SIMSD_ERR_CUDA;
  }
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
  const int cl = tc::ctas_per_unit(p);
  return tc::ws_layout(tc::grid_units(p, cl) * cl).bytes;
}

simsd_status launch_attn_tc(const simsd_attn_params* p, void* ws, size_t ws_bytes,
                            cudaStream_t stream) {
  const uintptr_t mask = 15;
  if ((((uintptr_t)p->q) | ((uintptr_t)p->k_resp) | ((uintptr_t)p->v_resp) |
       ((uintptr_t)p->out)) & mask)
    return SIMSD_ERR_UNSUPPORTED;
  if (p->cache_tokens > 0 && ((((uintptr_t)p->k_cache) | ((uintptr_t)p->v_cache)) & mask))
    return SIMSD_ERR_UNSUPPORTED;
  // up to 128 rows per pair: one CTA per schedule unit; 129..256 rows: a CTA pair
  return tc::launch(p, ws, ws_bytes, stream);
}

}  // namespace simsd
