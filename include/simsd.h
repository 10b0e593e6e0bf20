/*
 * simsd.h -- C interface of the GB300 (sm_103a) SimSD single-forward verification step.
 *
 * The step has three calls, run in this order on one CUDA stream:
 *
 *   simsd_build_layout      paired layout [prompt | D_1..D_B | D~_1..D~_B]: copied RoPE
 *                           position ids and packed step labels (no mask is stored).
 *   simsd_verify_attention  one attention layer of the verify forward over that layout
 *                           under the temporal-causal mask A_ij, evaluated on the fly.
 *   simsd_accept            min(1, p/q) prefix acceptance along the step order, then
 *                           residual resampling at the first rejected slot.
 *
 * and, before the verify forward when a caller routes requests, simsd_expected_prefix
 * (the expected accepted-prefix length K^ of every request from its draft logits).
 *
 * Conventions shared by every call
 *   - All array pointers are DEVICE pointers owned by the caller; the library keeps no
 *     reference after the call returns. Every call is asynchronous on `stream` (a
 *     cudaStream_t; NULL = legacy default stream), never synchronises and never
 *     allocates memory. Scratch memory is a caller-provided `workspace`, sized by the
 *     matching *_workspace() query.
 *   - Errors the host can see (null pointers, unsupported sizes, a workspace that is too
 *     small) are returned synchronously as a simsd_status and nothing is launched.
 *   - Errors that depend on device data are OR-ed into the caller's 32-bit device error
 *     word `dev_err` (SIMSD_DEVERR_* bits) and the affected request gets the documented
 *     sentinel outputs. Kernels never trap, assert or print.
 *   - Shapes: b = batch (requests), B = block size (1..32), Hq / Hkv query / key-value
 *     heads (Hq % Hkv == 0, G = Hq / Hkv), D = head dim (64 or 128), V = vocabulary.
 *     Response slot index s in [0, 2B): s < B is the data slot D_{s+1}, s >= B the mask
 *     slot D~_{s-B+1}.
 *
 * Passages cited (pages on SimSD / S2D2 / SPOT):
 *   [SimSD-1] SimSD notes (papernotes.org), "关键设计" item 1: paired data/mask layout.
 *   [SimSD-2] same page, item 2: step labels tau in 1..B (prompt tau = 0) and the
 *             four-case mask equation A_ij.
 *   [SimSD-3] same page, item 3: the mask slot D~_k reuses the RoPE position id of D_k.
 *   [SimSD-4] same page, item 4: alpha_r = min(1, p_theta / p_phi) in the draft's time
 *             order, longest accepted prefix, in-place resampling of the rejected slot.
 *   [SimSD-P] gist.science SimSD summary, sections 1-4 (same method; tau is a permutation).
 *   [S2D2-5]  S2D2 page, "方法步骤详情" step (5): residual distribution (P_ver - P)^+.
 *   [SPOT-G]  SPOT page, "Gumbel-Max 技巧与随机耦合": argmax(log p + G) samples p.
 *   [S2D2-4]  S2D2 page, "方法步骤详情" step (4): routing by the expected accepted-prefix
 *             length K^ = sum_k prod_{i<=k} alpha_i (margin- or entropy-based alpha_i).
 *   [SPOT-C]  SPOT page, core-innovation and Algorithm 2 paragraphs: coupled-noise
 *             verification, a Gumbel table G_{a,v} indexed by absolute output position
 *             shared by drafter and target; the target's transition Phi_G is then
 *             deterministic and an edge is accepted iff the states are equal.
 */
#ifndef SIMSD_H
#define SIMSD_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* simsd_stream_t; /* identical to cudaStream_t */

typedef enum {
  SIMSD_OK = 0,
  SIMSD_ERR_INVALID_ARG = 1, /* null pointer, bad size or combination of sizes        */
  SIMSD_ERR_UNSUPPORTED = 2, /* valid request this build does not implement           */
  SIMSD_ERR_WORKSPACE = 3,   /* workspace pointer null / misaligned / too small        */
  SIMSD_ERR_CUDA = 4,        /* a CUDA runtime or driver call failed (launch, encode)  */
  SIMSD_ERR_TIMEOUT = 5      /* reserved: a bounded device-side wait ran out           */
} simsd_status;

/* Bits of the device error word. */
#define SIMSD_DEVERR_TAU 1u        /* tau of a request: open labels not 1..R, or > B    */
#define SIMSD_DEVERR_PROMPT_LEN 2u /* prompt length < 0                                 */
#define SIMSD_DEVERR_TOKEN 4u      /* a verified draft token id is outside [0, V)       */
#define SIMSD_DEVERR_TIMEOUT 8u    /* a bounded wait inside a kernel gave up            */
#define SIMSD_DEVERR_BOUNDS 16u    /* checked builds only (compiled with SIMSD_CHECKED):
                                      a kernel computed a global index outside the array
                                      it addresses; that access was skipped             */

/* Label byte of a response slot: (segment << 7) | tau, segment 0 = D, 1 = D~.
 * 0xFF marks every slot of a request the layout call rejected. */
#define SIMSD_LABEL_INVALID 0xFFu

typedef enum { SIMSD_DTYPE_FP32 = 0, SIMSD_DTYPE_BF16 = 1 } simsd_dtype;

/* Estimators of the per-step acceptance alpha_i of simsd_expected_prefix. */
typedef enum { SIMSD_KHAT_MARGIN = 0, SIMSD_KHAT_ENTROPY = 1 } simsd_khat_mode;

/* Cache layouts of the packed prompt K/V (keys stored already rotated at positions
 * 0..P-1 of their request):
 *   NHD: [cache_tokens, Hkv, D]      HND: [Hkv, cache_tokens, D]   (both contiguous) */
typedef enum { SIMSD_CACHE_NHD = 0, SIMSD_CACHE_HND = 1 } simsd_cache_layout;

/* Human-readable name of a status code (static storage, never NULL). */
const char* simsd_status_str(simsd_status s);

/* Library interface version (major * 10000 + minor * 100 + patch).
 *   0.1.0  layout, verify attention, acceptance (+ workspace queries, allocation-free entry)
 *   0.2.0  adds simsd_accept_coupled, simsd_accept_ex / simsd_accept_coupled_ex (bf16
 *          logits), simsd_expected_prefix (+ workspace), simsd_build_layout_ex (flags);
 *          every 0.1.0 call is unchanged
 *   0.3.0  simsd_attn_params gains wait_limit_ns (its last field; zero keeps the 0.2.0
 *          behaviour, so callers that zero-initialise the struct need no other change) */
int simsd_version(void);

/* Text of the CUDA runtime/driver error behind the most recent SIMSD_ERR_CUDA returned
 * on the calling host thread ("" if none). Static/thread-local storage, never NULL. */
const char* simsd_last_cuda_error(void);

/* ---------------------------------------------------------------------------------
 * simsd_build_layout  [SimSD-1], [SimSD-2], [SimSD-3], [SimSD-P] sections 1-3.
 *
 * Lays out the response part of [prompt | D_1..D_B | D~_1..D~_B] for each request:
 *   pos_ids[r][k]     = P_r + k   for the data slot D_{k+1}         (k = 0..B-1)
 *   pos_ids[r][B + k] = P_r + k   for the mask slot D~_{k+1} (copied id)
 *   labels[r][k]      = tau[r][k]            (segment 0, data)
 *   labels[r][B + k]  = 0x80 | tau[r][k]     (segment 1, mask)
 * Prompt tokens have tau = 0 and positions 0..P_r-1 implicitly; no mask is stored.
 *
 *   tau        int32 [batch, B]   step label of each slot: a permutation of 1..B in a
 *                                 block's first round; in a later round 0 marks a slot
 *                                 committed earlier (seen like the prompt, [SimSD-2]) and
 *                                 the R open slots carry a permutation of 1..R ([SimSD-4]:
 *                                 the remaining positions)
 *   prompt_len int32 [batch]      prompt length P_r >= 0
 *   pos_ids    int32 [batch, 2B]  output
 *   labels     uint8 [batch, 2B]  output
 *   dev_err    uint32 [1]         error word, bits OR-ed in (never cleared here)
 * Data errors: a request whose tau breaks that rule (SIMSD_DEVERR_TAU) or
 * whose P_r < 0 (SIMSD_DEVERR_PROMPT_LEN) gets pos_ids = -1 and labels = 0xFF.
 * Returns SIMSD_ERR_INVALID_ARG for null pointers, batch < 0, B < 1 or B > 32.
 * --------------------------------------------------------------------------------- */
simsd_status simsd_build_layout(const int32_t* tau, const int32_t* prompt_len, int batch,
                                int B, int32_t* pos_ids, uint8_t* labels, uint32_t* dev_err,
                                simsd_stream_t stream);

/* simsd_build_layout_ex -- simsd_build_layout with layout flags (0: exactly
 * simsd_build_layout).
 *   SIMSD_LAYOUT_PHYSICAL_POSITIONS  pos_ids[r][B + k] = P_r + B + k: the mask slots take
 *     their own index in the sequence instead of D_k's id. This is the "Without Aligned
 *     RoPE" ablation of the SimSD notes' table ([SimSD-3]), kept as a negative control:
 *     the prediction rows then no longer equal the explicit denoising states.
 * Unknown flag bits return SIMSD_ERR_INVALID_ARG. */
#define SIMSD_LAYOUT_PHYSICAL_POSITIONS 1u

simsd_status simsd_build_layout_ex(const int32_t* tau, const int32_t* prompt_len, int batch,
                                   int B, uint32_t flags, int32_t* pos_ids, uint8_t* labels,
                                   uint32_t* dev_err, simsd_stream_t stream);

/* ---------------------------------------------------------------------------------
 * simsd_verify_attention  [SimSD-2], [SimSD-3], [SimSD-P] sections 2-4.
 *
 * One softmax-attention layer of the single verify forward. Response row s of request r
 * and query head h (kv head h / G) attends to
 *   - every prompt key of the request (tau = 0 is earlier than every step), and
 *   - the response keys allowed by A_ij: with t = tau(s) + [s is a data slot], a data
 *     key D_j is visible iff tau(j) < t and a mask key D~_j iff tau(j) >= t
 *     (equivalent to the four cases of A_ij; every row sees exactly B response keys).
 * Response queries and keys are rotated here (RoPE, pairs (d, d + D/2), angle
 * pos * theta^(-2d/D)) with the copied ids from simsd_build_layout; V is not rotated.
 * Output row = softmax(scale * q k^T) v over the visible keys; lse = natural-log
 * sum-exp of the scaled scores (optional).
 *
 * BF16 path: tcgen05 tensor-core kernel (fp32 accumulation), split over the prompt keys
 * and merged; FP32 path: CUDA-core kernel in fp32 throughout.
 * Zero-initialise the struct (e.g. `simsd_attn_params p = {0};`) and set every field
 * below; fields added by later versions then keep their default.
 * --------------------------------------------------------------------------------- */
typedef struct {
  simsd_dtype dtype;        /* element type of q, k_resp, v_resp, k_cache, v_cache, out */
  int batch, B, Hq, Hkv, D;
  const void* q;            /* [batch, 2B, Hq, D]   pre-RoPE                            */
  const void* k_resp;       /* [batch, 2B, Hkv, D]  pre-RoPE                            */
  const void* v_resp;       /* [batch, 2B, Hkv, D]                                      */
  const void* k_cache;      /* packed prompt keys (already rotated), see cache_layout   */
  const void* v_cache;      /* packed prompt values, same layout                        */
  simsd_cache_layout cache_layout;
  int64_t cache_tokens;     /* number of token rows in the packed cache                 */
  const int64_t* cache_start; /* int64 [batch]: first cache row of each request         */
  const int32_t* prompt_len;  /* int32 [batch]: P_r; rows cache_start[r] .. + P_r - 1  */
  const int32_t* pos_ids;   /* int32 [batch, 2B] from simsd_build_layout                */
  const uint8_t* labels;    /* uint8 [batch, 2B] from simsd_build_layout                */
  float rope_theta;         /* RoPE base theta (> 0)                                    */
  float softmax_scale;      /* <= 0 selects 1/sqrt(D)                                   */
  void* out;                /* [batch, 2B, Hq, D] output, dtype as the inputs           */
  float* lse;               /* fp32 [batch, 2B, Hq] output, or NULL                     */
  uint32_t* dev_err;        /* device error word                                        */
  uint64_t wait_limit_ns;   /* bound of every device-side wait of the BF16 kernel, in
                               ns; 0 selects 2 s (see below)                            */
} simsd_attn_params;
/* Data errors: a request with labels 0xFF or P_r < 0 (bit SIMSD_DEVERR_PROMPT_LEN for
 * the latter) gets zero output rows and lse = -inf.
 * Bounded waits: the BF16 kernel's warps wait on one another (copies, MMAs, softmax). A
 * wait that makes no progress for wait_limit_ns (0: 2 s, far beyond any legitimate wait)
 * sets SIMSD_DEVERR_TIMEOUT; the kernel then stops early and returns (it never hangs and
 * never traps): every output row it did not finish is NaN (lse NaN), the rows it finished
 * are valid. The context stays usable and the next call runs normally.
 * Host errors: SIMSD_ERR_INVALID_ARG (null pointer, Hq % Hkv != 0, B outside 1..32,
 * negative sizes, a BF16 prompt cache that is not device memory of the current device),
 * SIMSD_ERR_UNSUPPORTED (D not 64/128; BF16 needs D = 128 and 2B*G <= 256 on this
 * build; cache rows or pointers not 16-byte aligned), SIMSD_ERR_WORKSPACE. */

/* Bytes of workspace simsd_verify_attention needs for these sizes (on the current
 * device). The workspace must be 256-byte aligned; its contents need no initialisation
 * and are scratch after the call. */
size_t simsd_verify_attention_workspace(const simsd_attn_params* p);

simsd_status simsd_verify_attention(const simsd_attn_params* p, void* workspace,
                                    size_t workspace_bytes, simsd_stream_t stream);

/* ---------------------------------------------------------------------------------
 * simsd_accept  [SimSD-4], [SimSD-P] section 4, [S2D2-5], [SPOT-G].
 *
 * For each request r, with o_t = the slot whose step label is t (from labels' data
 * half) and x_t = draft_tokens[r][o_t], for t = 1..gamma_r, gamma_r = min(gamma, R_r)
 * (R_r = the request's open slots, B in a block's first round):
 *   p = softmax(target_logits[r][o_t] / T), q = softmax(draft_logits[r][o_t] / T)
 *   accept step t iff p[x_t] >= q[x_t] or u_t * q[x_t] < p[x_t]; stop at the first
 *   rejection. accepted_len = a (number of leading accepted steps).
 * If a < gamma_r, slot o_{a+1} is resampled from the normalised residual max(0, p - q)
 * by the exponential race y = argmax_v r_v / E_v, E_v = -ln(u_v) (ties -> smallest v;
 * if the residual is zero everywhere the race runs on p). No extra token is drawn when
 * all gamma steps are accepted.
 * Uniforms: Philox4x32-10 (Salmon et al., SC'11), key = (seed lo, seed hi);
 *   step t (0-based)  counter (r, offset lo, offset hi, t / 4), word t % 4;
 *   token v           counter (r, offset lo, offset hi, 0x80000000 | v / 4), word v % 4;
 *   u = (2 * (word >> 9) + 1) * 2^-24.
 *
 *   target_logits, draft_logits  fp32 [batch, B, V], row k = block slot k
 *   draft_tokens                 int32 [batch, B], token of data slot k
 *   labels                       uint8 [batch, 2B] from simsd_build_layout
 *   accepted_len                 int32 [batch]     a, or -1 for a rejected request
 *   n_commit                     int32 [batch]     a + (a < gamma_r), or 0
 *   out_tokens                   int32 [batch, B]  committed tokens in step order, -1 after
 *   out_pos                      int32 [batch, B]  their slot indices, -1 after
 * temperature = 0 is greedy verification [SPOT-G] (the SPOT page's Algorithm 2, which
 * verifies at T = 0 against the target's own deterministic commit): step t is accepted iff
 * x_t is the first index of the largest target logit at o_t, and at the first mismatch
 * that index is committed; draft logits, seed and offset are unused.
 * Requires 1 <= gamma <= B <= 32, V >= 1, temperature >= 0. Data errors: labels not a permutation (SIMSD_DEVERR_TAU) or a
 * verified token outside [0, V) (SIMSD_DEVERR_TOKEN) -> accepted_len = -1, n_commit = 0,
 * out_tokens = out_pos = -1 for that request.
 * --------------------------------------------------------------------------------- */
/* Bytes of workspace simsd_accept needs for these sizes on the current device (the work
 * split follows the device's resident warps). The workspace must be 256-byte aligned; its
 * contents need no initialisation and are scratch after the call. */
size_t simsd_accept_workspace(int batch, int B, int gamma, int V);

simsd_status simsd_accept(const float* target_logits, const float* draft_logits,
                          const int32_t* draft_tokens, const uint8_t* labels, int batch,
                          int B, int gamma, int V, float temperature, uint64_t seed,
                          uint64_t offset, int32_t* accepted_len, int32_t* out_tokens,
                          int32_t* out_pos, int32_t* n_commit, void* workspace,
                          size_t workspace_bytes, uint32_t* dev_err, simsd_stream_t stream);

/* ---------------------------------------------------------------------------------
 * simsd_accept_coupled  [SPOT-C], [SPOT-G]; steps and later rounds as simsd_accept.
 *
 * Coupled-noise verification: for t = 1..gamma_r, with a_t = pos_ids[r][o_t] (the absolute
 * output position of slot o_t, from simsd_build_layout), the target's own transition is
 *   y_t = argmax_v (target_logits[r][o_t][v] / T + G_{a_t, v}),  G = -ln(-ln u)
 * (ties -> smallest v), a sample of softmax(logits / T) by the Gumbel-max identity. Step t
 * is accepted iff x_t = y_t; at the first mismatch y_t is committed (same outputs as
 * simsd_accept). A drafter that proposes argmax_v (draft_logits / T + G) with the same table
 * is accepted with probability >= (1 - TV) / (1 + TV). T = 0 is the greedy verification of
 * simsd_accept. No draft logits are read.
 * Noise uniforms: Philox4x32-10, key = (seed lo, seed hi), counter (r, a, offset lo,
 * 0x40000000 | v / 4), word v % 4, u = (2 * (word >> 9) + 1) * 2^-24.
 *   pos_ids  int32 [batch, 2B] from simsd_build_layout; other arguments as simsd_accept.
 * Workspace: simsd_accept_workspace(batch, B, gamma, V) bytes, 256-byte aligned.
 * --------------------------------------------------------------------------------- */
simsd_status simsd_accept_coupled(const float* target_logits, const int32_t* draft_tokens,
                                  const uint8_t* labels, const int32_t* pos_ids, int batch, int B,
                                  int gamma, int V, float temperature, uint64_t seed,
                                  uint64_t offset, int32_t* accepted_len, int32_t* out_tokens,
                                  int32_t* out_pos, int32_t* n_commit, void* workspace,
                                  size_t workspace_bytes, uint32_t* dev_err, simsd_stream_t stream);

/* ---------------------------------------------------------------------------------
 * simsd_accept_ex, simsd_accept_coupled_ex -- simsd_accept and simsd_accept_coupled with
 * the element type of the logits as an argument. (Library addition: a model head that
 * emits bf16 logits is verified without a widening copy.)
 *   logit_dtype  SIMSD_DTYPE_FP32: the logit arrays are float, exactly simsd_accept /
 *                simsd_accept_coupled.
 *                SIMSD_DTYPE_BF16: the logit arrays are bf16 [batch, B, V]; every entry is
 *                widened exactly to fp32 on load and the operation proceeds on those fp32
 *                values: the outputs equal those of the fp32 call on the widened arrays.
 *                Other values return SIMSD_ERR_INVALID_ARG.
 *   All other arguments, the workspace size (simsd_accept_workspace, the same for both
 *   types), outputs, error bits and sentinels: as the fp32 calls.
 * --------------------------------------------------------------------------------- */
simsd_status simsd_accept_ex(const void* target_logits, const void* draft_logits,
                             simsd_dtype logit_dtype, const int32_t* draft_tokens,
                             const uint8_t* labels, int batch, int B, int gamma, int V,
                             float temperature, uint64_t seed, uint64_t offset,
                             int32_t* accepted_len, int32_t* out_tokens, int32_t* out_pos,
                             int32_t* n_commit, void* workspace, size_t workspace_bytes,
                             uint32_t* dev_err, simsd_stream_t stream);

simsd_status simsd_accept_coupled_ex(const void* target_logits, simsd_dtype logit_dtype,
                                     const int32_t* draft_tokens, const uint8_t* labels,
                                     const int32_t* pos_ids, int batch, int B, int gamma, int V,
                                     float temperature, uint64_t seed, uint64_t offset,
                                     int32_t* accepted_len, int32_t* out_tokens,
                                     int32_t* out_pos, int32_t* n_commit, void* workspace,
                                     size_t workspace_bytes, uint32_t* dev_err,
                                     simsd_stream_t stream);

/* ---------------------------------------------------------------------------------
 * simsd_expected_prefix  [S2D2-4]; steps and later rounds as simsd_accept.
 *
 * Routing statistic, computed from the draft logits alone (before the verify forward):
 * for every request r the expected accepted-prefix length
 *   K^_r = sum_{k=1..L} prod_{i=1..k} alpha_i,   L = min(gamma, R_r),
 * over the steps i = 1..L in the draft's time order (slot o_i, the slot labelled i), with
 *   SIMSD_KHAT_MARGIN:  alpha_i = 1 if m_i >= tau_margin else 0,
 *   SIMSD_KHAT_ENTROPY: alpha_i = exp(-beta * H~_i),
 * where p = softmax(draft_logits[r][o_i] / T) (T > 0), m_i = p_(1) - p_(2) (its two
 * largest probabilities; p_(2) = 0 when V = 1) and H~_i = H(p) / ln V (0 when V = 1).
 *   draft_logits  [batch, B, V] of logit_dtype (fp32, or bf16 widened exactly), indexed by
 *                 block slot; -inf entries hold no probability (every verified row needs a
 *                 finite entry).
 *   labels        uint8 [batch, 2B] from simsd_build_layout.
 *   temperature   T > 0; tau_margin any float; beta >= 0.
 *   khat          float [batch] out.
 *   alpha         float [batch, gamma] out, or NULL: alpha_i of step i + 1 (0 past L).
 * Numerics: fp32 with one pass over each row (top two values, sum of e^(z - m) and of
 * e^(z - m)(z - m)); alpha_i of the entropy estimator is within 2e-5 of its exact value
 * and K^ within L(L + 1)/2 * 2e-5; margin decisions are exact unless m_i is within a
 * relative 1e-5 of tau_margin.
 * Data errors: labels not a permutation (SIMSD_DEVERR_TAU) -> K^ = -1, alpha row 0.
 * Workspace: simsd_expected_prefix_workspace(batch, B, gamma, V) bytes (on the current
 * device), 256-byte aligned, no initialisation needed.
 * --------------------------------------------------------------------------------- */
size_t simsd_expected_prefix_workspace(int batch, int B, int gamma, int V);

simsd_status simsd_expected_prefix(const void* draft_logits, simsd_dtype logit_dtype,
                                   const uint8_t* labels, int batch, int B, int gamma, int V,
                                   float temperature, simsd_khat_mode mode, float tau_margin,
                                   float beta, float* khat, float* alpha, void* workspace,
                                   size_t workspace_bytes, uint32_t* dev_err,
                                   simsd_stream_t stream);

/* ---------------------------------------------------------------------------------
 * simsd_accept_noalloc -- the same operation as simsd_accept, for callers that cannot
 * allocate device memory. (Library addition: the pages have no counterpart to this call.)
 *
 * Some callers have no way to provide scratch memory: plugin hosts that hand the library
 * only its input and output buffers and expose no allocator, or runtimes that forbid
 * device allocation once serving has started (an allocation can synchronise the device
 * and has unbounded latency). This entry point takes no workspace and allocates nothing
 * (no cudaMalloc, cudaFree or allocating library routine): its scratch is a fixed
 * 1 MiB device array inside the library, present on every device that loads the library
 * until the process exits.
 *   - Arguments, outputs, error bits, sentinels and status codes: exactly as
 *     simsd_accept (the same argument checks run first, in the same order).
 *   - The first call on each device looks up that array's device address (a runtime
 *     query, with that device current) and caches it; make that first call before any
 *     stream capture. A device reset replaces the device's context, and with it the
 *     array's address: the next call notices the new context and looks the address up
 *     again (make it, too, outside any stream capture).
 *   - Sizes whose scratch would exceed the array (see simsd_accept_noalloc_max_scratch;
 *     simsd_accept_workspace(batch, B, gamma, V) must not exceed it) return
 *     SIMSD_ERR_WORKSPACE and launch nothing.
 *   - Every call shares the one array: calls that may overlap on the GPU (different
 *     streams without ordering between them) race and must not be issued; calls ordered
 *     on one stream are safe. The kernels reset the parts that must start at zero.
 * --------------------------------------------------------------------------------- */
simsd_status simsd_accept_noalloc(const float* target_logits, const float* draft_logits,
                                  const int32_t* draft_tokens, const uint8_t* labels,
                                  int batch, int B, int gamma, int V, float temperature,
                                  uint64_t seed, uint64_t offset, int32_t* accepted_len,
                                  int32_t* out_tokens, int32_t* out_pos, int32_t* n_commit,
                                  uint32_t* dev_err, simsd_stream_t stream);

/* Size in bytes of the fixed scratch array behind simsd_accept_noalloc. */
size_t simsd_accept_noalloc_max_scratch(void);

#ifdef __cplusplus
}
#endif

#endif /* SIMSD_H */
