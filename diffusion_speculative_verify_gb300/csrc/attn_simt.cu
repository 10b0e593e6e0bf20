// CUDA-core verify attention: one warp per (request, response row, query head).
//
// Serves the fp32 path (true fp32 arithmetic end to end: a tf32 tensor-core path would
// miss a 1e-5 tolerance) and bf16 shapes the tensor-core kernel does not take (D = 64,
// or more than 256 query rows per kv head). Lanes split the head dimension: lane l owns
// elements l + 32 j, so each RoPE pair (d, d + D/2) stays inside one lane.
#include "attn_common.cuh"

namespace simsd {

struct SimtArgs {
  int batch, B, Hq, Hkv, D, layout;
  int64_t cache_tokens;
  const void* q;
  const void* k_resp;
  const void* v_resp;
  const void* k_cache;
  const void* v_cache;
  const int64_t* cache_start;
  const int32_t* prompt_len;
  const int32_t* pos_ids;
  const uint8_t* labels;
  float scale_log2;  // softmax scale * log2(e)
  void* out;
  float* lse;
  uint32_t* dev_err;
  RopeTable rope;
};

template <typename T, int NPL>  // NPL = D / 32 elements per lane
__global__ void __launch_bounds__(256) attn_simt_kernel(const __grid_constant__ SimtArgs a) {
  const int lane = threadIdx.x & 31;
  const int64_t gw = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int twoB = 2 * a.B;
  const int64_t rows_total = (int64_t)a.batch * twoB * a.Hq;
  if (gw >= rows_total) return;
  const int hq = (int)(gw % a.Hq);
  const int s = (int)((gw / a.Hq) % twoB);
  const int r = (int)(gw / ((int64_t)a.Hq * twoB));
  const int G = a.Hq / a.Hkv;
  const int h = hq / G;
  const int D = a.D;
  const int half = D / 2;

  // checked build: the row's output, labels, position ids and request scalars lie inside
  // their arrays (else the row is skipped, SIMSD_DEVERR_BOUNDS raised)
  const int64_t orow = ((int64_t)r * twoB + s) * a.Hq + hq;
  const int64_t nrows = (int64_t)a.batch * twoB * a.Hq;
  if (!chk(orow * D, D, nrows * D, a.dev_err) || !chk((int64_t)r * twoB, twoB, (int64_t)a.batch * twoB, a.dev_err) ||
      !chk(r, 1, a.batch, a.dev_err))
    return;
  T* out = (T*)a.out + orow * D;
  const uint8_t* lab = a.labels + (int64_t)r * twoB;
  const uint8_t lab_s = lab[s];
  const int P = a.prompt_len[r];
  if (lab_s == kLabelInvalid || P < 0) {
    if (P < 0 && lane == 0 && s == 0 && hq == 0) atomicOr(a.dev_err, SIMSD_DEVERR_PROMPT_LEN);
#pragma unroll
    for (int j = 0; j < NPL; ++j) store_f(out + lane + 32 * j, 0.f);
    if (a.lse && lane == 0) a.lse[orow] = -INFINITY;
    return;
  }
  const int t = row_threshold(lab_s);
  const int pos_s = a.pos_ids[(int64_t)r * twoB + s];

  // rotated query, elements d = lane + 32 j
  float qv[NPL];
  {
    const T* qp = (const T*)a.q + orow * D;
#pragma unroll
    for (int j = 0; j < NPL; ++j) qv[j] = load_f(qp + lane + 32 * j);  // q has out's shape
#pragma unroll
    for (int j = 0; j < NPL / 2; ++j) {
      const int d = lane + 32 * j;  // first element of the pair (d, d + half)
      float sn, cs;
      rope_sincos(pos_s, a.rope.c_hi[d], a.rope.c_lo[d], &sn, &cs);
      const float x1 = qv[j], x2 = qv[j + NPL / 2];
      qv[j] = x1 * cs - x2 * sn;
      qv[j + NPL / 2] = x1 * sn + x2 * cs;
    }
  }
  (void)half;

  float m = -INFINITY, l = 0.f, acc[NPL];
#pragma unroll
  for (int j = 0; j < NPL; ++j) acc[j] = 0.f;

  auto consume = [&](const float* kv_k, const float* kv_v) {
    float dot = 0.f;
#pragma unroll
    for (int j = 0; j < NPL; ++j) dot = fmaf(qv[j], kv_k[j], dot);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
    const float sc = dot * a.scale_log2;
    if (sc > m) {
      const float corr = exp2f(m - sc);
      l *= corr;
#pragma unroll
      for (int j = 0; j < NPL; ++j) acc[j] *= corr;
      m = sc;
    }
    const float pr = exp2f(sc - m);
    l += pr;
#pragma unroll
    for (int j = 0; j < NPL; ++j) acc[j] = fmaf(pr, kv_v[j], acc[j]);
  };

  // every prompt key is visible (prompt tau = 0 precedes every step)
  const int64_t start = a.cache_start[r];
  const T* kc = (const T*)a.k_cache;
  const T* vc = (const T*)a.v_cache;
  const int64_t cache_elems = a.cache_tokens * a.Hkv * D;
  for (int jk = 0; jk < P; ++jk) {
    const int64_t base = cache_index(a.layout, a.cache_tokens, a.Hkv, D, start + jk, h);
    if (!chk(start + jk, 1, a.cache_tokens, a.dev_err) || !chk(base, D, cache_elems, a.dev_err))
      continue;
    float kk[NPL], vv[NPL];
#pragma unroll
    for (int j = 0; j < NPL; ++j) {
      kk[j] = load_f(kc + base + lane + 32 * j);
      vv[j] = load_f(vc + base + lane + 32 * j);
    }
    consume(kk, vv);
  }
  // response keys under the temporal-causal mask
  for (int js = 0; js < twoB; ++js) {
    if (!response_key_visible(lab[js], t)) continue;
    const int pos_j = a.pos_ids[(int64_t)r * twoB + js];
    const int64_t base = (((int64_t)r * twoB + js) * a.Hkv + h) * D;
    if (!chk(base, D, (int64_t)a.batch * twoB * a.Hkv * D, a.dev_err)) continue;
    float kk[NPL], vv[NPL];
#pragma unroll
    for (int j = 0; j < NPL; ++j) {
      kk[j] = load_f((const T*)a.k_resp + base + lane + 32 * j);
      vv[j] = load_f((const T*)a.v_resp + base + lane + 32 * j);
    }
#pragma unroll
    for (int j = 0; j < NPL / 2; ++j) {
      const int d = lane + 32 * j;
      float sn, cs;
      rope_sincos(pos_j, a.rope.c_hi[d], a.rope.c_lo[d], &sn, &cs);
      const float x1 = kk[j], x2 = kk[j + NPL / 2];
      kk[j] = x1 * cs - x2 * sn;
      kk[j + NPL / 2] = x1 * sn + x2 * cs;
    }
    consume(kk, vv);
  }
  const float inv = 1.f / l;
#pragma unroll
  for (int j = 0; j < NPL; ++j) store_f(out + lane + 32 * j, acc[j] * inv);
  if (a.lse && lane == 0) a.lse[orow] = (m + log2f(l)) * 0.69314718055994530942f;
}

simsd_status launch_attn_simt(const simsd_attn_params* p, cudaStream_t stream) {
  SimtArgs a;
  a.batch = p->batch;
  a.B = p->B;
  a.Hq = p->Hq;
  a.Hkv = p->Hkv;
  a.D = p->D;
  a.layout = (int)p->cache_layout;
  a.cache_tokens = p->cache_tokens;
  a.q = p->q;
  a.k_resp = p->k_resp;
  a.v_resp = p->v_resp;
  a.k_cache = p->k_cache;
  a.v_cache = p->v_cache;
  a.cache_start = p->cache_start;
  a.prompt_len = p->prompt_len;
  a.pos_ids = p->pos_ids;
  a.labels = p->labels;
  const float scale = p->softmax_scale > 0.f ? p->softmax_scale : (float)(1.0 / sqrt((double)p->D));
  a.scale_log2 = scale * 1.4426950408889634f;
  a.out = p->out;
  a.lse = p->lse;
  a.dev_err = p->dev_err;
  make_rope_table(&a.rope, (double)p->rope_theta, p->D);
  const int64_t warps_total = (int64_t)p->batch * 2 * p->B * p->Hq;
  const int threads = 256;
  const int64_t grid = (warps_total + (threads / 32) - 1) / (threads / 32);
  if (grid > 0x7fffffff) return SIMSD_ERR_UNSUPPORTED;
  if (p->dtype == SIMSD_DTYPE_FP32) {
    if (p->D == 64)
      attn_simt_kernel<float, 2><<<(unsigned)grid, threads, 0, stream>>>(a);
    else
      attn_simt_kernel<float, 4><<<(unsigned)grid, threads, 0, stream>>>(a);
  } else {
    if (p->D == 64)
      attn_simt_kernel<__nv_bfloat16, 2><<<(unsigned)grid, threads, 0, stream>>>(a);
    else
      attn_simt_kernel<__nv_bfloat16, 4><<<(unsigned)grid, threads, 0, stream>>>(a);
  }
  return last_launch_status();
}

}  // namespace simsd
