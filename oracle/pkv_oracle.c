/*
 * pkv_oracle.c -- plain, slow, fp64 CPU reference for single-token decode
 * attention against a paged KV cache.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may include, link,
 * load or call this file; only the tests, the package smoke check and the
 * bench's CPU-baseline leg use it.  It shares no code, header, table or
 * constant with the CUDA library.
 *
 * Sources (web pages; sections named by topic where the page has no heading):
 *   [KVFA] "KV Cache & Flash Attention." (kvcache-7e2.pages.dev)
 *   [DF]   "KV Cache & FlashAttention" (deepforge.srivtx.xyz)
 *   [AP]   "KV cache, paged, flash and sparse attention" (abhishekpatel.co)
 *   [OCP]  OCP 8-bit Floating Point Specification (OFP8), E4M3 format.
 *
 * The decode result has a plain definition (the pages call paged and flash
 * attention exact), so the attention reference is that definition written out
 * in fp64: two passes (max, then sum of exponentials), then the weighted sum
 * of V.  The streaming (online-softmax) functions are kept separately so the
 * tests can check the algorithm the kernels follow against the definition.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------ */
/* Cache size closed form.  [AP] "Opening the hood: how big is the     */
/* notebook?" and [DF] cache-size paragraph: one K and one V vector    */
/* per layer, per KV head, each d_head numbers wide.                   */
/* ------------------------------------------------------------------ */
uint64_t pkvo_kv_bytes_per_token(int32_t layers, int32_t kv_heads,
                                 int32_t head_dim, int32_t elem_bytes) {
  return (uint64_t)2 * (uint64_t)layers * (uint64_t)kv_heads *
         (uint64_t)head_dim * (uint64_t)elem_bytes;
}

/* [KVFA] memory-cost section, gqa_kv_bytes: whole-cache size for a batch. */
uint64_t pkvo_kv_bytes(int64_t tokens, int32_t layers, int32_t kv_heads,
                       int32_t head_dim, int32_t elem_bytes, int32_t batch) {
  return (uint64_t)batch * (uint64_t)tokens *
         pkvo_kv_bytes_per_token(layers, kv_heads, head_dim, elem_bytes);
}

/* ------------------------------------------------------------------ */
/* Work counts of [KVFA] opening section and [AP] "Arjun's first       */
/* attempt" / "Following one new token": without a cache, the step     */
/* run at sequence position i recomputes K/V for all i tokens present; */
/* the first step runs at the last prompt token (position 1 if the     */
/* prompt is empty).  With a cache each token is projected once: the   */
/* prompt once, then one row per new token.                            */
/* ------------------------------------------------------------------ */
int64_t pkvo_rows_recomputed(int64_t prompt, int64_t n_new) {
  int64_t rows = 0;
  int64_t first = prompt > 0 ? prompt : 1;
  for (int64_t step = 0; step < n_new; ++step) rows += first + step;
  return rows;
}

int64_t pkvo_rows_cached(int64_t prompt, int64_t n_new) {
  int64_t rows = prompt; /* the prompt is encoded once */
  for (int64_t step = 0; step < n_new; ++step) rows += 1;
  return rows;
}

/* ------------------------------------------------------------------ */
/* FP8 E4M3 (OCP OFP8): 1 sign bit, 4 exponent bits with bias 7, 3     */
/* mantissa bits; no infinities; S.1111.111 is NaN; the largest finite */
/* magnitude is 1.75 * 2^8 = 448; exponent field 0 holds subnormals    */
/* m/8 * 2^-6.                                                         */
/* ------------------------------------------------------------------ */
double pkvo_e4m3_decode(uint8_t code) {
  int sign = (code >> 7) & 1;
  int e = (code >> 3) & 0xF;
  int m = code & 0x7;
  double mag;
  if (e == 0xF && m == 0x7) return NAN;
  if (e == 0)
    mag = ldexp((double)m / 8.0, -6);
  else
    mag = ldexp(1.0 + (double)m / 8.0, e - 7);
  return sign ? -mag : mag;
}

/* Round to nearest representable E4M3 value, ties to the code with an even
 * last mantissa bit; magnitudes past 448 (including infinity) saturate to
 * 448 ("satfinite"); NaN encodes as 0x7F.  Done by brute force over the 127
 * non-negative finite codes, so that it follows the definition directly. */
uint8_t pkvo_e4m3_encode(float x) {
  if (isnan(x)) return 0x7F;
  int sign = signbit(x) ? 1 : 0;
  double a = fabs((double)x);
  int best = 0;
  double best_err = INFINITY;
  for (int c = 0; c <= 0x7E; ++c) {
    double v = pkvo_e4m3_decode((uint8_t)c);
    double err = fabs(v - a);
    if (err < best_err || (err == best_err && (c & 1) == 0 && (best & 1) == 1)) {
      best = c;
      best_err = err;
    }
  }
  if (a > 448.0) best = 0x7E;
  return (uint8_t)((sign << 7) | best);
}

/* Stored byte for a value x of KV head h under per-head scale s: the value
 * is divided by the scale in IEEE fp32, then encoded. */
uint8_t pkvo_e4m3_quantize(float x, float scale) {
  volatile float y = x / scale;
  return pkvo_e4m3_encode(y);
}

void pkvo_e4m3_quantize_array(const float* x, int64_t n, float scale,
                              uint8_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = pkvo_e4m3_quantize(x[i], scale);
}

void pkvo_e4m3_dequantize_array(const uint8_t* codes, int64_t n, double scale,
                                double* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = pkvo_e4m3_decode(codes[i]) * scale;
}

/* ------------------------------------------------------------------ */
/* One (1,N) attention row, by definition.  [KVFA] KV-cache section     */
/* (the decode step attends one query row against every cached key)    */
/* and [AP] "Following one new token through the cache" (the new       */
/* token is appended first, so the row covers it too).                 */
/*   s_t   = scale * sum_j q[j] * K[t][j]                              */
/*   out   = sum_t softmax(s)_t * V[t]                                 */
/* K and V rows are `stride` doubles apart.  ctx == 0 gives zeros.     */
/* ------------------------------------------------------------------ */
void pkvo_attend_row(const double* q, const double* K, const double* V,
                     int64_t ctx, int64_t stride, int32_t d, double scale,
                     double* out) {
  for (int32_t j = 0; j < d; ++j) out[j] = 0.0;
  if (ctx <= 0) return;
  /* pass 1: scores and their maximum */
  double mx = -INFINITY;
  for (int64_t t = 0; t < ctx; ++t) {
    double s = 0.0;
    for (int32_t j = 0; j < d; ++j) s += q[j] * K[t * stride + j];
    s *= scale;
    if (s > mx) mx = s;
  }
  /* pass 2: exponentials, their sum, and the weighted sum of V */
  double z = 0.0;
  for (int64_t t = 0; t < ctx; ++t) {
    double s = 0.0;
    for (int32_t j = 0; j < d; ++j) s += q[j] * K[t * stride + j];
    s *= scale;
    double e = exp(s - mx);
    z += e;
    for (int32_t j = 0; j < d; ++j) out[j] += e * V[t * stride + j];
  }
  for (int32_t j = 0; j < d; ++j) out[j] /= z;
}

/* Batched decode attention over the logical (unpaged) cache.
 *   q   [B][Hq][d]
 *   K,V [B][T][Hkv][d]      (T = logical capacity per sequence)
 *   ctx [B]                 (tokens attended, the appended one included)
 *   out [B][Hq][d]
 * Query head hq reads KV head hq / (Hq / Hkv): consecutive query heads
 * share one KV head ([KVFA] memory-cost section, GQA; [AP] "Opening the
 * hood", 32 query heads sharing each KV head among four). */
void pkvo_decode_attention(const double* q, const double* K, const double* V,
                           const int32_t* ctx, int32_t B, int32_t Hq,
                           int32_t Hkv, int32_t d, int64_t T, double scale,
                           double* out, int32_t nthreads) {
  int32_t g = Hq / Hkv;
  int64_t jobs = (int64_t)B * Hq;
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
  for (int64_t job = 0; job < jobs; ++job) {
    int64_t b = job / Hq;
    int32_t hq = (int32_t)(job % Hq);
    int32_t kv = hq / g;
    const double* Kb = K + ((b * T) * Hkv + kv) * d;
    const double* Vb = V + ((b * T) * Hkv + kv) * d;
    pkvo_attend_row(q + job * d, Kb, Vb, ctx[b], (int64_t)Hkv * d, d, scale,
                    out + job * d);
  }
}

int32_t pkvo_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* ------------------------------------------------------------------ */
/* Online softmax, in the order the pages give it ([KVFA] online-      */
/* softmax section; [DF] running-summary paragraph; [AP] "Flash        */
/* attention", the [1,2,3,0] walk-through):                            */
/*   per tile:  m_new = max(m, max(tile))                              */
/*              l     = l * exp(m - m_new) + sum exp(x - m_new)        */
/*   with the rescale factor taken as 0 while m is still -inf.         */
/* l_trace (optional, length ceil(n/tile)) receives l after each tile. */
/* ------------------------------------------------------------------ */
void pkvo_online_softmax_stats(const double* x, int64_t n, int64_t tile,
                               double* m_out, double* l_out, double* m_trace,
                               double* l_trace) {
  double m = -INFINITY, l = 0.0;
  int64_t k = 0;
  for (int64_t s = 0; s < n; s += tile, ++k) {
    int64_t e = s + tile < n ? s + tile : n;
    double m_new = m;
    for (int64_t i = s; i < e; ++i)
      if (x[i] > m_new) m_new = x[i];
    double factor = (m == -INFINITY) ? 0.0 : exp(m - m_new);
    double add = 0.0;
    for (int64_t i = s; i < e; ++i) add += exp(x[i] - m_new);
    l = l * factor + add;
    m = m_new;
    if (m_trace) m_trace[k] = m;
    if (l_trace) l_trace[k] = l;
  }
  *m_out = m;
  *l_out = l;
}

/* The same recurrence carried into the output ([KVFA] Flash Attention
 * section: the running output is rescaled by the same factor and the tile's
 * p*V is added; one division at the end).  Scores are taken in tiles of
 * `tile` tokens over one (1,N) row.  Also returns the unnormalised state. */
void pkvo_online_attend_row(const double* q, const double* K, const double* V,
                            int64_t ctx, int64_t stride, int32_t d,
                            double scale, int64_t tile, double* out,
                            double* m_out, double* l_out, double* o_unnorm) {
  double m = -INFINITY, l = 0.0;
  for (int32_t j = 0; j < d; ++j) o_unnorm[j] = 0.0;
  for (int64_t s0 = 0; s0 < ctx; s0 += tile) {
    int64_t e0 = s0 + tile < ctx ? s0 + tile : ctx;
    double m_new = m;
    for (int64_t t = s0; t < e0; ++t) {
      double s = 0.0;
      for (int32_t j = 0; j < d; ++j) s += q[j] * K[t * stride + j];
      s *= scale;
      if (s > m_new) m_new = s;
    }
    double factor = (m == -INFINITY) ? 0.0 : exp(m - m_new);
    l *= factor;
    for (int32_t j = 0; j < d; ++j) o_unnorm[j] *= factor;
    for (int64_t t = s0; t < e0; ++t) {
      double s = 0.0;
      for (int32_t j = 0; j < d; ++j) s += q[j] * K[t * stride + j];
      s *= scale;
      double p = exp(s - m_new);
      l += p;
      for (int32_t j = 0; j < d; ++j) o_unnorm[j] += p * V[t * stride + j];
    }
    m = m_new;
  }
  *m_out = m;
  *l_out = l;
  for (int32_t j = 0; j < d; ++j) out[j] = (ctx > 0) ? o_unnorm[j] / l : 0.0;
}

/* Merge of partial states over disjoint token sets ([DF] running-summary
 * paragraph: both the sum and the partial output are brought to a common
 * maximum by exp(m_old - m_new); [KVFA] online-softmax listing's guard for
 * an empty state).  Partials with l == 0 (empty) contribute nothing; if all
 * are empty the result is zero.
 *   m[n], l[n], o[n][d] (unnormalised)  ->  out[d] */
void pkvo_merge_partials(const double* m, const double* l, const double* o,
                         int32_t n, int32_t d, double* out) {
  double M = -INFINITY;
  for (int32_t i = 0; i < n; ++i)
    if (l[i] > 0.0 && m[i] > M) M = m[i];
  for (int32_t j = 0; j < d; ++j) out[j] = 0.0;
  if (M == -INFINITY) return;
  double L = 0.0;
  for (int32_t i = 0; i < n; ++i) {
    if (!(l[i] > 0.0)) continue;
    double w = exp(m[i] - M);
    L += w * l[i];
    for (int32_t j = 0; j < d; ++j) out[j] += w * o[(int64_t)i * d + j];
  }
  for (int32_t j = 0; j < d; ++j) out[j] /= L;
}

/* ------------------------------------------------------------------ */
/* Expected cache contents after an append ([KVFA] PagedAttention       */
/* section: block = table[pos // P], offset = pos % P; the slot number  */
/* written per token is block * P + offset, and -1 means "no slot").   */
/* The cache is [NB][Hkv][P][d] of elem_bytes-wide elements; rows of    */
/* `src` are [T][Hkv][d] of the same width.  16-bit caches copy bytes.  */
/* ------------------------------------------------------------------ */
void pkvo_append_bytes(uint8_t* cache, const uint8_t* src, const int64_t* slot,
                       int32_t T, int32_t NB, int32_t P, int32_t Hkv, int32_t d,
                       int32_t elem_bytes) {
  int64_t row = (int64_t)d * elem_bytes;
  for (int32_t t = 0; t < T; ++t) {
    if (slot[t] < 0) continue;
    int64_t blk = slot[t] / P, off = slot[t] % P;
    if (blk >= NB) continue;
    for (int32_t h = 0; h < Hkv; ++h) {
      uint8_t* dst = cache + (((blk * Hkv + h) * P) + off) * row;
      const uint8_t* s = src + ((int64_t)t * Hkv + h) * row;
      memcpy(dst, s, (size_t)row);
    }
  }
}

/* ------------------------------------------------------------------ */
/* Copy-on-write of whole blocks ([AP] "Paged attention: stop reserving */
/* empty tables": sequences point at the same physical blocks for a    */
/* shared beginning, copying only if one of them would change a block; */
/* [KVFA] PagedAttention section: sharing a prefix hands the second     */
/* sequence ceil(prefix / P) of the same blocks, so the last may be     */
/* partly filled).  Block b of the cache is the [Hkv][P][d] run at      */
/* b * block_bytes; dst[i] receives a copy of src[i]; pairs with either */
/* id outside [0, NB) are skipped.                                      */
/* ------------------------------------------------------------------ */
void pkvo_copy_blocks(uint8_t* cache, const int32_t* src, const int32_t* dst, int32_t n,
                      int32_t NB, int64_t block_bytes) {
  for (int32_t i = 0; i < n; ++i) {
    if (src[i] < 0 || src[i] >= NB || dst[i] < 0 || dst[i] >= NB) continue;
    memmove(cache + (int64_t)dst[i] * block_bytes, cache + (int64_t)src[i] * block_bytes,
            (size_t)block_bytes);
  }
}

/* Per-token FP8 scaling ("KV Cache & Flash Attention." (kvcache-7e2.pages.dev),
 * memory-cost section: the cache is quantized to fp8; Flash Attention
 * section: FP8 with finer-grained, per-block scales).  Reading: every appended
 * (token, KV head) row of K, and of V, gets its own fp32 scale, the row's
 * largest magnitude divided by 448 (the largest finite E4M3 value) in IEEE
 * fp32, so the row's largest element lands on +-448; an all-zero row takes
 * scale 1.  The row is then encoded under that scale like any E4M3 value. */
float pkvo_e4m3_token_scale(const float* row, int32_t d) {
  float amax = 0.0f;
  for (int32_t j = 0; j < d; ++j) {
    const float a = fabsf(row[j]);
    if (a > amax) amax = a;
  }
  if (amax == 0.0f) return 1.0f;
  volatile float s = amax / 448.0f;
  return s;
}

/* Per-token FP8 append: codes into the cache slot, the row's scale into the
 * same slot of the scale pool [NB][Hkv][P]. */
void pkvo_append_e4m3_token(uint8_t* cache, float* scales, const float* src,
                            const int64_t* slot, int32_t T, int32_t NB, int32_t P,
                            int32_t Hkv, int32_t d) {
  for (int32_t t = 0; t < T; ++t) {
    if (slot[t] < 0) continue;
    int64_t blk = slot[t] / P, off = slot[t] % P;
    if (blk >= NB) continue;
    for (int32_t h = 0; h < Hkv; ++h) {
      const int64_t r = (blk * Hkv + h) * P + off;
      const float* s = src + ((int64_t)t * Hkv + h) * d;
      const float sc = pkvo_e4m3_token_scale(s, d);
      scales[r] = sc;
      for (int32_t j = 0; j < d; ++j) cache[r * d + j] = pkvo_e4m3_quantize(s[j], sc);
    }
  }
}

/* fp64 rows [n][d] from codes and one fp32 scale per row. */
void pkvo_e4m3_dequantize_rows(const uint8_t* codes, const float* row_scale, int64_t n,
                               int32_t d, double* out) {
  for (int64_t i = 0; i < n; ++i)
    for (int32_t j = 0; j < d; ++j)
      out[i * d + j] = pkvo_e4m3_decode(codes[i * d + j]) * (double)row_scale[i];
}

/* FP8 cache: the row is divided by the KV head's fp32 scale and encoded. */
void pkvo_append_e4m3(uint8_t* cache, const float* src, const int64_t* slot,
                      const float* head_scale, int32_t T, int32_t NB, int32_t P,
                      int32_t Hkv, int32_t d) {
  for (int32_t t = 0; t < T; ++t) {
    if (slot[t] < 0) continue;
    int64_t blk = slot[t] / P, off = slot[t] % P;
    if (blk >= NB) continue;
    for (int32_t h = 0; h < Hkv; ++h) {
      uint8_t* dst = cache + (((blk * Hkv + h) * P) + off) * d;
      const float* s = src + ((int64_t)t * Hkv + h) * d;
      for (int32_t j = 0; j < d; ++j) dst[j] = pkvo_e4m3_quantize(s[j], head_scale[h]);
    }
  }
}
