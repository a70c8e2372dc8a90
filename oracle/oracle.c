/*
 * Float64 CPU oracle for batched decode attention over a paged KV cache.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: only the tests, __graft_entry__.smoke() and the CPU
 * baseline / reference leg of bench.py use it.  It shares no code, header or
 * constant with the CUDA library it checks.
 *
 * What it computes (each step is written out plainly, in float64, with no
 * blocking, fusion or reordering):
 *
 *  - Paged KV gather.  "Paged attention (vLLM) - the KV-cache layout FlashInfer
 *    targets" (page "FlashDecoding + FlashInfer - the decode-time attention
 *    story"): every request owns a list of page ids; request i owns
 *    indices[indptr[i] .. indptr[i+1]) and its last page holds
 *    last_page_len[i] valid slots.  The cache is one tensor
 *    [num_pages, 2, page_size, num_kv_heads, head_dim] with K at index 0 and
 *    V at index 1, as the benchmark suite of the page "FlashInfer vs
 *    FlashAttention-3" (File 2) allocates it.
 *  - Decode attention for one query token per request:
 *        s_t  = sm_scale * sum_d q[i,h,d] * K_t[d]
 *        m    = max_t s_t,  d = sum_t exp(s_t - m)
 *        o    = sum_t exp(s_t - m) * V_t / d,   lse = m + ln d
 *    with query head h reading kv head h / (num_qo_heads / num_kv_heads).
 *  - The merge rule for two partial softmax states (page "FlashDecoding +
 *    FlashInfer", section "FlashDecoding - the split-KV trick"):
 *        m = max(m_a, m_b)
 *        d = d_a e^(m_a - m) + d_b e^(m_b - m)
 *        o = o_a e^(m_a - m) + o_b e^(m_b - m)
 *  - Exact decoding of the stored element types: fp32, bf16 (upper half of an
 *    IEEE binary32), IEEE binary16, and OCP FP8 E4M3 (the "FN" variant: no
 *    infinities, S.1111.111 is NaN) multiplied by its per-tensor fp32 scale.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORACLE_F32 = 0, ORACLE_BF16 = 1, ORACLE_F16 = 2, ORACLE_E4M3 = 3 };

/* ---- element decoding --------------------------------------------------- */

/* OCP 8-bit floating point, E4M3: 1 sign bit, 4 exponent bits (bias 7),
 * 3 mantissa bits.  Exponent field 0 encodes subnormals m/8 * 2^-6.  The only
 * NaN encodings are S.1111.111; there is no infinity, so S.1111.110 = 448 is
 * the largest finite magnitude. */
double oracle_decode_e4m3(uint8_t code) {
  int sign = (code >> 7) & 1;
  int e = (code >> 3) & 0xF;
  int m = code & 0x7;
  double v;
  if (e == 0xF && m == 0x7) return NAN;
  if (e == 0)
    v = ((double)m / 8.0) * pow(2.0, 1 - 7);
  else
    v = (1.0 + (double)m / 8.0) * pow(2.0, e - 7);
  return sign ? -v : v;
}

/* IEEE binary16: 1 sign bit, 5 exponent bits (bias 15), 10 mantissa bits. */
double oracle_decode_f16(uint16_t bits) {
  int sign = (bits >> 15) & 1;
  int e = (bits >> 10) & 0x1F;
  int m = bits & 0x3FF;
  double v;
  if (e == 0x1F) v = m ? NAN : INFINITY;
  else if (e == 0) v = ((double)m / 1024.0) * pow(2.0, 1 - 15);
  else v = (1.0 + (double)m / 1024.0) * pow(2.0, e - 15);
  return sign ? -v : v;
}

/* bfloat16 is the upper 16 bits of an IEEE binary32. */
double oracle_decode_bf16(uint16_t bits) {
  uint32_t u = (uint32_t)bits << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

static double load_elem(const void* base, int dtype, int64_t idx) {
  switch (dtype) {
    case ORACLE_F32: return (double)((const float*)base)[idx];
    case ORACLE_BF16: return oracle_decode_bf16(((const uint16_t*)base)[idx]);
    case ORACLE_F16: return oracle_decode_f16(((const uint16_t*)base)[idx]);
    case ORACLE_E4M3: return oracle_decode_e4m3(((const uint8_t*)base)[idx]);
  }
  return NAN;
}

/* ---- decode attention ---------------------------------------------------- */

/* Offset of element (page, kv, slot, kvh, d) in [num_pages, 2, P, Hkv, D]. */
static int64_t kv_offset(int64_t page, int kv, int slot, int kvh, int d, int P,
                         int Hkv, int D) {
  return (((page * 2 + kv) * (int64_t)P + slot) * Hkv + kvh) * (int64_t)D + d;
}

/* Decode attention with dequantisation scales either per tensor (k_scale,
 * v_scale) or, when k_scales / v_scales are given, per token and kv head:
 * the stored K (V) element of page p, slot t, kv head h is multiplied by
 * k_scales[(p * Hkv + h) * P + t] (v_scales likewise) - the row-wise dynamic
 * FP8 scaling of the page "FlashInfer vs FlashAttention-3" (section
 * "Production War Story: The FP8 Precision Underflow Failure").
 * Returns 0 on success, 1 on invalid arguments (nothing written then). */
static int decode_impl(const void* q, int q_dtype, const void* paged_kv,
                       int kv_dtype, int64_t num_pages, const int32_t* indptr,
                       const int32_t* indices, const int32_t* last_page_len,
                       int B, int Hq, int Hkv, int D, int P, double sm_scale,
                       double k_scale, double v_scale, const float* k_scales,
                       const float* v_scales, double* o, double* lse,
                       int num_threads) {
  if (B < 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || P <= 0 || Hq % Hkv) return 1;
  if (indptr[0] != 0) return 1;
  for (int i = 0; i < B; ++i) {
    int np = indptr[i + 1] - indptr[i];
    if (np < 0) return 1;
    if (np > 0 && (last_page_len[i] < 1 || last_page_len[i] > P)) return 1;
    for (int p = indptr[i]; p < indptr[i + 1]; ++p)
      if (indices[p] < 0 || indices[p] >= num_pages) return 1;
  }
  const int g = Hq / Hkv;
  const int64_t units = (int64_t)B * Hq;
#ifdef _OPENMP
  if (num_threads > 0) omp_set_num_threads(num_threads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
  for (int64_t u = 0; u < units; ++u) {
    const int i = (int)(u / Hq);
    const int h = (int)(u % Hq);
    const int kvh = h / g;
    const int np = indptr[i + 1] - indptr[i];
    const int64_t len = np > 0 ? (int64_t)(np - 1) * P + last_page_len[i] : 0;
    double* out = o + u * D;
    if (len == 0) {
      for (int d = 0; d < D; ++d) out[d] = 0.0;
      lse[u] = -INFINITY;
      continue;
    }
    double* s = (double*)malloc(sizeof(double) * len);
    /* scores */
    for (int64_t t = 0; t < len; ++t) {
      const int64_t page = indices[indptr[i] + t / P];
      const int slot = (int)(t % P);
      const double ks =
          k_scales ? (double)k_scales[(page * Hkv + kvh) * P + slot] : k_scale;
      double acc = 0.0;
      for (int d = 0; d < D; ++d) {
        double qd = load_elem(q, q_dtype, u * D + d);
        double kd = ks * load_elem(paged_kv, kv_dtype,
                                   kv_offset(page, 0, slot, kvh, d, P, Hkv, D));
        acc += qd * kd;
      }
      s[t] = sm_scale * acc;
    }
    /* softmax statistics */
    double m = -INFINITY;
    for (int64_t t = 0; t < len; ++t)
      if (s[t] > m) m = s[t];
    double den = 0.0;
    for (int64_t t = 0; t < len; ++t) den += exp(s[t] - m);
    /* weighted sum of values */
    for (int d = 0; d < D; ++d) out[d] = 0.0;
    for (int64_t t = 0; t < len; ++t) {
      const int64_t page = indices[indptr[i] + t / P];
      const int slot = (int)(t % P);
      const double vs =
          v_scales ? (double)v_scales[(page * Hkv + kvh) * P + slot] : v_scale;
      const double w = exp(s[t] - m);
      for (int d = 0; d < D; ++d)
        out[d] += w * vs *
                  load_elem(paged_kv, kv_dtype,
                            kv_offset(page, 1, slot, kvh, d, P, Hkv, D));
    }
    for (int d = 0; d < D; ++d) out[d] /= den;
    lse[u] = m + log(den);
    free(s);
  }
  return 0;
}

int oracle_batch_decode(const void* q, int q_dtype, const void* paged_kv,
                        int kv_dtype, int64_t num_pages, const int32_t* indptr,
                        const int32_t* indices, const int32_t* last_page_len,
                        int B, int Hq, int Hkv, int D, int P, double sm_scale,
                        double k_scale, double v_scale, double* o, double* lse,
                        int num_threads) {
  return decode_impl(q, q_dtype, paged_kv, kv_dtype, num_pages, indptr, indices,
                     last_page_len, B, Hq, Hkv, D, P, sm_scale, k_scale, v_scale,
                     NULL, NULL, o, lse, num_threads);
}

/* Same with per-token, per-kv-head scales [num_pages, Hkv, P] for K and V. */
int oracle_batch_decode_token_scales(
    const void* q, int q_dtype, const void* paged_kv, int kv_dtype,
    int64_t num_pages, const int32_t* indptr, const int32_t* indices,
    const int32_t* last_page_len, int B, int Hq, int Hkv, int D, int P,
    double sm_scale, const float* k_scales, const float* v_scales, double* o,
    double* lse, int num_threads) {
  if (!k_scales || !v_scales) return 1;
  return decode_impl(q, q_dtype, paged_kv, kv_dtype, num_pages, indptr, indices,
                     last_page_len, B, Hq, Hkv, D, P, sm_scale, 1.0, 1.0,
                     k_scales, v_scales, o, lse, num_threads);
}

/* Multi-token decode (speculative verification): every request carries
 * q_len query tokens, q [B, q_len, Hq, D], whose own K/V are the last q_len
 * positions of its context.  Query token i (0-based) attends to positions
 * 0 .. len - q_len + i: the context before the draft and the draft tokens up
 * to itself (the causal rule among the draft tokens).  Outputs
 * o [B, q_len, Hq, D] and lse [B, q_len, Hq].  Each query row is computed
 * exactly as decode_impl does for one token, over its own prefix. */
int oracle_batch_decode_multi(const void* q, int q_dtype, const void* paged_kv,
                              int kv_dtype, int64_t num_pages,
                              const int32_t* indptr, const int32_t* indices,
                              const int32_t* last_page_len, int B, int q_len,
                              int Hq, int Hkv, int D, int P, double sm_scale,
                              double k_scale, double v_scale, double* o,
                              double* lse, int num_threads) {
  if (q_len < 1 || B < 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || P <= 0 || Hq % Hkv) return 1;
  if (indptr[0] != 0) return 1;
  for (int i = 0; i < B; ++i) {
    const int np = indptr[i + 1] - indptr[i];
    if (np < 0) return 1;
    if (np == 0 || last_page_len[i] < 1 || last_page_len[i] > P) return 1;
    if ((int64_t)(np - 1) * P + last_page_len[i] < q_len) return 1;
    for (int p = indptr[i]; p < indptr[i + 1]; ++p)
      if (indices[p] < 0 || indices[p] >= num_pages) return 1;
  }
  const int g = Hq / Hkv;
  const int64_t units = (int64_t)B * q_len * Hq;
#ifdef _OPENMP
  if (num_threads > 0) omp_set_num_threads(num_threads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
  for (int64_t u = 0; u < units; ++u) {
    const int i = (int)(u / ((int64_t)q_len * Hq));
    const int qi = (int)((u / Hq) % q_len);
    const int h = (int)(u % Hq);
    const int kvh = h / g;
    const int np = indptr[i + 1] - indptr[i];
    const int64_t len = (int64_t)(np - 1) * P + last_page_len[i];
    const int64_t visible = len - q_len + qi + 1; /* positions 0 .. len - q_len + qi */
    double* out = o + u * D;
    double* s = (double*)malloc(sizeof(double) * visible);
    for (int64_t t = 0; t < visible; ++t) {
      const int64_t page = indices[indptr[i] + t / P];
      const int slot = (int)(t % P);
      double acc = 0.0;
      for (int d = 0; d < D; ++d)
        acc += load_elem(q, q_dtype, u * D + d) * k_scale *
               load_elem(paged_kv, kv_dtype, kv_offset(page, 0, slot, kvh, d, P, Hkv, D));
      s[t] = sm_scale * acc;
    }
    double m = -INFINITY;
    for (int64_t t = 0; t < visible; ++t)
      if (s[t] > m) m = s[t];
    double den = 0.0;
    for (int64_t t = 0; t < visible; ++t) den += exp(s[t] - m);
    for (int d = 0; d < D; ++d) out[d] = 0.0;
    for (int64_t t = 0; t < visible; ++t) {
      const int64_t page = indices[indptr[i] + t / P];
      const int slot = (int)(t % P);
      const double w = exp(s[t] - m);
      for (int d = 0; d < D; ++d)
        out[d] += w * v_scale *
                  load_elem(paged_kv, kv_dtype, kv_offset(page, 1, slot, kvh, d, P, Hkv, D));
    }
    for (int d = 0; d < D; ++d) out[d] /= den;
    lse[u] = m + log(den);
    free(s);
  }
  return 0;
}

/* Decode with a different number of query tokens per request, laid out
 * ragged: request i owns query rows qo_indptr[i] .. qo_indptr[i+1] of q and o
 * ([total_q, Hq, D]) and of lse ([total_q, Hq]) - the indptr layout of
 * section "Ragged attention - variable-length batching" of the page
 * "FlashDecoding + FlashInfer", applied to the queries.  With n_i query
 * tokens (the draft tokens a speculative verifier checks), they are the last
 * n_i positions of the request's cache, and query token j (0-based) attends
 * to positions 0 .. len_i - n_i + j: the context and the drafts up to itself.
 * n_i may be 0 (the request contributes no rows); n_i <= len_i otherwise. */
int oracle_batch_decode_ragged_q(const void* q, int q_dtype, const void* paged_kv,
                                 int kv_dtype, int64_t num_pages,
                                 const int32_t* indptr, const int32_t* indices,
                                 const int32_t* last_page_len,
                                 const int32_t* qo_indptr, int B, int Hq, int Hkv,
                                 int D, int P, double sm_scale, double k_scale,
                                 double v_scale, double* o, double* lse,
                                 int num_threads) {
  if (B < 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || P <= 0 || Hq % Hkv) return 1;
  if (indptr[0] != 0 || qo_indptr[0] != 0) return 1;
  for (int i = 0; i < B; ++i) {
    const int np = indptr[i + 1] - indptr[i];
    const int nq = qo_indptr[i + 1] - qo_indptr[i];
    if (np < 0 || nq < 0) return 1;
    if (nq == 0) continue;
    if (np == 0 || last_page_len[i] < 1 || last_page_len[i] > P) return 1;
    if ((int64_t)(np - 1) * P + last_page_len[i] < nq) return 1;
    for (int p = indptr[i]; p < indptr[i + 1]; ++p)
      if (indices[p] < 0 || indices[p] >= num_pages) return 1;
  }
  const int g = Hq / Hkv;
  const int64_t rows = (int64_t)qo_indptr[B] * Hq;
#ifdef _OPENMP
  if (num_threads > 0) omp_set_num_threads(num_threads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
  for (int64_t u = 0; u < rows; ++u) {
    const int64_t row = u / Hq; /* query token row */
    const int h = (int)(u % Hq);
    int i = 0; /* the request owning this row */
    while (qo_indptr[i + 1] <= row) ++i;
    const int nq = qo_indptr[i + 1] - qo_indptr[i];
    const int j = (int)(row - qo_indptr[i]);
    const int kvh = h / g;
    const int np = indptr[i + 1] - indptr[i];
    const int64_t len = (int64_t)(np - 1) * P + last_page_len[i];
    const int64_t visible = len - nq + j + 1;
    double* out = o + u * D;
    double* s = (double*)malloc(sizeof(double) * visible);
    for (int64_t t = 0; t < visible; ++t) {
      const int64_t page = indices[indptr[i] + t / P];
      const int slot = (int)(t % P);
      double acc = 0.0;
      for (int d = 0; d < D; ++d)
        acc += load_elem(q, q_dtype, u * D + d) * k_scale *
               load_elem(paged_kv, kv_dtype, kv_offset(page, 0, slot, kvh, d, P, Hkv, D));
      s[t] = sm_scale * acc;
    }
    double m = -INFINITY;
    for (int64_t t = 0; t < visible; ++t)
      if (s[t] > m) m = s[t];
    double den = 0.0;
    for (int64_t t = 0; t < visible; ++t) den += exp(s[t] - m);
    for (int d = 0; d < D; ++d) out[d] = 0.0;
    for (int64_t t = 0; t < visible; ++t) {
      const int64_t page = indices[indptr[i] + t / P];
      const int slot = (int)(t % P);
      const double w = exp(s[t] - m);
      for (int d = 0; d < D; ++d)
        out[d] += w * v_scale *
                  load_elem(paged_kv, kv_dtype, kv_offset(page, 1, slot, kvh, d, P, Hkv, D));
    }
    for (int d = 0; d < D; ++d) out[d] /= den;
    lse[u] = m + log(den);
    free(s);
  }
  return 0;
}

/* ---- merge of partial states -------------------------------------------- */

/* Each state is stored as a normalised output o_x (length D) with its
 * log-sum-exp lse_x.  In the (m, d, o) notation of the merge rule that state
 * is m = lse_x, d = 1 and unnormalised o = o_x; the rule is applied to those
 * and the result is normalised again: o = o_new / d_new, lse = m_new + ln d_new.
 * Two empty states (lse = -inf) merge to o = 0, lse = -inf. */
void oracle_merge_states(const double* o_a, const double* lse_a,
                         const double* o_b, const double* lse_b, double* o,
                         double* lse, int64_t n_states, int D) {
  for (int64_t k = 0; k < n_states; ++k) {
    const double m_a = lse_a[k], d_a = 1.0;
    const double m_b = lse_b[k], d_b = 1.0;
    const double m_new = m_a > m_b ? m_a : m_b;
    if (m_new == -INFINITY) {
      for (int d = 0; d < D; ++d) o[k * D + d] = 0.0;
      lse[k] = -INFINITY;
      continue;
    }
    const double w_a = exp(m_a - m_new), w_b = exp(m_b - m_new);
    const double d_new = d_a * w_a + d_b * w_b;
    for (int d = 0; d < D; ++d)
      o[k * D + d] = (o_a[k * D + d] * w_a + o_b[k * D + d] * w_b) / d_new;
    lse[k] = m_new + log(d_new);
  }
}

int oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
