/*
 * pkd_oracle.c -- fp64 CPU oracle for batch decode attention over a paged KV cache.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or call this
 * file: only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline leg use it.
 * It shares no code, header, table or constant with the CUDA library.
 *
 * What it computes is the plain definition of the method, written out with plain loops:
 *
 *   FlashInfer attention API page (docs.flashinfer.cn, api/attention.html), section
 *   "flashinfer.decode / BatchDecodeWithPagedKVCacheWrapper":
 *     - plan(): indptr [batch+1], indices [indptr[-1]], last_page_len [batch] with
 *       1 <= last_page_len <= page_size; num_qo_heads a multiple of num_kv_heads (GQA);
 *       window_left is the left (inclusive) window, -1 = whole sequence;
 *       logits_soft_cap c > 0 turns a logit x into c * tanh(x / c).
 *     - run(): q [batch, num_qo_heads, head_dim]; paged_kv_cache as one 5-D tensor
 *       [pages, 2, page_size, H_kv, D] (NHD) / [pages, 2, H_kv, page_size, D] (HND) or a
 *       (k, v) pair of 4-D tensors; q_scale / k_scale / v_scale calibration scales;
 *       returns o [batch, num_qo_heads, head_dim] and lse [batch, num_qo_heads], the
 *       log-sum-exp of the attention logits.
 *   The same page, batch prefill example: kv_len = page_size * (pages - 1) + last_page_len.
 *
 * Readings taken where the page is silent (each is listed in the design notes):
 *   - the logit x includes sm_scale, and the soft cap is applied to it: s = c*tanh(x/c);
 *   - lse is the natural logarithm of sum_t exp(s_t) over the attended keys;
 *   - the decode query sits at position n-1, so the attended keys are t >= n-1-window_left;
 *   - qo head g reads kv head g / (num_qo_heads / num_kv_heads);
 *   - calibration scales multiply: q = q_scale*Q, k = k_scale*K, v = v_scale*V;
 *   - a request with zero pages has kv_len 0, o = 0 and lse = -inf;
 *   - sm_scale defaults to 1/sqrt(head_dim) (that default is applied by the caller);
 *   - run()'s q_len_per_req (query tokens per request, default 1): the q_len tokens are the
 *     last positions of the request, token j at n - q_len + j, each with the causal mask of
 *     the page's batch prefill example (keys t <= its position) and its own window; q / o
 *     rows are request-major [batch * q_len, ...].
 *
 * Every floating-point step is in double precision; inputs are decoded exactly from
 * their bit patterns (fp16, bf16, fp8 e4m3fn).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { OR_F16 = 0, OR_BF16 = 1, OR_E4M3 = 2, OR_F32 = 3, OR_F64 = 4 };

/* IEEE-754 binary16: 1 sign, 5 exponent (bias 15), 10 fraction bits. */
double oracle_f16_to_f64(uint16_t h) {
  int sign = (h >> 15) & 1;
  int e = (h >> 10) & 0x1f;
  int m = h & 0x3ff;
  double v;
  if (e == 0) {
    v = ldexp((double)m, -24); /* subnormal: m * 2^-10 * 2^-14 */
  } else if (e == 31) {
    v = (m == 0) ? INFINITY : NAN;
  } else {
    v = ldexp(1024.0 + (double)m, e - 25); /* (1 + m/1024) * 2^(e-15) */
  }
  return sign ? -v : v;
}

/* bfloat16: the upper 16 bits of an IEEE-754 binary32. */
double oracle_bf16_to_f64(uint16_t b) {
  uint32_t bits = ((uint32_t)b) << 16;
  float f;
  memcpy(&f, &bits, sizeof f);
  return (double)f;
}

/* fp8 e4m3fn: 1 sign, 4 exponent (bias 7), 3 fraction bits; no infinities; S.1111.111 is
 * NaN; the largest finite value is 1.75 * 2^8 = 448. */
double oracle_e4m3_to_f64(uint8_t x) {
  int sign = (x >> 7) & 1;
  int e = (x >> 3) & 0xf;
  int m = x & 0x7;
  double v;
  if (e == 15 && m == 7) return NAN;
  if (e == 0) {
    v = ldexp((double)m, -9); /* subnormal: m/8 * 2^-6 */
  } else {
    v = ldexp(8.0 + (double)m, e - 10); /* (1 + m/8) * 2^(e-7) */
  }
  return sign ? -v : v;
}

static double load_elem(const void* base, int64_t idx, int dtype) {
  switch (dtype) {
    case OR_F16: return oracle_f16_to_f64(((const uint16_t*)base)[idx]);
    case OR_BF16: return oracle_bf16_to_f64(((const uint16_t*)base)[idx]);
    case OR_E4M3: return oracle_e4m3_to_f64(((const uint8_t*)base)[idx]);
    case OR_F32: return (double)((const float*)base)[idx];
    case OR_F64: return ((const double*)base)[idx];
    default: return NAN;
  }
}

/* Decode a whole array (used by the tests to pin the decoders against library casts). */
int oracle_decode_array(const void* src, int dtype, int64_t n, double* dst) {
  if (dtype < OR_F16 || dtype > OR_F64) return -1;
  for (int64_t i = 0; i < n; ++i) dst[i] = load_elem(src, i, dtype);
  return 0;
}

/* kv_len of request i from its page count and last-page fill (batch prefill example on
 * the FlashInfer page).  Zero pages means an empty request. */
static int64_t kv_len_of(const int32_t* indptr, const int32_t* last_page_len, int i,
                         int page_size) {
  int64_t pages = (int64_t)indptr[i + 1] - indptr[i];
  if (pages <= 0) return 0;
  return (int64_t)page_size * (pages - 1) + last_page_len[i];
}

int oracle_kv_len(const int32_t* indptr, const int32_t* last_page_len, int batch,
                  int page_size, int64_t* kv_len_out) {
  for (int i = 0; i < batch; ++i) kv_len_out[i] = kv_len_of(indptr, last_page_len, i, page_size);
  return 0;
}

/* The problem as one struct, so the per-(request, head) routine takes few arguments. */
typedef struct {
  int batch, num_qo_heads, num_kv_heads, head_dim, page_size;
  const int32_t* indptr;
  const int32_t* indices;
  const int32_t* last_page_len;
  const void* q;
  int q_dtype;
  const void* k_base;
  const void* v_base;
  int kv_dtype;
  int64_t page_stride, slot_stride, head_stride; /* elements; the last dim is contiguous */
  double sm_scale, logits_soft_cap;
  int window_left;
  double q_scale, k_scale, v_scale;
  int q_len; /* query tokens per request (run's q_len_per_req), >= 1 */
  int pos_mode; /* 0 NONE, 1 ROPE_LLAMA, 2 ALIBI (plan's pos_encoding_mode) */
  double rope_scale, rope_theta;
} oracle_problem;

/* ROPE_LLAMA ("LLaMA-style rotary embedding"): the vector x[D] at position pos is rotated
 * pairwise, dims (i, i + D/2) for i < D/2, by the angle (pos / rope_scale) * theta^(-2i/D):
 *   x_i' = x_i cos a - x_{i+D/2} sin a,   x_{i+D/2}' = x_{i+D/2} cos a + x_i sin a. */
static void rope_rotate(double* x, int D, double pos, double rope_scale, double rope_theta) {
  const int half = D / 2;
  for (int i = 0; i < half; ++i) {
    const double a = (pos / rope_scale) * pow(rope_theta, -2.0 * i / D);
    const double c = cos(a), s = sin(a);
    const double x0 = x[i], x1 = x[i + half];
    x[i] = x0 * c - x1 * s;
    x[i + half] = x1 * c + x0 * s;
  }
}

/* ALIBI: the slope of qo head g of H.  With m the largest power of two <= H, heads g < m take
 * 2^(-8 (g+1) / m) (the geometric sequence of the ALiBi paper), and the remaining heads take
 * every other slope of the 2m-head sequence, 2^(-4 (2 (g-m) + 1) / m). */
static double alibi_slope(int g, int H) {
  int m = 1;
  while (m * 2 <= H) m *= 2;
  if (g < m) return pow(2.0, -8.0 * (g + 1) / m);
  return pow(2.0, -4.0 * (2 * (g - m) + 1) / m);
}

/* Element offset of K/V token t of request i, kv head h, dim 0: token t lives in page
 * indices[indptr[i] + t / page_size] at slot t % page_size. */
static int64_t kv_offset(const oracle_problem* p, int i, int64_t t, int h) {
  int64_t page = p->indices[(int64_t)p->indptr[i] + t / p->page_size];
  int64_t slot = t % p->page_size;
  return page * p->page_stride + slot * p->slot_stride + (int64_t)h * p->head_stride;
}

/* Attention of query token j of request i, qo head g, restricted to the tokens t in
 * [t_begin, t_end) that its mask admits.  The request's q_len query tokens are the last
 * q_len positions of its sequence: token j sits at position pos = n - q_len + j and sees the
 * keys t <= pos (the causal mask of the prefill example, tril(diagonal = kv_len - qo_len)),
 * and with a window only t >= pos - window_left.  With q_len = 1 that is the decode query at
 * n - 1.  Writes o[D] and lse; if no token is admitted, o = 0, lse = -inf.  Two passes over
 * the keys: the logits and their maximum, then the weights. */
static void attend_range(const oracle_problem* p, int i, int j, int g, int64_t t_begin,
                         int64_t t_end, double* o, double* lse, double* s_buf, double* qv,
                         double* kv) {
  const int D = p->head_dim;
  const int group = p->num_qo_heads / p->num_kv_heads;
  const int h = g / group;
  const int64_t n = kv_len_of(p->indptr, p->last_page_len, i, p->page_size);
  const int64_t pos = n - p->q_len + j;
  int64_t first = 0;
  if (p->window_left >= 0 && pos - p->window_left > 0) first = pos - p->window_left;
  if (t_begin < first) t_begin = first;
  if (t_end > pos + 1) t_end = pos + 1;
  for (int d = 0; d < D; ++d) o[d] = 0.0;
  if (t_end <= t_begin) {
    *lse = -INFINITY;
    return;
  }
  const int64_t q_off = (((int64_t)i * p->q_len + j) * p->num_qo_heads + g) * D;
  for (int d = 0; d < D; ++d) qv[d] = p->q_scale * load_elem(p->q, q_off + d, p->q_dtype);
  if (p->pos_mode == 1) rope_rotate(qv, D, (double)pos, p->rope_scale, p->rope_theta);
  const double slope = p->pos_mode == 2 ? alibi_slope(g, p->num_qo_heads) : 0.0;
  double m = -INFINITY;
  for (int64_t t = t_begin; t < t_end; ++t) {
    const int64_t off = kv_offset(p, i, t, h);
    for (int d = 0; d < D; ++d) kv[d] = p->k_scale * load_elem(p->k_base, off + d, p->kv_dtype);
    if (p->pos_mode == 1) rope_rotate(kv, D, (double)t, p->rope_scale, p->rope_theta);
    double dot = 0.0;
    for (int d = 0; d < D; ++d) dot += qv[d] * kv[d];
    /* ALiBi adds slope * (t - pos), a penalty growing with the distance to the query, to the
     * scaled logit before the soft cap */
    double x = p->sm_scale * dot + slope * (double)(t - pos);
    double s = (p->logits_soft_cap > 0.0) ? p->logits_soft_cap * tanh(x / p->logits_soft_cap) : x;
    s_buf[t - t_begin] = s;
    if (s > m) m = s;
  }
  double l = 0.0;
  for (int64_t t = t_begin; t < t_end; ++t) {
    const double w = exp(s_buf[t - t_begin] - m);
    const int64_t off = kv_offset(p, i, t, h);
    l += w;
    for (int d = 0; d < D; ++d) o[d] += w * p->v_scale * load_elem(p->v_base, off + d, p->kv_dtype);
  }
  for (int d = 0; d < D; ++d) o[d] /= l;
  *lse = m + log(l);
}

/* Combine partial results (o_c, lse_c), c = 0..n-1, each the attention over a disjoint
 * subset of the keys, into the attention over their union:
 *   M = max_c lse_c,  w_c = exp(lse_c - M),  o = sum_c w_c o_c / sum_c w_c,
 *   lse = M + log(sum_c w_c).
 * Partials with lse = -inf (no keys) carry zero weight. */
int oracle_merge_states(int n, int head_dim, const double* o_parts, const double* lse_parts,
                        double* o, double* lse) {
  double M = -INFINITY;
  for (int c = 0; c < n; ++c)
    if (lse_parts[c] > M) M = lse_parts[c];
  for (int d = 0; d < head_dim; ++d) o[d] = 0.0;
  if (M == -INFINITY) {
    *lse = -INFINITY;
    return 0;
  }
  double wsum = 0.0;
  for (int c = 0; c < n; ++c) {
    const double w = exp(lse_parts[c] - M);
    wsum += w;
    for (int d = 0; d < head_dim; ++d) o[d] += w * o_parts[(int64_t)c * head_dim + d];
  }
  for (int d = 0; d < head_dim; ++d) o[d] /= wsum;
  *lse = M + log(wsum);
  return 0;
}

static int check_problem(const oracle_problem* p) {
  if (p->batch < 0 || p->num_qo_heads <= 0 || p->num_kv_heads <= 0 || p->head_dim <= 0 ||
      p->page_size <= 0 || p->q_len < 1)
    return -1;
  if (p->pos_mode < 0 || p->pos_mode > 2) return -1;
  if (p->pos_mode == 1 && (p->head_dim % 2 != 0 || !(p->rope_scale > 0) || !(p->rope_theta > 0)))
    return -1;
  if (p->num_qo_heads % p->num_kv_heads != 0) return -2;
  for (int i = 0; i < p->batch; ++i) {
    if (p->indptr[i + 1] < p->indptr[i]) return -3;
    if (p->indptr[i + 1] > p->indptr[i] &&
        (p->last_page_len[i] < 1 || p->last_page_len[i] > p->page_size))
      return -4;
  }
  return 0;
}

static int64_t max_kv_len(const oracle_problem* p) {
  int64_t mx = 1;
  for (int i = 0; i < p->batch; ++i) {
    int64_t n = kv_len_of(p->indptr, p->last_page_len, i, p->page_size);
    if (n > mx) mx = n;
  }
  return mx;
}

/*
 * Full batch decode with q_len query tokens per request (q and o rows: request-major,
 * [batch * q_len, num_qo_heads, head_dim]; q_len = 1 is plain decode).  chunk_tokens <= 0:
 * every (query token, head) attends over all its keys in one pass.  chunk_tokens > 0: the
 * keys are cut into consecutive chunks of that many tokens counted from token 0, each chunk
 * is attended separately and the chunks are combined with oracle_merge_states in chunk order
 * (the split-KV path written plainly).  num_threads <= 0 uses the OpenMP default.
 */
int oracle_batch_decode_pos(int batch, int q_len, int num_qo_heads, int num_kv_heads,
                            int head_dim, int page_size, const int32_t* indptr,
                            const int32_t* indices, const int32_t* last_page_len, const void* q,
                            int q_dtype, const void* k_base, const void* v_base, int kv_dtype,
                            int64_t page_stride, int64_t slot_stride, int64_t head_stride,
                            double sm_scale, double logits_soft_cap, int window_left,
                            double q_scale, double k_scale, double v_scale, int pos_mode,
                            double rope_scale, double rope_theta, int64_t chunk_tokens,
                            double* o, double* lse, int num_threads) {
  oracle_problem p = {batch, num_qo_heads, num_kv_heads, head_dim, page_size, indptr,
                      indices, last_page_len, q, q_dtype, k_base, v_base, kv_dtype,
                      page_stride, slot_stride, head_stride, sm_scale, logits_soft_cap,
                      window_left, q_scale, k_scale, v_scale, q_len, pos_mode, rope_scale,
                      rope_theta};
  int rc = check_problem(&p);
  if (rc != 0) return rc;
  const int64_t nmax = max_kv_len(&p);
  const int64_t work = (int64_t)batch * q_len * num_qo_heads;
  int bad = 0;
#ifdef _OPENMP
  if (num_threads > 0) omp_set_num_threads(num_threads);
#pragma omp parallel reduction(| : bad)
#endif
  {
    double* s_buf = (double*)malloc(sizeof(double) * (size_t)nmax);
    double* qv = (double*)malloc(sizeof(double) * (size_t)head_dim);
    double* kv = (double*)malloc(sizeof(double) * (size_t)head_dim);
    if (!qv || !kv) bad = 1;
    int64_t max_chunks = chunk_tokens > 0 ? (nmax + chunk_tokens - 1) / chunk_tokens : 1;
    double* o_parts = (double*)malloc(sizeof(double) * (size_t)(max_chunks * head_dim));
    double* lse_parts = (double*)malloc(sizeof(double) * (size_t)max_chunks);
    if (!s_buf || !o_parts || !lse_parts) bad = 1;
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
    for (int64_t w = 0; w < work; ++w) {
      if (bad) continue;
      const int64_t row = w / num_qo_heads;  /* = i * q_len + j */
      const int i = (int)(row / q_len);
      const int j = (int)(row % q_len);
      const int g = (int)(w % num_qo_heads);
      double* o_ig = o + w * head_dim;
      if (chunk_tokens <= 0) {
        attend_range(&p, i, j, g, 0, nmax + 1, o_ig, &lse[w], s_buf, qv, kv);
      } else {
        const int64_t n = kv_len_of(indptr, last_page_len, i, page_size);
        int nc = 0;
        for (int64_t t0 = 0; t0 < n; t0 += chunk_tokens, ++nc)
          attend_range(&p, i, j, g, t0, t0 + chunk_tokens, o_parts + (int64_t)nc * head_dim,
                       &lse_parts[nc], s_buf, qv, kv);
        oracle_merge_states(nc, head_dim, o_parts, lse_parts, o_ig, &lse[w]);
      }
    }
    free(s_buf);
    free(qv);
    free(kv);
    free(o_parts);
    free(lse_parts);
  }
  return bad ? -5 : 0;
}

/* Several query tokens per request, no positional encoding. */
int oracle_batch_decode_q(int batch, int q_len, int num_qo_heads, int num_kv_heads,
                          int head_dim, int page_size, const int32_t* indptr,
                          const int32_t* indices, const int32_t* last_page_len, const void* q,
                          int q_dtype, const void* k_base, const void* v_base, int kv_dtype,
                          int64_t page_stride, int64_t slot_stride, int64_t head_stride,
                          double sm_scale, double logits_soft_cap, int window_left,
                          double q_scale, double k_scale, double v_scale, int64_t chunk_tokens,
                          double* o, double* lse, int num_threads) {
  return oracle_batch_decode_pos(batch, q_len, num_qo_heads, num_kv_heads, head_dim, page_size,
                                 indptr, indices, last_page_len, q, q_dtype, k_base, v_base,
                                 kv_dtype, page_stride, slot_stride, head_stride, sm_scale,
                                 logits_soft_cap, window_left, q_scale, k_scale, v_scale, 0, 1.0,
                                 1e4, chunk_tokens, o, lse, num_threads);
}

/* Plain decode: one query token per request. */
int oracle_batch_decode(int batch, int num_qo_heads, int num_kv_heads, int head_dim,
                        int page_size, const int32_t* indptr, const int32_t* indices,
                        const int32_t* last_page_len, const void* q, int q_dtype,
                        const void* k_base, const void* v_base, int kv_dtype,
                        int64_t page_stride, int64_t slot_stride, int64_t head_stride,
                        double sm_scale, double logits_soft_cap, int window_left,
                        double q_scale, double k_scale, double v_scale, int64_t chunk_tokens,
                        double* o, double* lse, int num_threads) {
  return oracle_batch_decode_q(batch, 1, num_qo_heads, num_kv_heads, head_dim, page_size, indptr,
                               indices, last_page_len, q, q_dtype, k_base, v_base, kv_dtype,
                               page_stride, slot_stride, head_stride, sm_scale, logits_soft_cap,
                               window_left, q_scale, k_scale, v_scale, chunk_tokens, o, lse,
                               num_threads);
}

/* The number of threads an OpenMP region would use (reported with timings). */
int oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/*
 * MLA paged decode (FlashInfer attention API page, flashinfer.mla /
 * BatchMLAPagedAttentionWrapper, plan() and run()).  With the matrix-absorption trick the
 * page describes, every query head attends over one shared latent cache: the key of token t is
 * the concatenation [ckv_t, kpe_t] (head_dim_ckv + head_dim_kpe) and its value is ckv_t.
 *   q_nope [batch, H, Dc], q_pe [batch, H, Dp]; ckv_cache [pages, page_size, Dc],
 *   kpe_cache [pages, page_size, Dp]; request i owns pages kv_indices[kv_indptr[i] ..] and
 *   kv_len[i] tokens (token t in page kv_indices[kv_indptr[i] + t / page_size], slot
 *   t % page_size).
 *   logit_t = sm_scale * (<q_nope, ckv_t> + <q_pe, kpe_t>),  o = sum_t softmax(logit)_t ckv_t,
 *   lse = ln sum_t exp(logit_t) (the caller converts to base 2, run()'s default).
 * Decode: one query per request (qo_indptr = 0, 1, ..., batch); causal changes nothing then.
 * ckv / kpe rows are contiguous: element (page, slot, d) at (page * page_size + slot) * D + d.
 */
int oracle_mla_decode(int batch, int num_heads, int dc, int dp, int page_size,
                      const int32_t* kv_indptr, const int32_t* kv_indices, const int32_t* kv_len,
                      const void* q_nope, const void* q_pe, int q_dtype, const void* ckv,
                      const void* kpe, int kv_dtype, double sm_scale, double* o, double* lse,
                      int num_threads) {
  if (batch < 0 || num_heads <= 0 || dc <= 0 || dp < 0 || page_size <= 0) return -1;
  int64_t nmax = 1;
  for (int i = 0; i < batch; ++i) {
    if (kv_len[i] < 0) return -4;
    const int64_t pages = (int64_t)kv_indptr[i + 1] - kv_indptr[i];
    if (pages < 0 || (int64_t)kv_len[i] > pages * page_size) return -3;
    if (kv_len[i] > nmax) nmax = kv_len[i];
  }
  const int64_t work = (int64_t)batch * num_heads;
  int bad = 0;
#ifdef _OPENMP
  if (num_threads > 0) omp_set_num_threads(num_threads);
#pragma omp parallel reduction(| : bad)
#endif
  {
    double* s = (double*)malloc(sizeof(double) * (size_t)nmax);
    if (!s) bad = 1;
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
    for (int64_t w = 0; w < work; ++w) {
      if (bad) continue;
      const int i = (int)(w / num_heads);
      const int64_t n = kv_len[i];
      double* ow = o + w * dc;
      for (int d = 0; d < dc; ++d) ow[d] = 0.0;
      if (n == 0) {
        lse[w] = -INFINITY;
        continue;
      }
      double m = -INFINITY;
      for (int64_t t = 0; t < n; ++t) {
        const int64_t row = (int64_t)kv_indices[(int64_t)kv_indptr[i] + t / page_size] * page_size +
                            t % page_size;
        double dot = 0.0;
        for (int d = 0; d < dc; ++d)
          dot += load_elem(q_nope, w * dc + d, q_dtype) * load_elem(ckv, row * dc + d, kv_dtype);
        for (int d = 0; d < dp; ++d)
          dot += load_elem(q_pe, w * dp + d, q_dtype) * load_elem(kpe, row * dp + d, kv_dtype);
        s[t] = sm_scale * dot;
        if (s[t] > m) m = s[t];
      }
      double l = 0.0;
      for (int64_t t = 0; t < n; ++t) {
        const int64_t row = (int64_t)kv_indices[(int64_t)kv_indptr[i] + t / page_size] * page_size +
                            t % page_size;
        const double p = exp(s[t] - m);
        l += p;
        for (int d = 0; d < dc; ++d) ow[d] += p * load_elem(ckv, row * dc + d, kv_dtype);
      }
      for (int d = 0; d < dc; ++d) ow[d] /= l;
      lse[w] = m + log(l);
    }
    free(s);
  }
  return bad ? -5 : 0;
}
