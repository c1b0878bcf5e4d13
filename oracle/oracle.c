/*
 * oracle.c -- plain fp64 CPU reference for paged decode attention.
 *
 * TEST INFRASTRUCTURE ONLY.  The test-suite, the smoke check and the benchmark's
 * CPU-baseline leg are the only callers.  The product library (libpagedattn) never
 * loads, links or shares code with this file, and this file includes nothing of it.
 *
 * What is computed follows "[TIL] Optimizing paged attention" (retepy.com):
 *   - section "Data Layout": the KV cache is [physical_page][page_size][kv_heads]
 *     [head_dim]; each sequence has one query token with query_heads heads;
 *   - section "Baseline": logical page = t / page_size, slot = t % page_size,
 *     physical page = block_tables[b * max_pages_per_sequence + logical page],
 *     kv_head = q_head / (query_heads / kv_heads), score = scale * (q . k),
 *     softmax over the sequence's context, softmax-weighted sum of V, fp32 output.
 * The softmax is evaluated in the plain two-pass form (maximum, then exponentials
 * and their sum), in fp64, from fp16 inputs widened exactly; the kernels' online
 * recurrence and split/merge give the same value in exact arithmetic.
 *
 * Two cache layouts: 0 = [page][slot][kv_head][head_dim] as section "Data Layout" gives it;
 * 1 = [page][kv_head][slot][head_dim], the alternative layout the pages suggest comparing
 * (section "V2 (Vectorization)"), where one head's rows of a page are contiguous.
 *
 * Readings where the pages are silent:
 *   - a context length of 0 yields an all-zero output row (empty sum);
 *   - indices are checked: a context longer than max_pages_per_sequence*page_size,
 *     a negative context or a page id outside [0, num_physical_pages) makes the call
 *     return a nonzero code instead of reading out of bounds.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* IEEE 754 binary16 -> double, from the format's definition: 1 sign bit, 5 exponent
 * bits (bias 15), 10 fraction bits; exponent 0 encodes subnormals f * 2^-24,
 * exponent 31 encodes infinities (f == 0) and NaNs. Exact for every pattern. */
double oracle_half_to_double(uint16_t h) {
  int sign = (h >> 15) & 1;
  int e = (h >> 10) & 0x1f;
  int f = h & 0x3ff;
  double v;
  if (e == 0)
    v = ldexp((double)f, -24);
  else if (e == 31)
    v = f ? NAN : INFINITY;
  else
    v = ldexp((double)(f + 1024), e - 25);
  return sign ? -v : v;
}

typedef struct {
  int batch, query_heads, kv_heads, head_dim, page_size, max_pages, num_pages, layout;
} dims_t;

/* Element offset of (physical page, slot, kv head, 0) in the cache. */
static int64_t cache_row(const dims_t *p, int64_t page, int slot, int kv) {
  if (p->layout == 1) return ((page * p->kv_heads + kv) * (int64_t)p->page_size + slot) * p->head_dim;
  return ((page * p->page_size + slot) * (int64_t)p->kv_heads + kv) * p->head_dim;
}

/* Scores s_t = scale * q . K_t for t in [t0, t1) of one (sequence, q head). Returns 0 on
 * success, 2 on an out-of-range page id. */
static int scores(const dims_t *p, const uint16_t *qrow, const uint16_t *key,
                  const int32_t *bt, int b, int h, double scale, int t0, int t1, double *s) {
  int g = p->query_heads / p->kv_heads;
  int kv = h / g;
  for (int t = t0; t < t1; ++t) {
    int lp = t / p->page_size;
    int slot = t % p->page_size;
    int page = bt[(int64_t)b * p->max_pages + lp];
    if (page < 0 || page >= p->num_pages) return 2;
    const uint16_t *krow = key + cache_row(p, page, slot, kv);
    double acc = 0.0;
    for (int d = 0; d < p->head_dim; ++d)
      acc += oracle_half_to_double(qrow[d]) * oracle_half_to_double(krow[d]);
    s[t - t0] = scale * acc;
  }
  return 0;
}

static int check_dims(const dims_t *p) {
  if (p->batch < 0 || p->query_heads <= 0 || p->kv_heads <= 0 || p->head_dim <= 0 ||
      p->page_size <= 0 || p->max_pages <= 0 || p->num_pages <= 0)
    return 1;
  if (p->query_heads % p->kv_heads) return 1;
  if (p->layout != 0 && p->layout != 1) return 1;
  return 0;
}

/* Attention of query vector qrow (query head h of sequence b) over tokens [0, n):
 * out[d] = sum_t w_t V_t[d] / sum_t w_t with w_t = exp(s_t - max s). */
static int attend(const dims_t *p, const uint16_t *qrow, const uint16_t *key,
                  const uint16_t *value, const int32_t *bt, int b, int h, int n, double scale,
                  double *out) {
  int hd = p->head_dim;
  for (int d = 0; d < hd; ++d) out[d] = 0.0;
  if (n < 0 || (int64_t)n > (int64_t)p->max_pages * p->page_size) return 3;
  if (n == 0) return 0;
  double *s = (double *)malloc(sizeof(double) * (size_t)n);
  if (!s) return 4;
  int rc = scores(p, qrow, key, bt, b, h, scale, 0, n, s);
  if (rc) {
    free(s);
    return rc;
  }
  /* pass 1: the maximum score */
  double m = -INFINITY;
  for (int t = 0; t < n; ++t)
    if (s[t] > m) m = s[t];
  /* pass 2: weights, their sum, and the weighted sum of V */
  int g = p->query_heads / p->kv_heads;
  int kv = h / g;
  double l = 0.0;
  for (int t = 0; t < n; ++t) {
    double w = exp(s[t] - m);
    l += w;
    int page = bt[(int64_t)b * p->max_pages + t / p->page_size];
    const uint16_t *vrow = value + cache_row(p, page, t % p->page_size, kv);
    for (int d = 0; d < hd; ++d) out[d] += w * oracle_half_to_double(vrow[d]);
  }
  for (int d = 0; d < hd; ++d) out[d] /= l;
  free(s);
  return 0;
}

/* One decode output row: the sequence's single query token attends to all ctx[b] tokens. */
static int decode_row(const dims_t *p, const uint16_t *q, const uint16_t *key,
                      const uint16_t *value, const int32_t *bt, const int32_t *ctx,
                      double scale, int64_t row, double *out) {
  int b = (int)(row / p->query_heads);
  int h = (int)(row % p->query_heads);
  return attend(p, q + row * p->head_dim, key, value, bt, b, h, ctx[b], scale, out);
}

/* Full decode (rows == NULL: every (b, h), out is [batch][query_heads][head_dim]) or the
 * listed rows r = b * query_heads + h (out is [n_rows][head_dim]). n_threads <= 0 uses
 * the OpenMP default. Returns 0, or the first nonzero row code. */
int oracle_decode(int batch, int query_heads, int kv_heads, int head_dim, int page_size,
                  int max_pages, int num_pages, int layout, const uint16_t *query,
                  const uint16_t *key_cache, const uint16_t *value_cache,
                  const int32_t *block_tables, const int32_t *context_lengths, double scale,
                  const int64_t *rows, int64_t n_rows, double *out, int n_threads) {
  dims_t p = {batch, query_heads, kv_heads, head_dim, page_size, max_pages, num_pages, layout};
  if (check_dims(&p)) return 1;
  int64_t total = rows ? n_rows : (int64_t)batch * query_heads;
  int status = 0;
#ifdef _OPENMP
  if (n_threads > 0) omp_set_num_threads(n_threads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
  for (int64_t i = 0; i < total; ++i) {
    int64_t r = rows ? rows[i] : i;
    int rc = 5;
    if (r >= 0 && r < (int64_t)batch * query_heads)
      rc = decode_row(&p, query, key_cache, value_cache, block_tables, context_lengths, scale,
                      r, out + i * head_dim);
    if (rc) {
#ifdef _OPENMP
#pragma omp critical
#endif
      if (!status) status = rc;
    }
  }
  (void)n_threads;
  return status;
}

/* Multi-token (prefill) attention: sequence b has n_b = query_start[b + 1] - query_start[b]
 * new query tokens (rows query_start[b] .. of query, [total][query_heads][head_dim]); they
 * are the last n_b of its context_lengths[b] tokens, so new token j sits at position
 * p = context_lengths[b] - n_b + j and attends causally to tokens 0..p (the causal
 * extension of the decode step: "[TIL] Optimizing paged attention", section "Paged
 * Attention", applied to every new token). rows == NULL computes every (query row, head)
 * into out [total][query_heads][head_dim]; otherwise the listed flat rows i * qh + h.
 * Returns 0, 6 for inconsistent query_start / lengths, or a row code as decode. */
int oracle_prefill(int batch, int query_heads, int kv_heads, int head_dim, int page_size,
                   int max_pages, int num_pages, int layout, const uint16_t *query,
                   const int32_t *query_start, const uint16_t *key_cache,
                   const uint16_t *value_cache, const int32_t *block_tables,
                   const int32_t *context_lengths, double scale, const int64_t *rows,
                   int64_t n_rows, double *out, int n_threads) {
  dims_t p = {batch, query_heads, kv_heads, head_dim, page_size, max_pages, num_pages, layout};
  if (check_dims(&p)) return 1;
  if (query_start[0] != 0) return 6;
  for (int b = 0; b < batch; ++b) {
    int nb = query_start[b + 1] - query_start[b];
    if (nb < 0 || nb > context_lengths[b]) return 6;
  }
  const int64_t total = (int64_t)query_start[batch] * query_heads;
  const int64_t count = rows ? n_rows : total;
  int status = 0;
#ifdef _OPENMP
  if (n_threads > 0) omp_set_num_threads(n_threads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
  for (int64_t i = 0; i < count; ++i) {
    int64_t r = rows ? rows[i] : i;
    int rc = 5;
    if (r >= 0 && r < total) {
      int qi = (int)(r / query_heads);
      int h = (int)(r % query_heads);
      int b = 0;
      while (query_start[b + 1] <= qi) ++b;
      int nb = query_start[b + 1] - query_start[b];
      int pos = context_lengths[b] - nb + (qi - query_start[b]);
      rc = attend(&p, query + r * head_dim, key_cache, value_cache, block_tables, b, h, pos + 1,
                  scale, out + i * head_dim);
    }
    if (rc) {
#ifdef _OPENMP
#pragma omp critical
#endif
      if (!status) status = rc;
    }
  }
  (void)n_threads;
  return status;
}

/* Softmax state of one (b, h) over tokens [t0, t1): m = max s_t, l = sum exp(s_t - m),
 * acc[d] = sum exp(s_t - m) V_t[d] (not normalised).  An empty range gives
 * m = -inf, l = 0, acc = 0.  This is the per-split state of the context-split scheme in
 * "[TIL] Optimizing paged attention", section "V4 (Context-axis parallelism)". */
int oracle_partial(int batch, int query_heads, int kv_heads, int head_dim, int page_size,
                   int max_pages, int num_pages, int layout, const uint16_t *query,
                   const uint16_t *key_cache, const uint16_t *value_cache,
                   const int32_t *block_tables, const int32_t *context_lengths, double scale,
                   int64_t row, int t0, int t1, double *m_out, double *l_out,
                   double *acc_out) {
  dims_t p = {batch, query_heads, kv_heads, head_dim, page_size, max_pages, num_pages, layout};
  if (check_dims(&p)) return 1;
  if (row < 0 || row >= (int64_t)batch * query_heads) return 5;
  int b = (int)(row / query_heads);
  int h = (int)(row % query_heads);
  int n = context_lengths[b];
  if (n < 0 || (int64_t)n > (int64_t)max_pages * page_size) return 3;
  if (t0 < 0) t0 = 0;
  if (t1 > n) t1 = n;
  for (int d = 0; d < head_dim; ++d) acc_out[d] = 0.0;
  *m_out = -INFINITY;
  *l_out = 0.0;
  if (t1 <= t0) return 0;
  double *s = (double *)malloc(sizeof(double) * (size_t)(t1 - t0));
  if (!s) return 4;
  int rc = scores(&p, query + row * head_dim, key_cache, block_tables, b, h, scale, t0, t1, s);
  if (rc) {
    free(s);
    return rc;
  }
  double m = -INFINITY;
  for (int t = t0; t < t1; ++t)
    if (s[t - t0] > m) m = s[t - t0];
  int kv = h / (query_heads / kv_heads);
  double l = 0.0;
  for (int t = t0; t < t1; ++t) {
    double w = exp(s[t - t0] - m);
    l += w;
    int page = block_tables[(int64_t)b * max_pages + t / page_size];
    const uint16_t *vrow = value_cache + cache_row(&p, page, t % page_size, kv);
    for (int d = 0; d < head_dim; ++d) acc_out[d] += w * oracle_half_to_double(vrow[d]);
  }
  *m_out = m;
  *l_out = l;
  free(s);
  return 0;
}

/* Log-sum-exp merge of n partial states (m_i, l_i, acc_i[head_dim]) into one normalised
 * row, in the order given, as in the merge kernel of "[TIL] Optimizing paged attention",
 * section "V4 (Context-axis parallelism)": states with l_i == 0 (empty splits) are
 * skipped; otherwise M' = max(M, m_i), alpha = exp(M - M'), beta = exp(m_i - M'),
 * L = alpha L + beta l_i, O = alpha O + beta acc_i; finally out = O / L (0 if L == 0). */
void oracle_combine(int n, int head_dim, const double *m, const double *l, const double *acc,
                    double *out) {
  double M = -INFINITY, L = 0.0;
  for (int d = 0; d < head_dim; ++d) out[d] = 0.0;
  for (int i = 0; i < n; ++i) {
    if (l[i] == 0.0) continue;
    double Mn = m[i] > M ? m[i] : M;
    double alpha = (M == -INFINITY) ? 0.0 : exp(M - Mn);
    double beta = exp(m[i] - Mn);
    L = alpha * L + beta * l[i];
    for (int d = 0; d < head_dim; ++d) out[d] = alpha * out[d] + beta * acc[(int64_t)i * head_dim + d];
    M = Mn;
  }
  if (L == 0.0) {
    for (int d = 0; d < head_dim; ++d) out[d] = 0.0;
    return;
  }
  for (int d = 0; d < head_dim; ++d) out[d] /= L;
}

/* Append one token per sequence: the new K and V rows (fp16 bits, [batch][kv_heads]
 * [head_dim]) are written at token index t = context_lengths[b], i.e. physical page
 * block_tables[b][t / page_size], slot t % page_size, in the given layout -- the cache write
 * that precedes a decode step ("[TIL] Optimizing paged attention", section "Paged Attention":
 * the K and V of earlier tokens are kept and reused). A sequence whose t is outside
 * [0, max_pages * page_size) or whose page id is outside the pool is skipped; the return
 * value has bit 1 set for a page id and bit 2 for a length (0 if all rows were written). */
int oracle_append_kv(int batch, int query_heads, int kv_heads, int head_dim, int page_size,
                     int max_pages, int num_pages, int layout, const uint16_t *new_key,
                     const uint16_t *new_value, const int32_t *block_tables,
                     const int32_t *context_lengths, uint16_t *key_cache,
                     uint16_t *value_cache) {
  dims_t p = {batch, query_heads, kv_heads, head_dim, page_size, max_pages, num_pages, layout};
  if (check_dims(&p)) return -1;
  int flags = 0;
  for (int b = 0; b < batch; ++b) {
    int t = context_lengths[b];
    if (t < 0 || (int64_t)t >= (int64_t)max_pages * page_size) {
      flags |= 2;
      continue;
    }
    int page = block_tables[(int64_t)b * max_pages + t / page_size];
    if (page < 0 || page >= num_pages) {
      flags |= 1;
      continue;
    }
    for (int kv = 0; kv < kv_heads; ++kv) {
      int64_t dst = cache_row(&p, page, t % page_size, kv);
      int64_t src = ((int64_t)b * kv_heads + kv) * head_dim;
      for (int d = 0; d < head_dim; ++d) {
        key_cache[dst + d] = new_key[src + d];
        value_cache[dst + d] = new_value[src + d];
      }
    }
  }
  return flags;
}

int oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
