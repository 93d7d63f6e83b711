/*
 * pskv_oracle.c -- plain fp64 CPU oracle for paged split-KV GQA decode attention.
 *
 * TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the bench's
 * CPU-baseline leg are its only users.  It shares no code with the CUDA path.
 *
 * What it computes (sources cited by page title and section; see the header):
 *  - decode attention is exact dense softmax attention, so the reference is
 *    the definition itself in double precision ([gem] "Fixed production
 *    shape": exact dense attention; intro: an independent double-precision
 *    direct-softmax reference);
 *  - keys are read through a page table ([tf1619] "Paged");
 *  - the split-KV path builds online-softmax partials (running max M, sum S,
 *    unnormalised numerator O) one key at a time in sequence order, merges
 *    them with M = max(Ma, Mb), S = Sa e^(Ma-M) + Sb e^(Mb-M),
 *    O = Oa e^(Ma-M) + Ob e^(Mb-M), and finalizes O / S ([gem] intro and
 *    "Candidate ownership and storage"); the merge runs in two levels
 *    ([pg1055] Description);
 *  - a window lower bound masks the oldest resident keys ([pg1057]
 *    Description).
 * Inputs are decoded exactly (bf16 and f32 values are exact doubles).
 */
#include "pskv_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

int orc_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* ---- input decoding ----------------------------------------------------- */

static double bf16_to_double(uint16_t bits) {
  uint32_t u = ((uint32_t)bits) << 16; /* bf16 is the top half of an f32 */
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

static double load_elem(const void *base, int dtype, size_t idx) {
  if (dtype == ORC_BF16) return bf16_to_double(((const uint16_t *)base)[idx]);
  return (double)((const float *)base)[idx];
}

static size_t elem_size(int dtype) { return dtype == ORC_BF16 ? 2 : 4; }

/* ---- dense attention for one query head --------------------------------- */

static double dot(const double *a, const double *b, int n) {
  double s = 0.0;
  for (int i = 0; i < n; ++i) s += a[i] * b[i];
  return s;
}

int orc_attend_direct(const double *q, const double *k, const double *v, int dk, int dv,
                      int begin, int end, double scale, double *out) {
  if (!q || !k || !v || !out || dk <= 0 || dv <= 0 || begin < 0 || end <= begin)
    return ORC_ERR_INVALID;
  int n = end - begin;
  double *s = (double *)malloc(sizeof(double) * (size_t)n);
  if (!s) return ORC_ERR_INVALID;
  double mx = -INFINITY;
  for (int i = 0; i < n; ++i) {
    s[i] = scale * dot(q, k + (size_t)(begin + i) * dk, dk);
    if (s[i] > mx) mx = s[i];
  }
  /* softmax(s)_i = e^(s_i - mx) / sum_j e^(s_j - mx) */
  double z = 0.0;
  for (int i = 0; i < n; ++i) {
    s[i] = exp(s[i] - mx);
    z += s[i];
  }
  for (int d = 0; d < dv; ++d) out[d] = 0.0;
  for (int i = 0; i < n; ++i) {
    const double w = s[i] / z;
    const double *vi = v + (size_t)(begin + i) * dv;
    for (int d = 0; d < dv; ++d) out[d] += w * vi[d];
  }
  free(s);
  return ORC_OK;
}

int orc_online_partial(const double *q, const double *k, const double *v, int dk, int dv,
                       int begin, int end, double scale, double *m, double *l, double *o) {
  if (!q || !k || !v || !m || !l || !o || dk <= 0 || dv <= 0 || begin < 0 || end < begin)
    return ORC_ERR_INVALID;
  double M = -INFINITY, S = 0.0;
  for (int d = 0; d < dv; ++d) o[d] = 0.0;
  for (int i = begin; i < end; ++i) {
    const double s = scale * dot(q, k + (size_t)i * dk, dk);
    const double *vi = v + (size_t)i * dv;
    if (s > M) {
      /* new running max: rescale what was accumulated under the old one */
      const double alpha = (M == -INFINITY) ? 0.0 : exp(M - s);
      S *= alpha;
      for (int d = 0; d < dv; ++d) o[d] *= alpha;
      M = s;
    }
    const double p = exp(s - M);
    S += p;
    for (int d = 0; d < dv; ++d) o[d] += p * vi[d];
  }
  *m = M;
  *l = S;
  return ORC_OK;
}

/* A state is valid when it is the empty state (-inf, 0, 0) or has a finite
 * max, a positive finite sum and a finite numerator.  Anything else (NaN
 * anywhere, +inf max, an empty max carrying mass) fails closed. */
static int state_valid(double m, double l, const double *o, int dv) {
  if (isnan(m) || isnan(l)) return 0;
  if (m == INFINITY) return 0;
  if (m == -INFINITY) {
    if (l != 0.0) return 0;
    for (int d = 0; d < dv; ++d)
      if (o[d] != 0.0) return 0;
    return 1;
  }
  if (!(l > 0.0) || isinf(l)) return 0;
  for (int d = 0; d < dv; ++d)
    if (!isfinite(o[d])) return 0;
  return 1;
}

int orc_merge(double ma, double la, const double *oa, double mb, double lb, const double *ob,
              int dv, double *m, double *l, double *o) {
  if (!oa || !ob || !m || !l || !o || dv <= 0) return ORC_ERR_INVALID;
  if (!state_valid(ma, la, oa, dv) || !state_valid(mb, lb, ob, dv)) return ORC_ERR_STATE;
  if (mb == -INFINITY) { /* b empty: a unchanged */
    *m = ma;
    *l = la;
    if (o != oa) memmove(o, oa, sizeof(double) * (size_t)dv);
    return ORC_OK;
  }
  if (ma == -INFINITY) { /* a empty: b unchanged */
    *m = mb;
    *l = lb;
    if (o != ob) memmove(o, ob, sizeof(double) * (size_t)dv);
    return ORC_OK;
  }
  const double M = ma > mb ? ma : mb;
  const double ea = exp(ma - M), eb = exp(mb - M);
  *l = la * ea + lb * eb;
  for (int d = 0; d < dv; ++d) o[d] = oa[d] * ea + ob[d] * eb;
  *m = M;
  return ORC_OK;
}

int orc_finalize(double m, double l, const double *o, int dv, double *out) {
  if (!o || !out || dv <= 0) return ORC_ERR_INVALID;
  if (!state_valid(m, l, o, dv) || m == -INFINITY) return ORC_ERR_STATE;
  for (int d = 0; d < dv; ++d) out[d] = o[d] / l;
  return ORC_OK;
}

int orc_attend_partitioned(const double *q, const double *k, const double *v, int dk, int dv,
                           const int *bounds, int num_parts, int group_size, double scale,
                           double *out) {
  if (!bounds || num_parts <= 0 || group_size <= 0 || dv <= 0) return ORC_ERR_INVALID;
  for (int p = 0; p < num_parts; ++p)
    if (bounds[p] < 0 || bounds[p + 1] < bounds[p]) return ORC_ERR_INVALID;
  int rc = ORC_OK;
  double *po = (double *)malloc(sizeof(double) * (size_t)dv); /* one partial */
  double *go = (double *)malloc(sizeof(double) * (size_t)dv); /* group fold */
  double *to = (double *)malloc(sizeof(double) * (size_t)dv); /* total fold */
  if (!po || !go || !to) {
    rc = ORC_ERR_INVALID;
    goto done;
  }
  double tm = -INFINITY, tl = 0.0;
  for (int d = 0; d < dv; ++d) to[d] = 0.0;
  for (int g0 = 0; g0 < num_parts; g0 += group_size) {
    double gm = -INFINITY, gl = 0.0;
    for (int d = 0; d < dv; ++d) go[d] = 0.0;
    const int g1 = g0 + group_size < num_parts ? g0 + group_size : num_parts;
    for (int p = g0; p < g1; ++p) { /* level 1: fold the group in order */
      double pm, pl;
      rc = orc_online_partial(q, k, v, dk, dv, bounds[p], bounds[p + 1], scale, &pm, &pl, po);
      if (rc) goto done;
      rc = orc_merge(gm, gl, go, pm, pl, po, dv, &gm, &gl, go);
      if (rc) goto done;
    }
    rc = orc_merge(tm, tl, to, gm, gl, go, dv, &tm, &tl, to); /* level 2 */
    if (rc) goto done;
  }
  rc = orc_finalize(tm, tl, to, dv, out);
done:
  free(po);
  free(go);
  free(to);
  return rc;
}

/* ---- single-precision twin of the online path --------------------------- */

static int partial_f32(const float *q, const float *k, const float *v, int dk, int dv, int begin,
                       int end, float scale, float *m, float *l, float *o) {
  float M = -INFINITY, S = 0.0f;
  for (int d = 0; d < dv; ++d) o[d] = 0.0f;
  for (int i = begin; i < end; ++i) {
    float acc = 0.0f;
    const float *ki = k + (size_t)i * dk;
    for (int d = 0; d < dk; ++d) acc += q[d] * ki[d];
    const float s = scale * acc;
    const float *vi = v + (size_t)i * dv;
    if (s > M) {
      const float alpha = (M == -INFINITY) ? 0.0f : expf(M - s);
      S *= alpha;
      for (int d = 0; d < dv; ++d) o[d] *= alpha;
      M = s;
    }
    const float p = expf(s - M);
    S += p;
    for (int d = 0; d < dv; ++d) o[d] += p * vi[d];
  }
  *m = M;
  *l = S;
  return ORC_OK;
}

int orc_attend_partitioned_f32(const float *q, const float *k, const float *v, int dk, int dv,
                               const int *bounds, int num_parts, float scale, float *out) {
  if (!q || !k || !v || !out || !bounds || num_parts <= 0 || dk <= 0 || dv <= 0)
    return ORC_ERR_INVALID;
  float *po = (float *)malloc(sizeof(float) * (size_t)dv);
  float *to = (float *)malloc(sizeof(float) * (size_t)dv);
  if (!po || !to) {
    free(po);
    free(to);
    return ORC_ERR_INVALID;
  }
  float tm = -INFINITY, tl = 0.0f;
  for (int d = 0; d < dv; ++d) to[d] = 0.0f;
  for (int p = 0; p < num_parts; ++p) {
    float pm, pl;
    partial_f32(q, k, v, dk, dv, bounds[p], bounds[p + 1], scale, &pm, &pl, po);
    if (pm == -INFINITY) continue; /* empty partition */
    if (tm == -INFINITY) {
      tm = pm;
      tl = pl;
      memcpy(to, po, sizeof(float) * (size_t)dv);
      continue;
    }
    const float M = tm > pm ? tm : pm;
    const float ea = expf(tm - M), eb = expf(pm - M);
    tl = tl * ea + pl * eb;
    for (int d = 0; d < dv; ++d) to[d] = to[d] * ea + po[d] * eb;
    tm = M;
  }
  int rc = ORC_OK;
  if (tm == -INFINITY)
    rc = ORC_ERR_STATE;
  else
    for (int d = 0; d < dv; ++d) out[d] = to[d] / tl;
  free(po);
  free(to);
  return rc;
}

/* ---- paged pool ---------------------------------------------------------- */

static int pool_valid(const orc_pool *p) {
  if (!(p && p->k && p->v && (p->dtype == ORC_F32 || p->dtype == ORC_BF16) &&
        p->num_pages > 0 && p->page_size > 0 && p->num_kv_heads > 0 && p->head_dim_k > 0 &&
        p->head_dim_v > 0))
    return 0;
  if (p->format == ORC_SPLIT) return 1;
  return p->format == ORC_FOLDED && p->head_dim_k < p->head_dim_v;
}

/* Width of the key a query meets (and of the query). */
static int key_width(const orc_pool *p) {
  return p->format == ORC_FOLDED ? p->head_dim_v : p->head_dim_k;
}

/* Element d of the key stored at element offsets kr (K region) and vr (V
 * region): a folded pool takes columns past its K width from V. */
static double key_elem(const orc_pool *p, size_t kr, size_t vr, int d) {
  if (p->format == ORC_FOLDED && d >= p->head_dim_k) return load_elem(p->v, p->dtype, vr + d);
  return load_elem(p->k, p->dtype, kr + d);
}

int orc_gather(const orc_pool *pool, const int32_t *page_tables, int table_stride, int b, int g,
               int len, double *k_out, double *v_out) {
  if (!pool_valid(pool) || !page_tables || table_stride <= 0 || b < 0 || g < 0 ||
      g >= pool->num_kv_heads || len < 0 || !k_out || !v_out)
    return ORC_ERR_INVALID;
  if ((int64_t)len > (int64_t)table_stride * pool->page_size) return ORC_ERR_INVALID;
  const int ps = pool->page_size, H = pool->num_kv_heads;
  const int dk = pool->head_dim_k, dv = pool->head_dim_v, kw = key_width(pool);
  for (int i = 0; i < len; ++i) {
    const int32_t page = page_tables[(size_t)b * table_stride + i / ps];
    if (page < 0 || page >= pool->num_pages) return ORC_ERR_BAD_PAGE;
    const size_t row = ((size_t)page * H + g) * ps + (size_t)(i % ps);
    for (int d = 0; d < kw; ++d) k_out[(size_t)i * kw + d] = key_elem(pool, row * dk, row * dv, d);
    for (int d = 0; d < dv; ++d) v_out[(size_t)i * dv + d] = load_elem(pool->v, pool->dtype, row * dv + d);
  }
  return ORC_OK;
}

int orc_append_rows(void *k_region, void *v_region, const orc_pool *pool, const void *k_new,
                    const void *v_new, const int32_t *row_of, const int32_t *pos_of, int n,
                    const int32_t *page_tables, int table_stride,
                    const int32_t *num_pages_of_row, int batch) {
  if (!k_region || !v_region || !pool_valid(pool) || n < 0 || (n > 0 && (!k_new || !v_new ||
      !row_of || !pos_of)) || !page_tables || table_stride <= 0 || !num_pages_of_row || batch <= 0)
    return ORC_ERR_INVALID;
  const int ps = pool->page_size, H = pool->num_kv_heads;
  /* check every row before writing any ([tf1619] "Leasing": rows past a slot's pages are refused) */
  for (int r = 0; r < n; ++r) {
    const int b = row_of[r], pos = pos_of[r];
    if (b < 0 || b >= batch || pos < 0) return ORC_ERR_INVALID;
    const int64_t lease = num_pages_of_row[b];
    if (lease < 0 || lease > table_stride) return ORC_ERR_INVALID;
    if ((int64_t)pos >= lease * ps) return ORC_ERR_PAST_PAGES;
    const int32_t page = page_tables[(size_t)b * table_stride + pos / ps];
    if (page < 0 || page >= pool->num_pages) return ORC_ERR_BAD_PAGE;
  }
  const size_t es = elem_size(pool->dtype);
  const size_t kbytes = (size_t)pool->head_dim_k * es, vbytes = (size_t)pool->head_dim_v * es;
  for (int r = 0; r < n; ++r) {
    const int b = row_of[r], pos = pos_of[r];
    const int32_t page = page_tables[(size_t)b * table_stride + pos / ps];
    for (int h = 0; h < H; ++h) {
      const size_t dst = ((size_t)page * H + h) * ps + (size_t)(pos % ps);
      const size_t src = (size_t)r * H + h;
      memcpy((char *)k_region + dst * kbytes, (const char *)k_new + src * kbytes, kbytes);
      memcpy((char *)v_region + dst * vbytes, (const char *)v_new + src * vbytes, vbytes);
    }
  }
  return ORC_OK;
}

/* First attended key index of a row: position first_pos + i must be >= window_lo. */
static int first_key(const int32_t *first_pos, const int32_t *window_lo, int b, int len) {
  if (!first_pos || !window_lo) return 0;
  int64_t i0 = (int64_t)window_lo[b] - (int64_t)first_pos[b];
  if (i0 < 0) i0 = 0;
  if (i0 > len) i0 = len;
  return (int)i0;
}

/* Index of element 0 of key i of (row b, kv head g), found through the page table. */
static size_t paged_row(const orc_pool *pool, int dim, const int32_t *page_tables, int table_stride,
                        int b, int g, int i) {
  const int32_t page = page_tables[(size_t)b * table_stride + i / pool->page_size];
  const size_t row = ((size_t)page * pool->num_kv_heads + g) * pool->page_size + (size_t)(i % pool->page_size);
  return row * (size_t)dim;
}

/* Checks shared by both decode paths. */
static int decode_args_ok(const orc_pool *pool, const void *q, const int32_t *page_tables,
                          int table_stride, const int32_t *seq_lens, const int32_t *first_pos,
                          const int32_t *window_lo, int batch, int num_q_heads, double *out) {
  if (!pool_valid(pool) || !q || !page_tables || !seq_lens || !out || batch <= 0 ||
      num_q_heads <= 0 || num_q_heads % pool->num_kv_heads != 0 || table_stride <= 0 ||
      (!first_pos) != (!window_lo))
    return ORC_ERR_INVALID;
  for (int b = 0; b < batch; ++b) {
    if (seq_lens[b] <= 0 || (int64_t)seq_lens[b] > (int64_t)table_stride * pool->page_size)
      return ORC_ERR_INVALID;
    if (first_key(first_pos, window_lo, b, seq_lens[b]) >= seq_lens[b]) return ORC_ERR_INVALID;
    for (int j = 0; j < (seq_lens[b] + pool->page_size - 1) / pool->page_size; ++j) {
      const int32_t page = page_tables[(size_t)b * table_stride + j];
      if (page < 0 || page >= pool->num_pages) return ORC_ERR_BAD_PAGE;
    }
  }
  return ORC_OK;
}

/* Direct decode of T query tokens per row: token t of row b (query row
 * (b*T + t)) sits at key position len - T + t and attends the keys up to and
 * including its own position, from the window bound if any. */
/* softmax(scale q.k_i) v_i over keys [i0, i1) of (row b, kv head g), into dst[dv].
 * s is caller scratch of at least i1 - i0 doubles. */
static void attend_paged(const orc_pool *pool, const double *qd, const int32_t *page_tables,
                         int table_stride, int b, int g, int i0, int i1, double scale, double *s,
                         double *dst) {
  const int dk = pool->head_dim_k, dv = pool->head_dim_v, kw = key_width(pool);
  /* s_i = scale * q . k_i over the attended keys */
  double mx = -INFINITY;
  for (int i = i0; i < i1; ++i) {
    const size_t kr = paged_row(pool, dk, page_tables, table_stride, b, g, i);
    const size_t vr = paged_row(pool, dv, page_tables, table_stride, b, g, i);
    double acc = 0.0;
    for (int d = 0; d < kw; ++d) acc += qd[d] * key_elem(pool, kr, vr, d);
    s[i - i0] = scale * acc;
    if (s[i - i0] > mx) mx = s[i - i0];
  }
  /* out = sum_i softmax(s)_i v_i */
  double z = 0.0;
  for (int i = i0; i < i1; ++i) {
    s[i - i0] = exp(s[i - i0] - mx);
    z += s[i - i0];
  }
  for (int d = 0; d < dv; ++d) dst[d] = 0.0;
  for (int i = i0; i < i1; ++i) {
    const double w = s[i - i0] / z;
    const size_t vr = paged_row(pool, dv, page_tables, table_stride, b, g, i);
    for (int d = 0; d < dv; ++d) dst[d] += w * load_elem(pool->v, pool->dtype, vr + d);
  }
}

static int decode_direct_tokens(const orc_pool *pool, const void *q, const int32_t *page_tables,
                                int table_stride, const int32_t *seq_lens,
                                const int32_t *first_pos, const int32_t *window_lo, int batch,
                                int num_tokens, int num_q_heads, double scale, double *out) {
  int rc = decode_args_ok(pool, q, page_tables, table_stride, seq_lens, first_pos, window_lo,
                          batch, num_q_heads, out);
  if (rc) return rc;
  if (num_tokens < 1) return ORC_ERR_INVALID;
  for (int b = 0; b < batch; ++b)
    if (seq_lens[b] < num_tokens) return ORC_ERR_INVALID;
  const int dv = pool->head_dim_v, kw = key_width(pool);
  const int G = num_q_heads / pool->num_kv_heads; /* head h reads kv head h / G */
  int rc_all = ORC_OK;
  const int T = num_tokens;
  const int jobs = batch * T * num_q_heads;
#pragma omp parallel for schedule(dynamic, 1)
  for (int job = 0; job < jobs; ++job) {
    const int h = job % num_q_heads, bt = job / num_q_heads, b = bt / T, t = bt % T, g = h / G;
    const int len = seq_lens[b] - T + t + 1; /* keys this token sees */
    const int i0 = first_key(first_pos, window_lo, b, len);
    double *qd = (double *)malloc(sizeof(double) * (size_t)kw);
    double *s = (double *)malloc(sizeof(double) * (size_t)(len - i0 + 1));
    if (!qd || !s) {
#pragma omp critical
      rc_all = ORC_ERR_INVALID;
    } else {
      for (int d = 0; d < kw; ++d) qd[d] = load_elem(q, pool->dtype, ((size_t)bt * num_q_heads + h) * kw + d);
      attend_paged(pool, qd, page_tables, table_stride, b, g, i0, len, scale, s,
                   out + ((size_t)bt * num_q_heads + h) * dv);
    }
    free(qd);
    free(s);
  }
  return rc_all;
}

/* softmax(scale q.k_i) v_i over the n keys listed in keys[] (increasing key
 * indices) of (row b, kv head g), into dst[dv].  s is caller scratch of n doubles. */
static void attend_paged_keys(const orc_pool *pool, const double *qd, const int32_t *page_tables,
                              int table_stride, int b, int g, const int *keys, int n,
                              double scale, double *s, double *dst) {
  const int dk = pool->head_dim_k, dv = pool->head_dim_v, kw = key_width(pool);
  double mx = -INFINITY;
  for (int j = 0; j < n; ++j) {
    const size_t kr = paged_row(pool, dk, page_tables, table_stride, b, g, keys[j]);
    const size_t vr = paged_row(pool, dv, page_tables, table_stride, b, g, keys[j]);
    double acc = 0.0;
    for (int d = 0; d < kw; ++d) acc += qd[d] * key_elem(pool, kr, vr, d);
    s[j] = scale * acc;
    if (s[j] > mx) mx = s[j];
  }
  double z = 0.0;
  for (int j = 0; j < n; ++j) {
    s[j] = exp(s[j] - mx);
    z += s[j];
  }
  for (int d = 0; d < dv; ++d) dst[d] = 0.0;
  for (int j = 0; j < n; ++j) {
    const double w = s[j] / z;
    const size_t vr = paged_row(pool, dv, page_tables, table_stride, b, g, keys[j]);
    for (int d = 0; d < dv; ++d) dst[d] += w * load_elem(pool->v, pool->dtype, vr + d);
  }
}

/* Tree attention over a drafted window: the window's T tokens are the row's
 * last T keys, in an order where every token comes after its ancestors.
 * Token t sees every key before the window and the window tokens j <= t
 * whose bit j is set in tree_mask[b * T + t] (its ancestors and itself). */
int orc_decode_tree_direct(const orc_pool *pool, const void *q, const int32_t *page_tables,
                           int table_stride, const int32_t *seq_lens, const uint64_t *tree_mask,
                           int batch, int num_tokens, int num_q_heads, double scale,
                           double *out) {
  int rc = decode_args_ok(pool, q, page_tables, table_stride, seq_lens, NULL, NULL, batch,
                          num_q_heads, out);
  if (rc) return rc;
  const int T = num_tokens;
  if (!tree_mask || T < 1 || T > 64) return ORC_ERR_INVALID;
  for (int b = 0; b < batch; ++b) {
    if (seq_lens[b] < T) return ORC_ERR_INVALID;
    for (int t = 0; t < T; ++t) {
      const uint64_t m = tree_mask[(size_t)b * T + t];
      const uint64_t later = t == 63 ? 0 : ~((((uint64_t)1) << (t + 1)) - 1);
      /* a token sees itself and none of the tokens after it */
      if (!((m >> t) & 1) || (m & later)) return ORC_ERR_INVALID;
    }
  }
  const int dv = pool->head_dim_v, kw = key_width(pool);
  const int G = num_q_heads / pool->num_kv_heads;
  int rc_all = ORC_OK;
  const int jobs = batch * T * num_q_heads;
#pragma omp parallel for schedule(dynamic, 1)
  for (int job = 0; job < jobs; ++job) {
    const int h = job % num_q_heads, bt = job / num_q_heads, b = bt / T, t = bt % T, g = h / G;
    const int w0 = seq_lens[b] - T; /* the window's first key */
    const uint64_t m = tree_mask[(size_t)bt];
    double *qd = (double *)malloc(sizeof(double) * (size_t)kw);
    double *s = (double *)malloc(sizeof(double) * (size_t)(w0 + t + 1));
    int *keys = (int *)malloc(sizeof(int) * (size_t)(w0 + t + 1));
    if (!qd || !s || !keys) {
#pragma omp critical
      rc_all = ORC_ERR_INVALID;
    } else {
      int n = 0;
      for (int i = 0; i < w0; ++i) keys[n++] = i;
      for (int j = 0; j <= t; ++j)
        if ((m >> j) & 1) keys[n++] = w0 + j;
      for (int d = 0; d < kw; ++d) qd[d] = load_elem(q, pool->dtype, ((size_t)bt * num_q_heads + h) * kw + d);
      attend_paged_keys(pool, qd, page_tables, table_stride, b, g, keys, n, scale, s,
                        out + ((size_t)bt * num_q_heads + h) * dv);
    }
    free(qd);
    free(s);
    free(keys);
  }
  return rc_all;
}

int orc_prefill_direct(const orc_pool *pool, const void *q, const int32_t *cu_q,
                       const int32_t *page_tables, int table_stride, const int32_t *seq_lens,
                       int window, int batch, int num_q_heads, double scale, double *out) {
  int rc = decode_args_ok(pool, q, page_tables, table_stride, seq_lens, NULL, NULL, batch,
                          num_q_heads, out);
  if (rc) return rc;
  if (!cu_q || cu_q[0] != 0 || window < 0) return ORC_ERR_INVALID;
  for (int b = 0; b < batch; ++b) {
    const int T = cu_q[b + 1] - cu_q[b];
    if (T < 0 || T > seq_lens[b]) return ORC_ERR_INVALID;
  }
  const int dv = pool->head_dim_v, kw = key_width(pool);
  const int G = num_q_heads / pool->num_kv_heads;
  const int total = cu_q[batch];
  int rc_all = ORC_OK;
  const int jobs = total * num_q_heads;
#pragma omp parallel for schedule(dynamic, 1)
  for (int job = 0; job < jobs; ++job) {
    const int h = job % num_q_heads, r = job / num_q_heads, g = h / G;
    int b = 0;
    while (cu_q[b + 1] <= r) ++b; /* the row token r belongs to */
    const int T = cu_q[b + 1] - cu_q[b], t = r - cu_q[b];
    const int own = seq_lens[b] - T + t; /* the token's own key index */
    const int i0 = (window > 0 && own - window + 1 > 0) ? own - window + 1 : 0;
    double *qd = (double *)malloc(sizeof(double) * (size_t)kw);
    double *s = (double *)malloc(sizeof(double) * (size_t)(own - i0 + 2));
    if (!qd || !s) {
#pragma omp critical
      rc_all = ORC_ERR_INVALID;
    } else {
      for (int d = 0; d < kw; ++d) qd[d] = load_elem(q, pool->dtype, ((size_t)r * num_q_heads + h) * kw + d);
      attend_paged(pool, qd, page_tables, table_stride, b, g, i0, own + 1, scale, s,
                   out + ((size_t)r * num_q_heads + h) * dv);
    }
    free(qd);
    free(s);
  }
  return rc_all;
}

int orc_decode_direct(const orc_pool *pool, const void *q, const int32_t *page_tables,
                      int table_stride, const int32_t *seq_lens, const int32_t *first_pos,
                      const int32_t *window_lo, int batch, int num_q_heads, double scale,
                      double *out) {
  return decode_direct_tokens(pool, q, page_tables, table_stride, seq_lens, first_pos, window_lo,
                              batch, 1, num_q_heads, scale, out);
}

int orc_decode_multirow_direct(const orc_pool *pool, const void *q, const int32_t *page_tables,
                               int table_stride, const int32_t *seq_lens, int batch,
                               int num_tokens, int num_q_heads, double scale, double *out) {
  return decode_direct_tokens(pool, q, page_tables, table_stride, seq_lens, NULL, NULL, batch,
                              num_tokens, num_q_heads, scale, out);
}

int orc_decode_online(const orc_pool *pool, const void *q, const int32_t *page_tables,
                      int table_stride, const int32_t *seq_lens, const int32_t *first_pos,
                      const int32_t *window_lo, int batch, int num_q_heads, double scale,
                      int chunk_tokens, int num_splits, int group_size, double *out) {
  int rc = decode_args_ok(pool, q, page_tables, table_stride, seq_lens, first_pos, window_lo,
                          batch, num_q_heads, out);
  if (rc) return rc;
  if (chunk_tokens <= 0 || num_splits <= 0 || group_size <= 0) return ORC_ERR_INVALID;
  const int H = pool->num_kv_heads, dk = key_width(pool), dv = pool->head_dim_v;
  const int G = num_q_heads / H;
  int rc_all = ORC_OK;
  const int jobs = batch * H;
#pragma omp parallel for schedule(dynamic, 1)
  for (int job = 0; job < jobs; ++job) {
    const int b = job / H, g = job % H, len = seq_lens[b];
    double *K = (double *)malloc(sizeof(double) * (size_t)len * dk);
    double *V = (double *)malloc(sizeof(double) * (size_t)len * dv);
    double *qd = (double *)malloc(sizeof(double) * (size_t)dk);
    int *bounds = (int *)malloc(sizeof(int) * (size_t)(num_splits + 1));
    int jrc = (K && V && qd && bounds) ? ORC_OK : ORC_ERR_INVALID;
    if (!jrc) jrc = orc_gather(pool, page_tables, table_stride, b, g, len, K, V);
    const int i0 = first_key(first_pos, window_lo, b, len);
    if (!jrc) {
      /* chunks aligned to key 0; partitions of ceil(n_chunks / P) chunks over [i0, len) */
      const int c_lo = i0 / chunk_tokens, c_hi = (len + chunk_tokens - 1) / chunk_tokens;
      const int per = (c_hi - c_lo + num_splits - 1) / num_splits;
      for (int p = 0; p <= num_splits; ++p) {
        int64_t e = (int64_t)(c_lo + (int64_t)p * per) * chunk_tokens;
        if (e < i0) e = i0;
        if (e > len) e = len;
        bounds[p] = (int)e;
      }
    }
    for (int j = 0; j < G && !jrc; ++j) {
      const int h = g * G + j;
      const size_t qoff = ((size_t)b * num_q_heads + h) * dk;
      for (int d = 0; d < dk; ++d) qd[d] = load_elem(q, pool->dtype, qoff + d);
      jrc = orc_attend_partitioned(qd, K, V, dk, dv, bounds, num_splits, group_size, scale,
                                   out + ((size_t)b * num_q_heads + h) * dv);
    }
    if (jrc) {
#pragma omp critical
      rc_all = jrc;
    }
    free(K);
    free(V);
    free(qd);
    free(bounds);
  }
  return rc_all;
}

/* ---- scratch byte contract ([gem] "Candidate ownership and storage") ----- */

int orc_partial_scratch_bytes(int64_t batch, int64_t num_q_heads, int64_t head_dim_v,
                              int64_t num_splits, size_t *maxima, size_t *denominators,
                              size_t *numerators, size_t *total) {
  if (batch <= 0 || num_q_heads <= 0 || head_dim_v <= 0 || num_splits <= 0) return ORC_ERR_INVALID;
  size_t states, nums, two, all;
  if (__builtin_mul_overflow((size_t)batch, (size_t)num_q_heads, &states) ||
      __builtin_mul_overflow(states, (size_t)num_splits, &states) ||
      __builtin_mul_overflow(states, (size_t)head_dim_v, &nums) ||
      __builtin_mul_overflow(nums, (size_t)4, &nums) ||
      __builtin_mul_overflow(states, (size_t)4, &states) ||
      __builtin_mul_overflow(states, (size_t)2, &two) ||
      __builtin_add_overflow(two, nums, &all))
    return ORC_ERR_OVERFLOW;
  if (maxima) *maxima = states;
  if (denominators) *denominators = states;
  if (numerators) *numerators = nums;
  if (total) *total = all;
  return ORC_OK;
}

/* ---- K/V prep (the rows a forward writes into the pages) ------------------
 * pegainfer #1055, Description: the hd512 prep writes the split or the folded
 * row and folds K's norm weight into the query; pegainfer #1057, Description:
 * the preps are elementwise with one RMS reduction per head row.  Reading
 * (the pages give no formula): each head row x of D columns is normalised by
 * its root mean square, x / sqrt(mean(x^2) + eps), multiplied column-wise by
 * the head's norm multiplier (none for V), and its first R columns are rotated
 * as R/2 pairs (i, i + R/2) by the angle whose cosine and sine the caller's
 * tables hold for the token's position.  V is normalised only. */

int orc_prep_head(const double *x, int d, double eps, const double *w, int rot,
                  const double *cos_row, const double *sin_row, double *out) {
  if (!x || !out || d <= 0 || rot < 0 || rot > d || (rot & 1) || !(eps >= 0.0) ||
      (rot > 0 && (!cos_row || !sin_row)))
    return ORC_ERR_INVALID;
  double ss = 0.0;
  for (int i = 0; i < d; ++i) ss += x[i] * x[i];
  const double inv = 1.0 / sqrt(ss / d + eps);
  if (!isfinite(inv)) return ORC_ERR_INVALID;
  for (int i = 0; i < d; ++i) out[i] = x[i] * inv * (w ? w[i] : 1.0);
  const int half = rot / 2;
  for (int i = 0; i < half; ++i) {
    const double a = out[i], b = out[i + half];
    out[i] = a * cos_row[i] - b * sin_row[i];
    out[i + half] = b * cos_row[i] + a * sin_row[i];
  }
  return ORC_OK;
}

int orc_prep_tokens(const void *x, int x_dtype, int64_t x_stride, int q_col, int k_col, int v_col,
                    int n, int num_q_heads, int num_kv_heads, int d, int rot, double eps,
                    const float *w_q, const float *w_k, const float *rope_cos,
                    const float *rope_sin, int max_pos, const int32_t *rope_pos, int folded,
                    double *q_out, double *k_out, double *v_out) {
  if (!x || (x_dtype != ORC_F32 && x_dtype != ORC_BF16) || n < 0 || num_q_heads <= 0 ||
      num_kv_heads <= 0 || d <= 0 || rot < 0 || rot > d || (rot & 1) || max_pos <= 0 ||
      !rope_pos || !q_out || !k_out || !v_out || (rot > 0 && (!rope_cos || !rope_sin)) ||
      q_col < 0 || k_col < 0 || v_col < 0 ||
      (int64_t)q_col + (int64_t)num_q_heads * d > x_stride ||
      (int64_t)k_col + (int64_t)num_kv_heads * d > x_stride ||
      (int64_t)v_col + (int64_t)num_kv_heads * d > x_stride)
    return ORC_ERR_INVALID;
  /* the folded query meets V's columns past R: K's multiplier moves into q
   * there, which presumes K and V come from one projection row */
  if (folded && (k_col != v_col || !w_k)) return ORC_ERR_INVALID;
  double *xin = (double *)malloc(sizeof(double) * (size_t)d);
  double *wd = (double *)malloc(sizeof(double) * (size_t)d);
  double *cs = (double *)malloc(sizeof(double) * (size_t)(rot / 2 + 1));
  double *sn = (double *)malloc(sizeof(double) * (size_t)(rot / 2 + 1));
  int rc = (xin && wd && cs && sn) ? ORC_OK : ORC_ERR_INVALID;
  for (int t = 0; t < n && !rc; ++t) {
    const int pos = rope_pos[t];
    if (pos < 0 || pos >= max_pos) {
      rc = ORC_ERR_INVALID;
      break;
    }
    for (int i = 0; i < rot / 2; ++i) {
      cs[i] = rope_cos[(size_t)pos * (rot / 2) + i];
      sn[i] = rope_sin[(size_t)pos * (rot / 2) + i];
    }
    const size_t base = (size_t)t * (size_t)x_stride;
    for (int h = 0; h < num_q_heads && !rc; ++h) {
      for (int i = 0; i < d; ++i) xin[i] = load_elem(x, x_dtype, base + q_col + (size_t)h * d + i);
      for (int i = 0; i < d; ++i) wd[i] = w_q ? (double)w_q[i] : 1.0;
      double *o = q_out + ((size_t)t * num_q_heads + h) * d;
      rc = orc_prep_head(xin, d, eps, wd, rot, cs, sn, o);
      if (!rc && folded)
        for (int i = rot; i < d; ++i) o[i] *= (double)w_k[i];
    }
    for (int h = 0; h < num_kv_heads && !rc; ++h) {
      for (int i = 0; i < d; ++i) xin[i] = load_elem(x, x_dtype, base + k_col + (size_t)h * d + i);
      for (int i = 0; i < d; ++i) wd[i] = w_k ? (double)w_k[i] : 1.0;
      rc = orc_prep_head(xin, d, eps, wd, rot, cs, sn, k_out + ((size_t)t * num_kv_heads + h) * d);
      if (rc) break;
      for (int i = 0; i < d; ++i) xin[i] = load_elem(x, x_dtype, base + v_col + (size_t)h * d + i);
      rc = orc_prep_head(xin, d, eps, NULL, 0, NULL, NULL, v_out + ((size_t)t * num_kv_heads + h) * d);
    }
  }
  free(xin);
  free(wd);
  free(cs);
  free(sn);
  return rc;
}
