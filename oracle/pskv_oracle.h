/*
 * pskv_oracle.h -- plain fp64 CPU oracle for paged split-KV GQA decode attention.
 *
 * TEST INFRASTRUCTURE ONLY.  This code exists to check the CUDA library; only
 * the tests, the smoke check and the bench's CPU-baseline leg may build, load
 * or call it.  It shares no code, header, table or helper with the CUDA path.
 *
 * Sources (web pages, cited by title and section):
 *  [gem]    "Parked D512 fused split-KV decode design" (gem, docs/research):
 *           intro (online partials, exact rescaling merge, empty states,
 *           fail-closed states and scratch overflow, fp64 direct reference),
 *           "Fixed production shape", "Candidate ownership and storage"
 *           (per-key state update in sequence order, merge identity, scratch
 *           byte contract).
 *  [pg1055] pegainfer #1055 "decode the global family through a generated
 *           split-KV kernel over a folded 640-column pool": Description
 *           (partial over key chunks, merge in two levels).
 *  [pg1057] pegainfer #1057 "serve the sliding family through generated
 *           kernels...": Description (window lower bound; resident pages hold
 *           up to a page more than the window, those keys masked).
 *  [tf1619] TensorFold #1619 "gemma4 CUDA: the global layers' caches in pages
 *           of the core pool...": description "Paged" (K region then V region,
 *           page p = rows [ps*p, ps*(p+1))), "Leasing" (refuse rows past a
 *           slot's pages), "Writes" (rows copied into pages keep their bits).
 *
 * Pool layout (the library's documented layout, restated here): element
 * (page, kv_head, row, d) of a region lives at
 *   ((page * num_kv_heads + kv_head) * page_size + row) * head_dim + d.
 * Key i of table row b is in page tables[b * table_stride + i / page_size],
 * row i % page_size.  Query head h reads kv head h / (Hq / Hkv).
 */
#ifndef PSKV_ORACLE_H
#define PSKV_ORACLE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define ORC_OK 0
#define ORC_ERR_INVALID (-1)
#define ORC_ERR_PAST_PAGES (-2)
#define ORC_ERR_OVERFLOW (-3)
#define ORC_ERR_STATE (-4)
#define ORC_ERR_BAD_PAGE (-5)

#define ORC_F32 0
#define ORC_BF16 1

#define ORC_SPLIT 0
#define ORC_FOLDED 1

/* Geometry of one paged pool (both regions share it).
 * Split pools store whole K rows (head_dim_k == head_dim_v).  Folded pools
 * ([pg1055] Description: K kept only where the rotation touches it, V in
 * full, K's norm weight folded into the query) store only the first
 * head_dim_k < head_dim_v columns of K; the key a query meets is then
 * [k[0:head_dim_k], v[head_dim_k:head_dim_v]] and queries are head_dim_v wide. */
typedef struct orc_pool {
  const void *k;  /* K region */
  const void *v;  /* V region */
  int dtype;      /* ORC_F32 or ORC_BF16 */
  int64_t num_pages;
  int page_size;
  int num_kv_heads;
  int head_dim_k;
  int head_dim_v;
  int format;     /* ORC_SPLIT or ORC_FOLDED */
} orc_pool;

/* Online-softmax state of one query head over a set of keys:
 * m = max score, l = sum exp(s - m), o[dv] = sum exp(s - m) * v.
 * The empty state is (m = -inf, l = 0, o = 0). */
typedef struct orc_state {
  double m;
  double l;
  double *o; /* caller-owned, length dv */
} orc_state;

/* ---- dense (unpaged) attention for one query head ---------------------- */

/* Direct softmax attention over keys [begin, end) of dense K[L][dk], V[L][dv]. */
int orc_attend_direct(const double *q, const double *k, const double *v, int dk, int dv,
                      int begin, int end, double scale, double *out);

/* Online partial over keys [begin, end), one key at a time in sequence order. */
int orc_online_partial(const double *q, const double *k, const double *v, int dk, int dv,
                       int begin, int end, double scale, double *m, double *l, double *o);

/* Exact rescaling merge of two states into (m, l, o); fails closed on invalid
 * states.  Merging with an empty state returns the other state bit for bit. */
int orc_merge(double ma, double la, const double *oa, double mb, double lb, const double *ob,
              int dv, double *m, double *l, double *o);

/* Finalize out = o / l; fails on the empty state. */
int orc_finalize(double m, double l, const double *o, int dv, double *out);

/* Online attention over an explicit partition: keys split at bounds[0..P]
 * (non-decreasing, bounds[0] = begin, bounds[P] = end), one partial per part,
 * partials folded in groups of group_size (level 1), then the group results
 * folded (level 2), then finalized. */
int orc_attend_partitioned(const double *q, const double *k, const double *v, int dk, int dv,
                           const int *bounds, int num_parts, int group_size, double scale,
                           double *out);

/* Single-precision twin of the online path (partials + merge + finalize in
 * float), for the accuracy audit of the gem design's CPU oracle. */
int orc_attend_partitioned_f32(const float *q, const float *k, const float *v, int dk, int dv,
                               const int *bounds, int num_parts, float scale, float *out);

/* ---- paged pool ------------------------------------------------------- */

/* Gather the keys and values of (row b, kv head g) into dense double arrays
 * k_out[len][key width], v_out[len][dv]; the key width is head_dim_k for a
 * split pool and head_dim_v (the assembled key) for a folded one.  Fails on
 * a page id outside the pool or a length past the table. */
int orc_gather(const orc_pool *pool, const int32_t *page_tables, int table_stride, int b, int g,
               int len, double *k_out, double *v_out);

/* Append n rows: row r (k_new/v_new[r][num_kv_heads][head_dim]) goes to table
 * row row_of[r] at position pos_of[r].  All rows are checked first; a
 * position at or past num_pages_of_row[row] * page_size refuses the whole
 * call (ORC_ERR_PAST_PAGES) and nothing is written.  Bytes are copied as is. */
int orc_append_rows(void *k_region, void *v_region, const orc_pool *pool, const void *k_new,
                    const void *v_new, const int32_t *row_of, const int32_t *pos_of, int n,
                    const int32_t *page_tables, int table_stride,
                    const int32_t *num_pages_of_row, int batch);

/* Direct fp64 decode: out[b][h][dv] for every row and query head.
 * first_pos / window_lo may be NULL (no window); key i of row b has position
 * first_pos[b] + i and is attended iff that position >= window_lo[b]. */
int orc_decode_direct(const orc_pool *pool, const void *q, const int32_t *page_tables,
                      int table_stride, const int32_t *seq_lens, const int32_t *first_pos,
                      const int32_t *window_lo, int batch, int num_q_heads, double scale,
                      double *out);

/* Direct fp64 decode of num_tokens query tokens per row (a verify window:
 * the row's last num_tokens key positions are its query tokens; TensorFold
 * #1619 reads such windows and tree-attention rows through the page table).
 * q is [batch][num_tokens][num_q_heads][key width], out the same with head_dim_v;
 * token t of row b sits at key position seq_lens[b] - num_tokens + t and
 * attends keys [0, seq_lens[b] - num_tokens + t] (causal).  num_tokens = 1 is
 * orc_decode_direct without a window. */
int orc_decode_multirow_direct(const orc_pool *pool, const void *q, const int32_t *page_tables,
                               int table_stride, const int32_t *seq_lens, int batch,
                               int num_tokens, int num_q_heads, double scale, double *out);

/* Direct fp64 tree attention over a drafted window read through the page
 * table (TensorFold #1619, description "Reads" and review thread: tree
 * attention rows read their keys from a page table).  The window's
 * num_tokens (1..64) tokens are row b's last keys, ordered so that every
 * token comes after its ancestors; token t sits at key w0 + t, w0 =
 * seq_lens[b] - num_tokens, and attends keys [0, w0) and the keys w0 + j,
 * j <= t, whose bit j is set in tree_mask[b * num_tokens + t].  q and out as
 * in orc_decode_multirow_direct.  Fails closed (ORC_ERR_INVALID) unless every
 * mask has its own bit t set and no bit above t, and every row holds at least
 * num_tokens keys.  A chain (mask of token t = bits 0..t) is
 * orc_decode_multirow_direct. */
int orc_decode_tree_direct(const orc_pool *pool, const void *q, const int32_t *page_tables,
                           int table_stride, const int32_t *seq_lens, const uint64_t *tree_mask,
                           int batch, int num_tokens, int num_q_heads, double scale,
                           double *out);

/* Direct fp64 paged prefill over variable-length chunks (pegainfer #1057,
 * Description: prompt rows read through a windowed varlen kernel with a
 * window lower bound; pegainfer #1055, Description: the generated prefill
 * beside the decode).  Row b's new tokens are its last T_b = cu_q[b+1] -
 * cu_q[b] keys (already in the pool); token t of row b sits at key index
 * own = seq_lens[b] - T_b + t and attends keys [lo, own], lo = own - window + 1
 * clipped at 0 when window > 0, else 0.  q is packed [cu_q[batch]][Hq][key
 * width], out [cu_q[batch]][Hq][head_dim_v]; cu_q[0] = 0, non-decreasing.
 * A one-token chunk is orc_decode_direct with window_lo = own - window + 1. */
int orc_prefill_direct(const orc_pool *pool, const void *q, const int32_t *cu_q,
                       const int32_t *page_tables, int table_stride, const int32_t *seq_lens,
                       int window, int batch, int num_q_heads, double scale, double *out);

/* Online fp64 decode: the attended keys of a row are cut into chunks of
 * chunk_tokens (aligned to key index 0), the chunks into num_splits
 * contiguous partitions of ceil(n_chunks / num_splits) chunks (trailing
 * partitions may be empty), then orc_attend_partitioned. */
int orc_decode_online(const orc_pool *pool, const void *q, const int32_t *page_tables,
                      int table_stride, const int32_t *seq_lens, const int32_t *first_pos,
                      const int32_t *window_lo, int batch, int num_q_heads, double scale,
                      int chunk_tokens, int num_splits, int group_size, double *out);

/* Scratch byte contract of the partial buffer: maxima (B*Hq*P*4 bytes),
 * denominators (same) and numerators (B*Hq*P*Dv*4), each product checked for
 * size_t overflow. */
int orc_partial_scratch_bytes(int64_t batch, int64_t num_q_heads, int64_t head_dim_v,
                              int64_t num_splits, size_t *maxima, size_t *denominators,
                              size_t *numerators, size_t *total);

/* K/V prep of one head row (pegainfer #1055 and #1057, Description: the
 * elementwise preps with one RMS reduction per head row write the rows the
 * pages hold).  out = x / sqrt(mean(x^2) + eps) * w (w NULL: 1), then the
 * first rot columns rotated as pairs (i, i + rot/2):
 *   out[i] = a cos_i - b sin_i,  out[i + rot/2] = b cos_i + a sin_i
 * with (a, b) the normalised pair. */
int orc_prep_head(const double *x, int d, double eps, const double *w, int rot,
                  const double *cos_row, const double *sin_row, double *out);

/* Prep of n tokens from projection rows x ([n][x_stride], bf16 or f32):
 * the q band at column q_col (num_q_heads heads of d), the K band at k_col
 * and the V band at v_col (num_kv_heads heads each).  Token t uses row
 * rope_pos[t] of the cos/sin tables ([max_pos][rot/2]).  Outputs in fp64:
 * q_out [n][Hq][d] (normalised with w_q, rotated), k_out [n][Hkv][d]
 * (w_k, rotated), v_out [n][Hkv][d] (normalised only).  folded: q_out's
 * columns past rot are further multiplied by w_k (K's norm multiplier folded
 * into the query; needs k_col == v_col and w_k). */
int orc_prep_tokens(const void *x, int x_dtype, int64_t x_stride, int q_col, int k_col, int v_col,
                    int n, int num_q_heads, int num_kv_heads, int d, int rot, double eps,
                    const float *w_q, const float *w_k, const float *rope_cos,
                    const float *rope_sin, int max_pos, const int32_t *rope_pos, int folded,
                    double *q_out, double *k_out, double *v_out);

/* Number of OpenMP threads the oracle's parallel loops use (1 without OpenMP). */
int orc_num_threads(void);

#ifdef __cplusplus
}
#endif
#endif
