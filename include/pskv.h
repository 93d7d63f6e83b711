/*
 * pskv.h -- paged split-KV GQA attention for single-token decode on GB300
 * (sm_103a).  C ABI: plain pointers and sizes, no C++ or framework types.
 *
 * The operation (sources are web pages, cited by title and section):
 *   For every table row b and query head h, with G = num_q_heads / num_kv_heads
 *   query heads per KV head and kv head g = h / G,
 *     out[b][h][:] = sum_i softmax_i(scale * q[b][h] . k_i) * v_i
 *   over the keys i of row b, where key i lives in page page_tables[b][i / ps]
 *   at row i % ps ("TensorFold #1619 ... caches in pages of the core pool",
 *   description "Paged"; "Parked D512 fused split-KV decode design" (gem),
 *   "Fixed production shape": exact dense attention, 32 q heads over 4 KV
 *   heads, D = 512).
 *   It is computed split-KV: the keys of a row are cut into partitions, each
 *   produces an online-softmax partial (running max m, sum l, unnormalised
 *   numerator o), and the partials are merged in two levels by the exact
 *   rescaling identity m = max(ma, mb), l = la e^(ma-m) + lb e^(mb-m),
 *   o = oa e^(ma-m) + ob e^(mb-m), then out = o / l (gem design, introduction
 *   and "Candidate ownership and storage"; pegainfer #1055 "decode the global
 *   family through a generated split-KV kernel...", Description).
 *   The windowed variant masks keys below a window lower bound (pegainfer
 *   #1057 "serve the sliding family through generated kernels...",
 *   Description).
 *
 * Conventions for every entry point:
 *   - Device pointers are CUDA device memory of the current device; host
 *     pointers are ordinary host memory.  The caller owns all memory; the
 *     library never allocates device memory and never synchronizes a stream.
 *   - Work is enqueued on `stream` (NULL = the legacy default stream) and is
 *     asynchronous; a return of PSKV_OK means it was enqueued.
 *   - Every call returns a status code (PSKV_OK or a negative PSKV_ERR_*).
 *     Host-visible arguments are checked before anything is enqueued; on an
 *     error nothing is enqueued.  Device-side faults (a bad page id, a length
 *     out of range) never trap: the kernel skips the bad access and ORs a
 *     PSKV_FAULT_* bit into the layout's status word, which the caller reads.
 *   - bf16 data is IEEE bfloat16 (1-8-7), f32 is IEEE binary32.
 */
#ifndef PSKV_H
#define PSKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same types as cudaStream_t / cudaEvent_t, declared without CUDA headers. */
typedef struct CUstream_st *pskv_stream_t;
typedef struct CUevent_st *pskv_event_t;

/* ---- status codes --------------------------------------------------------- */
#define PSKV_OK 0
#define PSKV_ERR_INVALID_ARG (-1)          /* a null pointer, a bad size or value */
#define PSKV_ERR_UNSUPPORTED (-2)          /* a shape or format this build refuses */
#define PSKV_ERR_OVERFLOW (-3)             /* a size product overflows size_t */
#define PSKV_ERR_WORKSPACE_TOO_SMALL (-4)
#define PSKV_ERR_PAST_PAGES (-5)           /* an append position past its row's pages */
#define PSKV_ERR_CUDA (-6)                 /* a CUDA runtime call failed */

/* ---- element types and pool formats ---------------------------------------- */
#define PSKV_DTYPE_F32 0
#define PSKV_DTYPE_BF16 1

#define PSKV_FORMAT_SPLIT 0   /* K and V rows kept whole, one region each */
#define PSKV_FORMAT_FOLDED 1  /* K keeps only its first head_dim_v/4 columns (pegainfer #1055's
                                 640-column row at head dim 512), V in full; bf16 only */

/* ---- device fault bits, ORed into status[0] of the layout's status word ------ */
#define PSKV_FAULT_BAD_PAGE 1u      /* a table entry outside [0, num_pages): that tile or row skipped */
#define PSKV_FAULT_PAST_PAGES 2u    /* an append past its row's pages: that row skipped */
#define PSKV_FAULT_BAD_LENGTH 4u    /* a device length outside [tokens, table_stride * page_size]: clamped */
#define PSKV_FAULT_WAIT_TIMEOUT 8u  /* a bounded wait on a copy expired: the partition was dropped */
#define PSKV_FAULT_EMPTY_ROW 16u    /* a row had no attended key: its output was written as zeros */
#define PSKV_FAULT_BAD_STATE 32u    /* merge input with m = -inf but l != 0, or a NaN m: treated as empty */
#define PSKV_FAULT_BAD_POSITION 64u /* a prep token whose rotation position is outside the table: skipped */
#define PSKV_FAULT_BAD_MASK 128u    /* a tree mask without its own bit or with a later one: later bits ignored */

/* ---- limits ---------------------------------------------------------------- */
#define PSKV_MAX_SPLITS 1024       /* most partitions one decode call may use */
#define PSKV_AUTO_MAX_SPLITS 256   /* most partitions the automatic plan picks */
#define PSKV_MERGE_GROUP 16        /* partials folded per level-1 group of the merge */
#define PSKV_KEY_TILE 16           /* keys per kernel tile; partitions are whole tiles */
#define PSKV_MAX_WINDOW_TOKENS 64  /* query tokens per row of decode_attn_multirow */

/* Description of one paged KV pool.
 *
 * k_pool / v_pool are the pool's K region and V region (TensorFold #1619,
 * "Paged": per layer a K region, then a V region; page p is rows
 * [ps*p, ps*(p+1)) of each).  Within a page the rows are head-major, so
 * element (page, kv_head, row, d) of a region is at
 *     ((page * num_kv_heads + kv_head) * page_size + row) * head_dim + d.
 * This keeps one head's keys of a page contiguous (a design choice of this
 * library; the pages do not fix the order inside a page).
 *
 * status: device int32[4] the caller zeroes; kernels OR PSKV_FAULT_* bits into
 * status[0].  May be NULL (faults are then skipped silently).
 * The format is fixed for the pool's life (pegainfer #1055, Description).
 *
 * Folded format (pegainfer #1055, Description: the folded row holds K only
 * where the rotation touches it, V in full, and the prep folds K's norm
 * weight into the query): the K region keeps the first head_dim_v/4 columns
 * of each key (the rotated quarter), the V region all head_dim_v; queries
 * are head_dim_v wide and the score of key i is
 *     scale * (q[0:Dr] . k_i[0:Dr] + q[Dr:Dv] . v_i[Dr:Dv]),  Dr = Dv/4,
 * i.e. the key is taken to equal V outside the rotated quarter once the norm
 * weight sits in q (this library's reading of the page). */
typedef struct pskv_layout_desc {
  int64_t num_pages;   /* pages in each region, >= 1 */
  int32_t page_size;   /* keys per page: a multiple of PSKV_KEY_TILE */
  int32_t num_kv_heads;
  int32_t head_dim_k;  /* stored K columns: head_dim_v (split) or head_dim_v / 4 (folded) */
  int32_t head_dim_v;  /* 256 or 512 */
  int32_t kv_dtype;    /* PSKV_DTYPE_F32 or PSKV_DTYPE_BF16 (queries use the same type) */
  int32_t format;      /* PSKV_FORMAT_SPLIT or PSKV_FORMAT_FOLDED */
  void *k_pool;        /* device, 16-byte aligned */
  void *v_pool;        /* device, 16-byte aligned */
  int32_t *status;     /* device int32[4] or NULL */
} pskv_layout_desc;

/* Opaque handle: holds a copy of the description (host memory only). */
typedef struct pskv_layout pskv_layout;

/* Optional per-call settings; pass NULL (or zeroed fields) for the defaults.
 *
 * append_k / append_v / append_pages (single-token decode_attn_splitkv and
 * decode_attn_windowed only): the step's new K/V row of each table row, its
 * key seq_lens[b] - 1, is written into its page by the decode itself, as
 * kv_append_rows would write it (same bits, same checks and fault bits:
 * PSKV_FAULT_PAST_PAGES, PSKV_FAULT_BAD_PAGE) -- TensorFold #1619, "Writes"
 * and "Leasing"; pegainfer #1055, Description (the row written where it is
 * produced).  The CTA whose partition holds that key copies the row before it
 * loads the tile, so the call takes two launches (partial kernel, merge)
 * instead of an append launch plus those two.
 *   append_k      device [batch][num_kv_heads][head_dim_k] of the pool's dtype, 16-byte aligned
 *   append_v      device [batch][num_kv_heads][head_dim_v], 16-byte aligned
 *   append_pages  device int32[batch]: pages leased to each row */
typedef struct pskv_decode_opts {
  int32_t merge_group;        /* partials per level-1 merge group, 1..PSKV_MERGE_GROUP; 0 = PSKV_MERGE_GROUP */
  pskv_event_t partial_begin; /* if not NULL, recorded on the stream just before the partial kernel */
  pskv_event_t partial_end;   /* if not NULL, recorded on the stream just after the partial kernel */
  const void *append_k;       /* the step's new K rows, or NULL (no append) */
  const void *append_v;       /* the step's new V rows */
  const int32_t *append_pages; /* pages leased per row */
} pskv_decode_opts;

/* Validate `desc` and make a layout handle.  Touches no device.
 * Errors: INVALID_ARG (null pointers, sizes < 1, misaligned pools,
 * page_size not a multiple of PSKV_KEY_TILE, unknown format), UNSUPPORTED
 * (head_dim_v not 256/512; split with head_dim_k != head_dim_v; folded with
 * head_dim_k != head_dim_v / 4 or an f32 pool). */
int paged_kv_layout_create(const pskv_layout_desc *desc, pskv_layout **out);

/* Free a handle (NULL is ignored).  The pools are the caller's. */
void paged_kv_layout_destroy(pskv_layout *layout);

/* Append n new rows into the pool, bit for bit (TensorFold #1619, "Writes":
 * rows copied into the pages keep the linear cache's bits).
 *   k_new, v_new     device [n][num_kv_heads][head_dim_k] and [n][num_kv_heads][head_dim_v],
 *                    the pool's dtype, 16-byte aligned
 *   row_of, pos_of   device int32[n]: table row and key position of each new row
 *   page_tables      device int32[batch][table_stride]
 *   pages_of_row     device int32[batch]: pages row b holds (its lease)
 *   row_of_host, pos_of_host, pages_of_row_host: optional host copies of the
 *     same arrays (all three or none).  When given they are checked before
 *     launch and a position at or past pages_of_row[row] * page_size refuses
 *     the whole call with PSKV_ERR_PAST_PAGES (TensorFold #1619, "Leasing":
 *     rows past a slot's pages are refused), nothing enqueued.  Without them
 *     the kernel checks each row and skips a bad one, setting
 *     PSKV_FAULT_PAST_PAGES or PSKV_FAULT_BAD_PAGE.
 * (row, pos) pairs must be distinct within one call. */
int kv_append_rows(const pskv_layout *layout, const void *k_new, const void *v_new,
                   const int32_t *row_of, const int32_t *pos_of, int32_t n,
                   const int32_t *page_tables, int32_t table_stride,
                   const int32_t *pages_of_row, int32_t batch,
                   const int32_t *row_of_host, const int32_t *pos_of_host,
                   const int32_t *pages_of_row_host, pskv_stream_t stream);

/* Rotation and normalisation parameters of kv_prep_append. */
typedef struct pskv_prep_desc {
  int32_t rot_dims;       /* leading columns of each head row rotated: even, 0..head_dim */
  float eps;              /* added to the mean square before the square root */
  const float *w_q;       /* device float[head_dim], 16-byte aligned: query norm
                             multiplier, or NULL (1) */
  const float *w_k;       /* device float[head_dim], 16-byte aligned: key norm
                             multiplier, or NULL (1); required for a folded pool */
  const float *rope_cos;  /* device float[max_pos][rot_dims / 2] */
  const float *rope_sin;  /* device float[max_pos][rot_dims / 2] */
  int32_t max_pos;        /* rows of the tables */
} pskv_prep_desc;

/* K/V prep with the page write fused in (pegainfer #1055, Description: the
 * hd512 prep writes the split or the folded row and folds K's norm weight
 * into the query; pegainfer #1057, Description: elementwise preps with one RMS
 * reduction per head row; TensorFold #1619, "Writes" and "Leasing").  For
 * each new token t (n of them) it takes the projection row
 *   x          device bf16 [n][x_stride], 16-byte aligned, x_stride a multiple of 8;
 *              the query band starts at column q_col (num_q_heads head rows of
 *              head_dim), the key band at k_col and the value band at v_col
 *              (num_kv_heads head rows each); columns multiples of 8
 * and computes per head row r of head_dim columns
 *   r' = r / sqrt(mean(r^2) + eps) * w        (w = w_q for q, w_k for K, 1 for V)
 * then, for q and K, turns the first rot_dims columns as pairs (i, i + rot/2):
 *   r''[i] = a cos - b sin,  r''[i + rot/2] = b cos + a sin
 * with (a, b) = (r'[i], r'[i + rot/2]) and cos, sin = table row p, column i,
 * p = first_pos[row_of[t]] + pos_of[t] (first_pos NULL: 0).  K (its first
 * head_dim_k columns: all of them in a split pool, the rotated quarter in a
 * folded one) and V go straight into page slot pos_of[t] of table row
 * row_of[t], as kv_append_rows would place them; the prepared query goes to
 *   q_out      device bf16 [n][num_q_heads][head_dim], 16-byte aligned
 * and, for a folded pool, its columns past rot_dims are further multiplied by
 * w_k, which makes q_out the folded query decode_attn_* expect.  A folded pool
 * needs rot_dims == head_dim_k, k_col == v_col (K and V from one projection)
 * and w_k.  Values are computed in f32 and rounded to nearest even bf16.
 * Checks, the host copies and the device fault bits are those of
 * kv_append_rows, plus PSKV_FAULT_BAD_POSITION for a table row p outside
 * [0, max_pos) (that token is skipped).  bf16 pools only.
 * Errors: INVALID_ARG, UNSUPPORTED, PAST_PAGES (from the host copies), CUDA. */
int kv_prep_append(const pskv_layout *layout, const pskv_prep_desc *prep, const void *x,
                   int64_t x_stride, int32_t q_col, int32_t k_col, int32_t v_col, int32_t n,
                   int32_t num_q_heads, const int32_t *row_of, const int32_t *pos_of,
                   const int32_t *first_pos, const int32_t *page_tables, int32_t table_stride,
                   const int32_t *pages_of_row, int32_t batch, const int32_t *row_of_host,
                   const int32_t *pos_of_host, const int32_t *pages_of_row_host, void *q_out,
                   pskv_stream_t stream);

/* Split-KV decode: one query token per row.
 *   q              device [batch][num_q_heads][head_dim_v], the pool's dtype (for a
 *                  folded pool, the folded query: see pskv_layout_desc)
 *   page_tables    device int32[batch][table_stride]; entries past a row's
 *                  pages are never read
 *   seq_lens_host  host int32[batch]: keys per row, each in [1, table_stride * page_size];
 *                  the plan (split count, grid) is made from these
 *   seq_lens       device int32[batch]: the same lengths, read by the kernels
 *   scale          score scale (e.g. 1/sqrt(head_dim)); no softcap
 *   num_splits     partitions per (row, KV head): 1..PSKV_MAX_SPLITS, or 0 for
 *                  the automatic plan (pskv_plan_splits).  Keys are cut into
 *                  tiles of PSKV_KEY_TILE; partition p of a row takes tiles
 *                  [p*c, (p+1)*c) of its attended tiles, c = ceil(tiles / num_splits);
 *                  trailing partitions may be empty.
 *   workspace      device scratch of at least decode_attn_workspace_bytes(...)
 *                  bytes, 256-byte aligned (NULL is fine with num_splits = 1 on
 *                  a bf16 pool with 1/2/4/8 query heads per KV head: the one
 *                  partition then writes the output itself and no merge runs).
 *                  Otherwise, on return its head holds the partials: float
 *                  m[batch][num_q_heads][P], then (at the next 256-byte
 *                  boundary) float l[...][P], then float
 *                  o[batch][num_q_heads][P][head_dim] (m in units of the scaled
 *                  score; o of a partition with m = -inf is left unwritten).
 *   out            device [batch][num_q_heads][head_dim] of out_dtype
 *                  (PSKV_DTYPE_BF16, round to nearest even, or PSKV_DTYPE_F32)
 * The result is run-to-run deterministic for a fixed split count.
 * Errors: INVALID_ARG, UNSUPPORTED (num_q_heads % num_kv_heads != 0, or a
 * query-group size this build has no kernel for: bf16 takes 1/2/4/8 query heads
 * per KV head (and 16 at head dim 256, split only), f32 takes 1/2/4/8 (16 at
 * head dim 256)), WORKSPACE_TOO_SMALL, CUDA. */
int decode_attn_splitkv(const pskv_layout *layout, const void *q, const int32_t *page_tables,
                        int32_t table_stride, const int32_t *seq_lens_host,
                        const int32_t *seq_lens, int32_t batch, int32_t num_q_heads, float scale,
                        int32_t num_splits, void *workspace, size_t workspace_bytes, void *out,
                        int32_t out_dtype, const pskv_decode_opts *opts, pskv_stream_t stream);

/* Windowed split-KV decode (pegainfer #1057, Description: the resident pages
 * hold up to a page more than the window and those keys are masked).  As
 * decode_attn_splitkv, plus:
 *   first_pos   device int32[batch]: key i of row b has position first_pos[b] + i
 *   window_lo   device int32[batch]: key i is attended iff its position >= window_lo[b]
 * Keys below the bound are neither loaded nor used; partitions cover only the
 * tiles from the one holding the first attended key.  A row whose bound
 * excludes every key gets zeros and PSKV_FAULT_EMPTY_ROW. */
int decode_attn_windowed(const pskv_layout *layout, const void *q, const int32_t *page_tables,
                         int32_t table_stride, const int32_t *seq_lens_host,
                         const int32_t *seq_lens, const int32_t *first_pos,
                         const int32_t *window_lo, int32_t batch, int32_t num_q_heads,
                         float scale, int32_t num_splits, void *workspace,
                         size_t workspace_bytes, void *out, int32_t out_dtype,
                         const pskv_decode_opts *opts, pskv_stream_t stream);

/* Multi-row split-KV decode: num_tokens query tokens per row, the row's last
 * num_tokens keys (a verify window; TensorFold #1619, description "Reads" and
 * the review thread: drafted verify windows and tree-attention rows read
 * their keys through the page table).  Token t of row b sits at key
 * seq_lens[b] - num_tokens + t and attends keys [0, seq_lens[b] - num_tokens + t]
 * (causal inside the window).  As decode_attn_splitkv, except:
 *   q           device [batch][num_tokens][num_q_heads][head_dim_v]
 *   out         device [batch][num_tokens][num_q_heads][head_dim_v] of out_dtype
 *   num_tokens  1..PSKV_MAX_WINDOW_TOKENS.  The window's query columns per KV
 *               head (query heads per KV head x num_tokens) are served 8 per
 *               CTA when they fit in 8, else 16 per CTA, the CTAs of one
 *               partition reading the same keys (the later ones mostly from L2);
 *               on bf16 split pools of head dim 256 or 512, 17 to 64 columns
 *               by the key-major tensor-memory kernel when the longest row
 *               has at least 8,192 keys (128 keys per tile as the MMA's M,
 *               the columns as its N, one CTA per partition streaming the
 *               keys once), and otherwise from 40 columns on by the
 *               query-major tensor-memory kernel, 128 columns per CTA (pair)
 *   seq_lens    every length at least num_tokens
 *   workspace   decode_attn_workspace_bytes(batch * num_tokens, num_q_heads, ...)
 *               bytes; its partials are laid out as for batch * num_tokens rows
 *               (row b * num_tokens + t)
 * bf16 pools with 1/2/4/8 query heads per KV head (any power of two up to
 * 128 when the window has more than 16 columns on a split pool); no key window.
 * num_tokens = 1 gives decode_attn_splitkv's bits.
 * Errors: INVALID_ARG (also a host length below num_tokens), UNSUPPORTED,
 * WORKSPACE_TOO_SMALL, CUDA. */
int decode_attn_multirow(const pskv_layout *layout, const void *q, const int32_t *page_tables,
                         int32_t table_stride, const int32_t *seq_lens_host,
                         const int32_t *seq_lens, int32_t batch, int32_t num_tokens,
                         int32_t num_q_heads, float scale, int32_t num_splits, void *workspace,
                         size_t workspace_bytes, void *out, int32_t out_dtype,
                         const pskv_decode_opts *opts, pskv_stream_t stream);

/* Tree attention over a drafted window read through the page table
 * (TensorFold #1619, description "Reads" and review thread: tree-attention
 * rows read their keys from a page table, next to drafted verify windows).
 * The window's num_tokens drafted tokens are row b's last keys (already
 * appended), ordered so that every token comes after its ancestors.  Token t
 * sits at key w0 + t, w0 = seq_lens[b] - num_tokens, and attends every key
 * before the window and the window keys w0 + j, j <= t, whose bit j is set in
 * its mask.  As decode_attn_multirow, except:
 *   tree_mask   device uint64[batch][num_tokens]: bit j of the mask of token t
 *               of row b marks window token j as visible to it; a valid mask
 *               holds bit t (the token itself) and no bit above t.  A mask
 *               without bit t or with a later bit sets PSKV_FAULT_BAD_MASK
 *               (the later bits are ignored; the token attends what the
 *               remaining bits and the prefix give it)
 * A chain (the mask of token t = bits 0..t) gives decode_attn_multirow's
 * causal window.  Routing as for decode_attn_multirow, except that windows
 * the query-major tensor-memory kernel would take run on the split-KV
 * kernels instead: bf16 (or folded) pools with 1/2/4/8 query heads per KV
 * head, 8 or 16 columns per CTA; on bf16 split pools of head dim 256 or 512,
 * 17 to 64 columns per KV head on the key-major kernel when the longest row
 * has at least 8,192 keys (there also with 16 to 64 query heads per KV head).
 * Errors: INVALID_ARG (also a host length below num_tokens, a null mask),
 * UNSUPPORTED, WORKSPACE_TOO_SMALL, CUDA. */
int decode_attn_tree(const pskv_layout *layout, const void *q, const int32_t *page_tables,
                     int32_t table_stride, const int32_t *seq_lens_host, const int32_t *seq_lens,
                     const uint64_t *tree_mask, int32_t batch, int32_t num_tokens,
                     int32_t num_q_heads, float scale, int32_t num_splits, void *workspace,
                     size_t workspace_bytes, void *out, int32_t out_dtype,
                     const pskv_decode_opts *opts, pskv_stream_t stream);

/* Paged prefill over variable-length chunks (pegainfer #1057, Description:
 * the sliding family's prompt rows read through a windowed varlen kernel
 * with a window lower bound; pegainfer #1055, Description: a generated
 * prefill beside the split-KV decode).  Row b's new tokens are its last
 * T_b = cu_q[b+1] - cu_q[b] keys, already in the pool (kv_append_rows or
 * kv_prep_append); token t sits at key own = seq_lens[b] - T_b + t and
 * attends keys [lo, own], lo = max(0, own - window + 1) when window > 0, else
 * 0.  As decode_attn_multirow, except:
 *   q            device [cu_q[batch]][num_q_heads][head_dim_v] (packed rows)
 *   cu_q_host    host int32[batch + 1]: 0, then non-decreasing, T_b <= seq_lens[b]
 *   cu_q         device int32[batch + 1]: the same offsets, read by the kernels
 *                (rows outside [0, cu_q_host[batch]] are never addressed)
 *   window       keys a token sees, itself included; 0 = all earlier keys
 *   out          device [cu_q[batch]][num_q_heads][head_dim_v] of out_dtype
 *   workspace    decode_attn_workspace_bytes(cu_q[batch], num_q_heads, ...)
 *                bytes; NULL is fine when the plan has one partition (the
 *                automatic plan for long chunks): each CTA then writes its
 *                normalised output directly and no merge runs
 * Split-format bf16 pools of head dim 256 or 512 run on the tensor-memory
 * kernel: a CTA (head dim 512: a cluster of two, each holding half of the
 * head dim) serves 128 query columns (query heads of a KV head x tokens) of
 * one row, for 1, 2, 4, ..., 128 query heads per KV head; its keys are those
 * its tokens see.  Folded bf16 pools run 16 columns per CTA on the split-KV
 * kernels, with 1/2/4/8 query heads per KV head.  Other pools: UNSUPPORTED.
 * Errors: INVALID_ARG, UNSUPPORTED, WORKSPACE_TOO_SMALL, CUDA. */
int prefill_attn_paged(const pskv_layout *layout, const void *q, const int32_t *cu_q_host,
                       const int32_t *cu_q, const int32_t *page_tables, int32_t table_stride,
                       const int32_t *seq_lens_host, const int32_t *seq_lens, int32_t batch,
                       int32_t num_q_heads, int32_t window, float scale, int32_t num_splits,
                       void *workspace, size_t workspace_bytes, void *out, int32_t out_dtype,
                       const pskv_decode_opts *opts, pskv_stream_t stream);

/* Merge P partials per row in two levels by the exact rescaling identity and
 * normalise (gem design, "Candidate ownership and storage"; pegainfer #1055,
 * Description).  One launch: level 1 folds each group of merge_group partials
 * into a group state held in shared memory (never into the inputs), level 2
 * folds a row's group states; both in index order.
 *   m, l         device float[rows][num_splits]; m in units of the scaled score
 *   o            device float[rows][num_splits][head_dim_v], 16-byte aligned
 *   head_dim_v   a multiple of 4
 *   out          device [rows][head_dim_v] of out_dtype
 *   workspace    not used (the group states stay on chip): NULL and 0 are fine
 *   status       device int32[4] fault word or NULL
 * The empty state is (m = -inf, l = 0); its o is never used (it may be
 * uninitialised); merging an empty state changes nothing.  At most 64 groups
 * per row (num_splits <= 64 * merge_group). */
int merge_partials(const float *m, const float *l, const float *o, int32_t rows,
                   int32_t num_splits, int32_t head_dim_v, void *out, int32_t out_dtype,
                   void *workspace, size_t workspace_bytes, int32_t *status,
                   const pskv_decode_opts *opts, pskv_stream_t stream);

/* Scratch bytes a decode call needs for `num_splits` partitions (0 = enough
 * for any automatic plan).  Host-only.  Errors: INVALID_ARG, OVERFLOW. */
int decode_attn_workspace_bytes(int32_t batch, int32_t num_q_heads, int32_t head_dim_v,
                                int32_t num_splits, size_t *bytes);

/* Scratch bytes merge_partials needs: 0 in this build.  Host-only. */
int merge_partials_workspace_bytes(int32_t rows, int32_t num_splits, int32_t head_dim_v,
                                   size_t *bytes);

/* The partial buffer's byte contract (gem design, "Candidate ownership and
 * storage"): maxima batch*num_q_heads*P*4 bytes, denominators the same,
 * numerators batch*num_q_heads*P*head_dim_v*4; every product checked for
 * overflow.  Host-only.  Any output pointer may be NULL. */
int pskv_partial_scratch_bytes(int64_t batch, int64_t num_q_heads, int64_t head_dim_v,
                               int64_t num_splits, size_t *maxima, size_t *denominators,
                               size_t *numerators, size_t *total);

/* The split count the automatic plan picks for these lengths on the current
 * device (num_splits = 0 in a decode call).  It reads the device's SM count
 * and how many CTAs of the serving kernel fit on an SM; no kernel runs.  The
 * plan aims for one wave of CTAs: for one row, floor(slots / num_kv_heads)
 * partitions (slots = SMs x CTAs per SM); for a batch, enough partitions that
 * the longest row's pieces carry about half a slot's fair share of all
 * tiles.  It depends on the lengths only, never on a window bound. */
int pskv_plan_splits(const pskv_layout *layout, int32_t batch, int32_t num_q_heads,
                     const int32_t *seq_lens_host, int32_t *num_splits);

/* The workspace a prefill_attn_paged call needs under its plan.  A sizing
 * helper: the pages give the workspace only as the partial buffer's byte
 * contract (gem design, "Candidate ownership and storage"), which this
 * applies to the plan's split count.  The same
 * arguments' host-visible parts (cu_q_host, seq_lens_host, table_stride,
 * batch, num_q_heads, window, num_splits, 0 = automatic) are checked and
 * planned exactly as the call does, and *bytes receives the bytes its
 * partials take, or 0 when the plan has one partition (each CTA writes its
 * output directly and no workspace is read).  Nothing is enqueued.  The
 * answer depends on the device (its SM count) for automatic plans.
 * Errors: as prefill_attn_paged's host-side checks. */
int prefill_attn_workspace_bytes(const pskv_layout *layout, const int32_t *cu_q_host,
                                 const int32_t *seq_lens_host, int32_t table_stride,
                                 int32_t batch, int32_t num_q_heads, int32_t window,
                                 int32_t num_splits, size_t *bytes);

/* The workspace a decode_attn_multirow (tree = 0) or decode_attn_tree
 * (tree = 1) call needs under its plan, with the same meaning as
 * prefill_attn_workspace_bytes (the same sizing helper, no passage of its
 * own); the two calls can route a window to different kernels, so the flag
 * selects whose plan. */
int decode_attn_multirow_workspace_bytes(const pskv_layout *layout, const int32_t *seq_lens_host,
                                         int32_t table_stride, int32_t batch, int32_t num_tokens,
                                         int32_t num_q_heads, int32_t tree, int32_t num_splits,
                                         size_t *bytes);

/* Bytes of the scratch array that decode_attn_splitkv_static uses (16 MiB). */
#define PSKV_STATIC_SCRATCH_BYTES (16 * 1024 * 1024)

/* decode_attn_splitkv for callers that cannot allocate device memory.
 * No passage of the source pages corresponds to this entry point: it exists
 * for callers that have no way to obtain a workspace (code that must not call
 * cudaMalloc, such as a host callback, a real-time or signal-safe path, or a
 * plugin whose host framework owns every device allocation).
 * It takes the arguments of decode_attn_splitkv except the workspace and the
 * options, and uses instead a scratch array of PSKV_STATIC_SCRATCH_BYTES
 * compiled into the library (held on every GPU that loads the library until
 * the process exits).  It allocates nothing and frees nothing.
 *   - num_splits = 0 picks the automatic plan, lowered to the largest split
 *     count whose workspace (decode_attn_workspace_bytes) fits the array;
 *     an explicit count whose workspace does not fit is refused with
 *     PSKV_ERR_WORKSPACE_TOO_SMALL before anything is enqueued.
 *   - The first call on a device looks up the array's device address (with
 *     that device current) and keeps it; make that first call before any
 *     stream capture on the device.  The kept address is not looked up
 *     again: calling this entry point after cudaDeviceReset on that device
 *     is not supported.
 *   - All calls share the array.  Calls that may run at the same time on the
 *     GPU (other streams or host threads without ordering) overwrite each
 *     other's partials: order them.  Nothing in the array needs clearing;
 *     every call writes what it reads. */
int decode_attn_splitkv_static(const pskv_layout *layout, const void *q,
                               const int32_t *page_tables, int32_t table_stride,
                               const int32_t *seq_lens_host, const int32_t *seq_lens,
                               int32_t batch, int32_t num_q_heads, float scale,
                               int32_t num_splits, void *out, int32_t out_dtype,
                               pskv_stream_t stream);

/* Read the layout's fault word: copies status[0] to *flags after all work
 * already enqueued on `stream`, and optionally clears it for the next calls.
 * This call synchronizes the stream (the only one that does).  A layout made
 * without a status word reads as 0.  Errors: INVALID_ARG, CUDA. */
int pskv_check_flags(const pskv_layout *layout, int32_t clear, pskv_stream_t stream,
                     uint32_t *flags);

/* Static text for a status code. */
const char *pskv_strerror(int status);

/* Text of the last CUDA error seen by this thread (empty if none). */
const char *pskv_last_cuda_error(void);

/* Number of kernels this library has launched in this process. */
uint64_t pskv_kernel_launches(void);

/* Library version: major * 10000 + minor * 100 + patch. */
int pskv_version(void);

#ifdef __cplusplus
}
#endif
#endif /* PSKV_H */
