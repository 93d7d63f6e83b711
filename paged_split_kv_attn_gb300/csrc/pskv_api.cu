// pskv_api.cu -- the C entry points declared in include/pskv.h.
//
// Each entry point checks its host-visible arguments (pskv_plan.cpp), makes
// the plan, carves the caller's workspace and enqueues the kernels on the
// caller's stream.  It never allocates device memory and never synchronizes.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <new>

#include "attn_tc.h"
#include "pskv_internal.cuh"
#include "pskv_plan.h"

using namespace pskv;

namespace {

std::atomic<uint64_t> g_launches{0};
thread_local char g_cuda_error[256] = "";

int cuda_fail(cudaError_t e) {
  std::snprintf(g_cuda_error, sizeof g_cuda_error, "%s: %s", cudaGetErrorName(e),
                cudaGetErrorString(e));
  return PSKV_ERR_CUDA;
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

int sm_count(int *out) {
  static std::atomic<int> cache[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  if (dev >= 0 && dev < 64) {
    const int c = cache[dev].load(std::memory_order_relaxed);
    if (c > 0) {
      *out = c;
      return PSKV_OK;
    }
  }
  int n = 0;
  e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return cuda_fail(e);
  if (dev >= 0 && dev < 64) cache[dev].store(n, std::memory_order_relaxed);
  *out = n;
  return PSKV_OK;
}

// CTA slots of the partial kernel serving (dtype, head_dim, group, format, n-tiles): SMs x CTAs per SM.
int partial_slots(int kv_dtype, int head_dim, int group, int format, int nt, int *slots) {
  int n_sm = 0, rc = sm_count(&n_sm);
  if (rc) return rc;
  const int kernel = pick_kernel(kv_dtype, head_dim, group, format);
  int per = 0;
  cudaError_t e;
  if (kernel == kKernelMma)
    e = occupancy_partial_mma(head_dim, group, format == PSKV_FORMAT_FOLDED, nt, &per);
  else if (kernel == kKernelSimt && kv_dtype == PSKV_DTYPE_F32)
    e = occupancy_partial_simt_f32(head_dim, group, &per);
  else if (kernel == kKernelSimt)
    e = occupancy_partial_simt_bf16(head_dim, group, &per);
  else
    return PSKV_ERR_UNSUPPORTED;
  if (e != cudaSuccess) return cuda_fail(e);
  *slots = n_sm * (per > 0 ? per : 1);
  return PSKV_OK;
}

// The automatic split count of the split-KV partial kernels for a call whose
// rows carry `columns` query columns per KV head (query heads per KV head x
// tokens): one n-tile of 8 columns when they fit, else CTAs of two n-tiles,
// `col_blocks` of them per partition.  decode_attn_* (num_splits = 0) and
// pskv_plan_splits both take their plan from here.
int auto_partial_splits(const pskv_layout_desc &d, int32_t batch, int group, int64_t columns,
                        const int32_t *seq_lens_host, int *P) {
  const int kernel = pick_kernel(d.kv_dtype, d.head_dim_v, group, d.format);
  if (kernel < 0) return PSKV_ERR_UNSUPPORTED;
  const int nt = columns > 8 ? 2 : 1;
  const int64_t col_blocks = (columns + 8 * nt - 1) / (8 * nt);
  int slots = 0;
  const int rc = partial_slots(d.kv_dtype, d.head_dim_v, group, d.format, nt, &slots);
  if (rc) return rc;
  // every partition launches col_blocks CTAs
  const int64_t per = slots / col_blocks;
  const bool bytes_bound = kernel == kKernelMma && d.format != PSKV_FORMAT_FOLDED && columns <= 8;
  *P = plan_splits(per > 0 ? (int)per : 1, batch, d.num_kv_heads, seq_lens_host,
                   bytes_bound ? kFillBytes32 : 32);
  return PSKV_OK;
}

int merge_group_of(const pskv_decode_opts *opts, int *group) {
  int g = (opts && opts->merge_group) ? opts->merge_group : PSKV_MERGE_GROUP;
  if (g < 1 || g > PSKV_MERGE_GROUP) return PSKV_ERR_INVALID_ARG;
  *group = g;
  return PSKV_OK;
}

// Level 2 folds at most this many group results per row.
constexpr int kMaxGroups = 64;

// Verify windows of 17 to 64 query columns per KV head (tokens x query heads
// per KV head) on bf16 split pools run on the key-major tensor-memory kernel
// (keys as the MMA's M, the columns zero-padded to an N of 32 or 64) when the
// longest row has at least kVerifyMinKeys keys: one CTA per (partition, KV
// head, row) streams the keys once.  At 40,002 keys (head dim 512, 8 query
// heads per KV head) 3 / 4 / 5 / 8 tokens took 74 / 75 / 89 / 91 us there
// against ~108 / 108 / 160 / 117 us on the split-KV or query-major kernels, at
// 20,000 keys 51 / 53 / 63 / 65 against 59 / 60 / 85 / 108 us, at 10,602 keys
// 39 / 39 / 48 / 49 against 37 / 38 / 51 / 63 us; below that a CTA's first
// tile (its K tile through two stages, then the softmax, then the values),
// ~10 us, outweighs the few tiles behind it (4,096 keys: 29 / 29 / 34 / 35
// against 23 / 22 / 27 / 32 us).  2 tokens (16 columns) stay on the split-KV
// kernels (61 against 76 us at 40,002 keys).  Otherwise windows of at least
// kTcMinColumns columns run on the query-major kernel, whose blocks of 128
// columns cost the same whatever their real columns (at 40,002 keys ~115 us
// against 109 / 160 us for 4 / 6 tokens on the split-KV kernels).
#ifndef PSKV_VERIFY_MIN_COLUMNS
#define PSKV_VERIFY_MIN_COLUMNS 17  // compile-time tuning knob (65 routes no window there)
#endif
constexpr int64_t kVerifyMinColumns = PSKV_VERIFY_MIN_COLUMNS;
constexpr int64_t kVerifyMaxColumns = 64;
constexpr int64_t kVerifyMinKeys = 8192;
constexpr int64_t kTcMinColumns = 40;

// The query side of a call: a uniform number of tokens per row (single-token
// decode, verify windows), or variable-length chunks given by row offsets
// (prefill), optionally with a per-token window.
struct QuerySpec {
  int tokens = 1;
  const int32_t *cu_q_host = nullptr;  // [B + 1] host copy of the offsets, or null
  const int32_t *cu_q = nullptr;       // [B + 1] device offsets
  int window = 0;
  const uint64_t *tree_mask = nullptr;  // [B][tokens] ancestor masks of a drafted tree, or null
  bool tree_plan = false;               // plan a drafted tree without its masks (size queries)
};

// Checks, plans and enqueues one call.  With `plan_bytes` set it only checks
// the host-visible arguments and plans: *plan_bytes = the workspace the plan
// needs (0 when one partition writes the output directly); device pointers
// are not required and nothing is enqueued.
int decode_common(const pskv_layout *layout, const void *q, const int32_t *page_tables,
                  int32_t table_stride, const int32_t *seq_lens_host, const int32_t *seq_lens,
                  const int32_t *first_pos, const int32_t *window_lo, bool windowed,
                  int32_t batch, const QuerySpec &qs, int32_t num_q_heads, float scale,
                  int32_t num_splits, void *workspace, size_t workspace_bytes, void *out,
                  int32_t out_dtype, const pskv_decode_opts *opts, pskv_stream_t stream,
                  size_t *plan_bytes = nullptr) {
  if (!layout || !seq_lens_host) return PSKV_ERR_INVALID_ARG;
  if (!plan_bytes && (!q || !page_tables || !seq_lens || !out)) return PSKV_ERR_INVALID_ARG;
  if (windowed && !plan_bytes && (!first_pos || !window_lo)) return PSKV_ERR_INVALID_ARG;
  if (batch < 1 || batch > 65535 || num_q_heads < 1 || table_stride < 1) return PSKV_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return PSKV_ERR_INVALID_ARG;
  if (num_splits < 0 || num_splits > PSKV_MAX_SPLITS) return PSKV_ERR_INVALID_ARG;
  if (out_dtype != PSKV_DTYPE_F32 && out_dtype != PSKV_DTYPE_BF16) return PSKV_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(workspace, 16) || !aligned(out, 16)) return PSKV_ERR_INVALID_ARG;
  const pskv_layout_desc &d = layout->d;
  if (num_q_heads % d.num_kv_heads != 0) return PSKV_ERR_UNSUPPORTED;
  if (d.num_kv_heads > 65535) return PSKV_ERR_UNSUPPORTED;
  const int group = num_q_heads / d.num_kv_heads;
  const int kernel = pick_kernel(d.kv_dtype, d.head_dim_v, group, d.format);
  const bool folded = d.format == PSKV_FORMAT_FOLDED;
  const bool varlen = qs.cu_q_host != nullptr;
  if (varlen && !qs.cu_q && !plan_bytes) return PSKV_ERR_INVALID_ARG;
  // Prefill of bf16 split pools at head dim 256 or 512 runs on the
  // query-major tensor-memory kernel: blocks of 128 query columns (any
  // power-of-two group up to 128 query heads per KV head), one CTA (head dim
  // 512: a CTA pair) per block and partition; so do verify windows of at
  // least kTcMinColumns query columns per KV head that the key-major kernel
  // does not take.
  const bool tc_pools = !folded && d.kv_dtype == PSKV_DTYPE_BF16 &&
                        d.head_dim_k == d.head_dim_v &&
                        (d.head_dim_v == 256 || d.head_dim_v == 512) && group <= 128 &&
                        (group & (group - 1)) == 0 && aligned(d.k_pool, 16) &&
                        aligned(d.v_pool, 16) &&
                        (int64_t)d.num_pages * d.num_kv_heads * d.page_size <= INT32_MAX;
  const int64_t window_cols = (int64_t)qs.tokens * group;
  int64_t longest = 0;  // the host lengths (checked below); the routing only reads them
  for (int32_t b = 0; b < batch; ++b)
    longest = seq_lens_host[b] > longest ? seq_lens_host[b] : longest;
  const bool tree = qs.tree_mask != nullptr || qs.tree_plan;
  if (tree && (varlen || windowed)) return PSKV_ERR_INVALID_ARG;
  // drafted trees run on the split-KV kernels and the key-major kernel (both
  // take the tokens' masks), never on the query-major one
  const bool verify_tc = tc_pools && !varlen && !windowed && qs.tokens >= 2 &&
                         window_cols >= kVerifyMinColumns && window_cols <= kVerifyMaxColumns &&
                         longest >= kVerifyMinKeys;
  const bool many_rows = varlen || (!windowed && qs.tokens >= 2 && window_cols >= kTcMinColumns);
  const bool tc_path = !tree && many_rows && tc_pools && !verify_tc;
  // the tensor-core split-KV consumer is the other kernel that takes tree masks
  if (tree && !verify_tc && kernel != kKernelMma) return PSKV_ERR_UNSUPPORTED;
  if (kernel < 0 && !tc_path && !verify_tc) return PSKV_ERR_UNSUPPORTED;
  const bool append = opts && opts->append_k;
  if (append) {
    if (!opts->append_v || !opts->append_pages) return PSKV_ERR_INVALID_ARG;
    if (!aligned(opts->append_k, 16) || !aligned(opts->append_v, 16)) return PSKV_ERR_INVALID_ARG;
    if (varlen || qs.tokens != 1) return PSKV_ERR_UNSUPPORTED;  // single-token decode only
  }
  if (qs.window < 0) return PSKV_ERR_INVALID_ARG;
  int rc = check_lengths(layout, batch, table_stride, seq_lens_host, varlen ? 1 : qs.tokens);
  if (rc) return rc;
  // query rows and the longest chunk
  int64_t rows = 0, max_t = 0;
  if (varlen) {
    if (qs.cu_q_host[0] != 0) return PSKV_ERR_INVALID_ARG;
    for (int32_t b = 0; b < batch; ++b) {
      const int64_t t = (int64_t)qs.cu_q_host[b + 1] - qs.cu_q_host[b];
      if (t < 0 || t > seq_lens_host[b]) return PSKV_ERR_INVALID_ARG;
      max_t = t > max_t ? t : max_t;
    }
    rows = qs.cu_q_host[batch];
    if (rows < 1) return PSKV_ERR_INVALID_ARG;
  } else {
    if (qs.tokens < 1 || qs.tokens > PSKV_MAX_WINDOW_TOKENS) return PSKV_ERR_INVALID_ARG;
    max_t = qs.tokens;
    rows = (int64_t)batch * qs.tokens;
  }
  // Query columns per KV head (heads x tokens): one n-tile of 8 when they fit,
  // else blocks of two n-tiles, one CTA per block (several tokens only on the
  // tensor-core family).
  if ((max_t > 1 || varlen) && !tc_path && !verify_tc && (kernel != kKernelMma || windowed))
    return PSKV_ERR_UNSUPPORTED;
  const int64_t columns = group * max_t;
  const int nt = columns > 8 ? 2 : 1;
  const int64_t col_blocks = (columns + 8 * nt - 1) / (8 * nt);
  if (rows * num_q_heads > INT32_MAX || col_blocks * PSKV_MAX_SPLITS > INT32_MAX)
    return PSKV_ERR_INVALID_ARG;
  int mgroup = 0;
  if ((rc = merge_group_of(opts, &mgroup))) return rc;

  const int64_t tc_qblocks = (columns + 127) / 128;
  if (tc_path && tc_qblocks * PSKV_MAX_SPLITS > INT32_MAX) return PSKV_ERR_INVALID_ARG;
  int P = num_splits;
  if (P == 0 && verify_tc) {
    int n_sm = 0;
    if ((rc = sm_count(&n_sm))) return rc;
    int64_t max_len = 1;
    for (int32_t b = 0; b < batch; ++b) max_len = seq_lens_host[b] > max_len ? seq_lens_host[b] : max_len;
    P = plan_verify_splits((int64_t)d.num_kv_heads * batch, n_sm, (max_len + 127) / 128);
  } else if (P == 0 && tc_path) {
    int n_sm = 0;
    if ((rc = sm_count(&n_sm))) return rc;
    int64_t max_len = 1;
    for (int32_t b = 0; b < batch; ++b) max_len = seq_lens_host[b] > max_len ? seq_lens_host[b] : max_len;
    P = plan_tc_splits(tc_qblocks * d.num_kv_heads * batch, d.head_dim_v == 512 ? n_sm / 2 : n_sm,
                       (max_len + 63) / 64);
  } else if (P == 0) {
    if ((rc = auto_partial_splits(d, batch, group, columns, seq_lens_host, &P))) return rc;
  }
  // one partition on the tensor-core kernels: the partial is the output
  const bool direct = P == 1 && (kernel == kKernelMma || tc_path || verify_tc);
  WorkspacePlan w;
  if ((rc = plan_workspace(rows, num_q_heads, d.head_dim_v, P, mgroup, &w))) return rc;
  if (w.groups > kMaxGroups) return PSKV_ERR_INVALID_ARG;
  if (plan_bytes) {
    *plan_bytes = direct ? 0 : w.total;
    return PSKV_OK;
  }
  if (!direct && (!workspace || workspace_bytes < w.total)) return PSKV_ERR_WORKSPACE_TOO_SMALL;

  char *ws = static_cast<char *>(workspace);
  PartialArgs a;
  a.q = q;
  a.k_pool = d.k_pool;
  a.v_pool = d.v_pool;
  a.page_tables = page_tables;
  a.seq_lens = seq_lens;
  a.first_pos = windowed ? first_pos : nullptr;
  a.window_lo = windowed ? window_lo : nullptr;
  a.status = d.status;
  a.ws_m = direct ? nullptr : reinterpret_cast<float *>(ws + w.m_off);
  a.ws_l = direct ? nullptr : reinterpret_cast<float *>(ws + w.l_off);
  a.ws_o = direct ? nullptr : reinterpret_cast<float *>(ws + w.o_off);
  a.num_pages = d.num_pages;
  a.table_stride = table_stride;
  a.page_size = d.page_size;
  a.num_kv_heads = d.num_kv_heads;
  a.num_q_heads = num_q_heads;
  a.num_splits = P;
  a.num_tokens = varlen ? 0 : qs.tokens;
  a.col_blocks = (int)col_blocks;
  a.scale_log2 = scale * kLog2e;
  a.cu_q = varlen ? qs.cu_q : nullptr;
  a.total_rows = (int)rows;
  a.window = qs.window;
  a.out = out;
  a.out_dtype = out_dtype;
  a.direct = direct ? 1 : 0;
  a.append_k = append ? opts->append_k : nullptr;
  a.append_v = append ? opts->append_v : nullptr;
  a.append_pages = append ? opts->append_pages : nullptr;
  a.k_row_bytes = layout->k_row_bytes;
  a.v_row_bytes = layout->v_row_bytes;
  a.tree_mask = reinterpret_cast<const unsigned long long *>(qs.tree_mask);
  for (int i = 0; i < kLenHints; ++i)
    a.len_hint[i] = (i < batch && !varlen && !windowed && !tree) ? seq_lens_host[i] : -1;

  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const dim3 grid((unsigned)(P * col_blocks), d.num_kv_heads, batch);
  cudaError_t e;
  if (opts && opts->partial_begin) {
    e = cudaEventRecord(reinterpret_cast<cudaEvent_t>(opts->partial_begin), s);
    if (e != cudaSuccess) return cuda_fail(e);
  }
  if (tc_path || verify_tc) {
    TcArgs t;
    t.q = q;
    t.page_tables = page_tables;
    t.seq_lens = seq_lens;
    t.cu_q = varlen ? qs.cu_q : nullptr;
    t.num_tokens = varlen ? 0 : qs.tokens;
    t.status = d.status;
    t.ws_m = a.ws_m;
    t.ws_l = a.ws_l;
    t.ws_o = a.ws_o;
    t.out = out;
    t.out_dtype = out_dtype;
    t.direct = direct ? 1 : 0;
    t.num_pages = d.num_pages;
    t.table_stride = table_stride;
    t.page_size = d.page_size;
    t.num_kv_heads = d.num_kv_heads;
    t.num_q_heads = num_q_heads;
    t.group_shift = __builtin_ctz((unsigned)group);
    t.num_splits = P;
    t.qblocks = verify_tc ? 1 : (int)tc_qblocks;
    t.total_rows = (int)rows;
    t.window = qs.window;
    t.box_rows = d.page_size % 64 == 0 ? 64 : 16;
    t.scale_log2 = scale * kLog2e;
    t.tree_mask = verify_tc ? reinterpret_cast<const unsigned long long *>(qs.tree_mask) : nullptr;
    if (verify_tc)
      e = launch_attn_verify(t, d.k_pool, d.v_pool, d.head_dim_v,
                             dim3((unsigned)P, d.num_kv_heads, batch), s);
    else
      e = launch_attn_tc(t, d.k_pool, d.v_pool, d.head_dim_v,
                         dim3((unsigned)(tc_qblocks * P), d.num_kv_heads, batch), s);
  } else if (kernel == kKernelMma)
    e = launch_partial_mma(a, d.head_dim_v, group, folded, nt, grid, s);
  else if (d.kv_dtype == PSKV_DTYPE_F32)
    e = launch_partial_simt_f32(a, d.head_dim_v, group, grid, s);
  else
    e = launch_partial_simt_bf16(a, d.head_dim_v, group, grid, s);
  if (e != cudaSuccess) return cuda_fail(e);
  g_launches.fetch_add(1, std::memory_order_relaxed);
  if (opts && opts->partial_end) {
    e = cudaEventRecord(reinterpret_cast<cudaEvent_t>(opts->partial_end), s);
    if (e != cudaSuccess) return cuda_fail(e);
  }
  if (direct) return PSKV_OK;

  MergeArgs m;
  m.m = a.ws_m;
  m.l = a.ws_l;
  m.o = a.ws_o;
  m.rows = (int)(rows * num_q_heads);
  m.count = P;
  m.dv = d.head_dim_v;
  m.group = mgroup;
  m.out = out;
  m.out_dtype = out_dtype;
  m.status = d.status;
  int launched = 0;
  e = launch_merge(m, s, &launched);
  g_launches.fetch_add((uint64_t)launched, std::memory_order_relaxed);
  if (e != cudaSuccess) return cuda_fail(e);
  return PSKV_OK;
}

}  // namespace

extern "C" {

int paged_kv_layout_create(const pskv_layout_desc *desc, pskv_layout **out) {
  if (!out) return PSKV_ERR_INVALID_ARG;
  *out = nullptr;
  const int rc = check_layout_desc(desc);
  if (rc) return rc;
  pskv_layout *l = new (std::nothrow) pskv_layout;
  if (!l) return PSKV_ERR_INVALID_ARG;
  l->d = *desc;
  l->elem_size = desc->kv_dtype == PSKV_DTYPE_BF16 ? 2 : 4;
  l->k_row_bytes = desc->head_dim_k * l->elem_size;
  l->v_row_bytes = desc->head_dim_v * l->elem_size;
  *out = l;
  return PSKV_OK;
}

void paged_kv_layout_destroy(pskv_layout *layout) { delete layout; }

int kv_append_rows(const pskv_layout *layout, const void *k_new, const void *v_new,
                   const int32_t *row_of, const int32_t *pos_of, int32_t n,
                   const int32_t *page_tables, int32_t table_stride,
                   const int32_t *pages_of_row, int32_t batch, const int32_t *row_of_host,
                   const int32_t *pos_of_host, const int32_t *pages_of_row_host,
                   pskv_stream_t stream) {
  if (!layout || n < 0 || batch < 1 || table_stride < 1) return PSKV_ERR_INVALID_ARG;
  if (n == 0) return PSKV_OK;
  if (!k_new || !v_new || !row_of || !pos_of || !page_tables || !pages_of_row)
    return PSKV_ERR_INVALID_ARG;
  if (!aligned(k_new, 16) || !aligned(v_new, 16)) return PSKV_ERR_INVALID_ARG;
  const int hosts = (row_of_host != nullptr) + (pos_of_host != nullptr) +
                    (pages_of_row_host != nullptr);
  if (hosts != 0 && hosts != 3) return PSKV_ERR_INVALID_ARG;
  if (hosts == 3) {
    const int rc = check_append_host(layout, n, table_stride, batch, row_of_host, pos_of_host,
                                     pages_of_row_host);
    if (rc) return rc;
  }
  AppendArgs a;
  a.k_new = k_new;
  a.v_new = v_new;
  a.row_of = row_of;
  a.pos_of = pos_of;
  a.n = n;
  a.page_tables = page_tables;
  a.table_stride = table_stride;
  a.pages_of_row = pages_of_row;
  a.batch = batch;
  a.k_pool = layout->d.k_pool;
  a.v_pool = layout->d.v_pool;
  a.num_pages = layout->d.num_pages;
  a.page_size = layout->d.page_size;
  a.num_kv_heads = layout->d.num_kv_heads;
  a.k_row_bytes = layout->k_row_bytes;
  a.v_row_bytes = layout->v_row_bytes;
  a.status = layout->d.status;
  const cudaError_t e = launch_append(a, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e);
  g_launches.fetch_add(1, std::memory_order_relaxed);
  return PSKV_OK;
}

int kv_prep_append(const pskv_layout *layout, const pskv_prep_desc *prep, const void *x,
                   int64_t x_stride, int32_t q_col, int32_t k_col, int32_t v_col, int32_t n,
                   int32_t num_q_heads, const int32_t *row_of, const int32_t *pos_of,
                   const int32_t *first_pos, const int32_t *page_tables, int32_t table_stride,
                   const int32_t *pages_of_row, int32_t batch, const int32_t *row_of_host,
                   const int32_t *pos_of_host, const int32_t *pages_of_row_host, void *q_out,
                   pskv_stream_t stream) {
  if (!layout || !prep || n < 0 || batch < 1 || table_stride < 1 || num_q_heads < 1)
    return PSKV_ERR_INVALID_ARG;
  const pskv_layout_desc &d = layout->d;
  if (d.kv_dtype != PSKV_DTYPE_BF16) return PSKV_ERR_UNSUPPORTED;
  if (num_q_heads % d.num_kv_heads != 0) return PSKV_ERR_UNSUPPORTED;
  const int hd = d.head_dim_v, rot = prep->rot_dims;
  const bool folded = d.format == PSKV_FORMAT_FOLDED;
  if (rot < 0 || rot > hd || (rot & 1) || !(prep->eps >= 0.f) || !std::isfinite(prep->eps))
    return PSKV_ERR_INVALID_ARG;
  if (rot > 0 && (!prep->rope_cos || !prep->rope_sin || prep->max_pos < 1))
    return PSKV_ERR_INVALID_ARG;
  if (folded && (rot != d.head_dim_k || k_col != v_col || !prep->w_k)) return PSKV_ERR_UNSUPPORTED;
  if (x_stride < 8 || x_stride % 8 != 0 || q_col < 0 || k_col < 0 || v_col < 0 || q_col % 8 ||
      k_col % 8 || v_col % 8 || (int64_t)q_col + (int64_t)num_q_heads * hd > x_stride ||
      (int64_t)k_col + (int64_t)d.num_kv_heads * hd > x_stride ||
      (int64_t)v_col + (int64_t)d.num_kv_heads * hd > x_stride)
    return PSKV_ERR_INVALID_ARG;
  if (n == 0) return PSKV_OK;
  if (!x || !row_of || !pos_of || !page_tables || !pages_of_row || !q_out)
    return PSKV_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(q_out, 16) || !aligned(prep->w_q, 16) ||
      !aligned(prep->w_k, 16))
    return PSKV_ERR_INVALID_ARG;
  const int hosts = (row_of_host != nullptr) + (pos_of_host != nullptr) +
                    (pages_of_row_host != nullptr);
  if (hosts != 0 && hosts != 3) return PSKV_ERR_INVALID_ARG;
  if (hosts == 3) {
    const int rc = check_append_host(layout, n, table_stride, batch, row_of_host, pos_of_host,
                                     pages_of_row_host);
    if (rc) return rc;
  }
  PrepArgs a;
  a.x = x;
  a.x_stride = x_stride;
  a.q_col = q_col;
  a.k_col = k_col;
  a.v_col = v_col;
  a.n = n;
  a.num_q_heads = num_q_heads;
  a.num_kv_heads = d.num_kv_heads;
  a.d = hd;
  a.rot = rot;
  a.eps = prep->eps;
  a.w_q = prep->w_q;
  a.w_k = prep->w_k;
  a.rope_cos = prep->rope_cos;
  a.rope_sin = prep->rope_sin;
  a.max_pos = rot > 0 ? prep->max_pos : 0x7fffffff;
  a.row_of = row_of;
  a.pos_of = pos_of;
  a.first_pos = first_pos;
  a.page_tables = page_tables;
  a.table_stride = table_stride;
  a.pages_of_row = pages_of_row;
  a.batch = batch;
  a.k_pool = d.k_pool;
  a.v_pool = d.v_pool;
  a.num_pages = d.num_pages;
  a.page_size = d.page_size;
  a.k_cols = d.head_dim_k;
  a.folded = folded ? 1 : 0;
  a.q_out = q_out;
  a.status = d.status;
  const cudaError_t e = launch_prep(a, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e);
  g_launches.fetch_add(1, std::memory_order_relaxed);
  return PSKV_OK;
}

int decode_attn_splitkv(const pskv_layout *layout, const void *q, const int32_t *page_tables,
                        int32_t table_stride, const int32_t *seq_lens_host,
                        const int32_t *seq_lens, int32_t batch, int32_t num_q_heads, float scale,
                        int32_t num_splits, void *workspace, size_t workspace_bytes, void *out,
                        int32_t out_dtype, const pskv_decode_opts *opts, pskv_stream_t stream) {
  return decode_common(layout, q, page_tables, table_stride, seq_lens_host, seq_lens, nullptr,
                       nullptr, false, batch, QuerySpec{}, num_q_heads, scale, num_splits,
                       workspace, workspace_bytes, out, out_dtype, opts, stream);
}

int decode_attn_windowed(const pskv_layout *layout, const void *q, const int32_t *page_tables,
                         int32_t table_stride, const int32_t *seq_lens_host,
                         const int32_t *seq_lens, const int32_t *first_pos,
                         const int32_t *window_lo, int32_t batch, int32_t num_q_heads,
                         float scale, int32_t num_splits, void *workspace,
                         size_t workspace_bytes, void *out, int32_t out_dtype,
                         const pskv_decode_opts *opts, pskv_stream_t stream) {
  return decode_common(layout, q, page_tables, table_stride, seq_lens_host, seq_lens, first_pos,
                       window_lo, true, batch, QuerySpec{}, num_q_heads, scale, num_splits,
                       workspace, workspace_bytes, out, out_dtype, opts, stream);
}

int decode_attn_multirow(const pskv_layout *layout, const void *q, const int32_t *page_tables,
                         int32_t table_stride, const int32_t *seq_lens_host,
                         const int32_t *seq_lens, int32_t batch, int32_t num_tokens,
                         int32_t num_q_heads, float scale, int32_t num_splits, void *workspace,
                         size_t workspace_bytes, void *out, int32_t out_dtype,
                         const pskv_decode_opts *opts, pskv_stream_t stream) {
  QuerySpec qs;
  qs.tokens = num_tokens;
  return decode_common(layout, q, page_tables, table_stride, seq_lens_host, seq_lens, nullptr,
                       nullptr, false, batch, qs, num_q_heads, scale, num_splits, workspace,
                       workspace_bytes, out, out_dtype, opts, stream);
}

int decode_attn_tree(const pskv_layout *layout, const void *q, const int32_t *page_tables,
                     int32_t table_stride, const int32_t *seq_lens_host, const int32_t *seq_lens,
                     const uint64_t *tree_mask, int32_t batch, int32_t num_tokens,
                     int32_t num_q_heads, float scale, int32_t num_splits, void *workspace,
                     size_t workspace_bytes, void *out, int32_t out_dtype,
                     const pskv_decode_opts *opts, pskv_stream_t stream) {
  if (!tree_mask || (reinterpret_cast<uintptr_t>(tree_mask) & 7u)) return PSKV_ERR_INVALID_ARG;
  QuerySpec qs;
  qs.tokens = num_tokens;
  qs.tree_mask = tree_mask;
  return decode_common(layout, q, page_tables, table_stride, seq_lens_host, seq_lens, nullptr,
                       nullptr, false, batch, qs, num_q_heads, scale, num_splits, workspace,
                       workspace_bytes, out, out_dtype, opts, stream);
}

int prefill_attn_paged(const pskv_layout *layout, const void *q, const int32_t *cu_q_host,
                       const int32_t *cu_q, const int32_t *page_tables, int32_t table_stride,
                       const int32_t *seq_lens_host, const int32_t *seq_lens, int32_t batch,
                       int32_t num_q_heads, int32_t window, float scale, int32_t num_splits,
                       void *workspace, size_t workspace_bytes, void *out, int32_t out_dtype,
                       const pskv_decode_opts *opts, pskv_stream_t stream) {
  if (!cu_q_host || !cu_q) return PSKV_ERR_INVALID_ARG;
  QuerySpec qs;
  qs.cu_q_host = cu_q_host;
  qs.cu_q = cu_q;
  qs.window = window;
  return decode_common(layout, q, page_tables, table_stride, seq_lens_host, seq_lens, nullptr,
                       nullptr, false, batch, qs, num_q_heads, scale, num_splits, workspace,
                       workspace_bytes, out, out_dtype, opts, stream);
}

int prefill_attn_workspace_bytes(const pskv_layout *layout, const int32_t *cu_q_host,
                                 const int32_t *seq_lens_host, int32_t table_stride,
                                 int32_t batch, int32_t num_q_heads, int32_t window,
                                 int32_t num_splits, size_t *bytes) {
  if (!bytes || !cu_q_host) return PSKV_ERR_INVALID_ARG;
  QuerySpec qs;
  qs.cu_q_host = cu_q_host;
  qs.window = window;
  return decode_common(layout, nullptr, nullptr, table_stride, seq_lens_host, nullptr, nullptr,
                       nullptr,
                       false, batch, qs, num_q_heads, 1.f, num_splits, nullptr, 0, nullptr,
                       PSKV_DTYPE_BF16, nullptr, nullptr, bytes);
}

int decode_attn_multirow_workspace_bytes(const pskv_layout *layout, const int32_t *seq_lens_host,
                                         int32_t table_stride, int32_t batch, int32_t num_tokens,
                                         int32_t num_q_heads, int32_t tree, int32_t num_splits,
                                         size_t *bytes) {
  if (!bytes) return PSKV_ERR_INVALID_ARG;
  QuerySpec qs;
  qs.tokens = num_tokens;
  qs.tree_plan = tree != 0;
  return decode_common(layout, nullptr, nullptr, table_stride, seq_lens_host, nullptr, nullptr,
                       nullptr, false, batch, qs, num_q_heads, 1.f, num_splits, nullptr, 0,
                       nullptr, PSKV_DTYPE_BF16, nullptr, nullptr, bytes);
}

int merge_partials(const float *m, const float *l, const float *o, int32_t rows,
                   int32_t num_splits, int32_t head_dim_v, void *out, int32_t out_dtype,
                   void *workspace, size_t workspace_bytes, int32_t *status,
                   const pskv_decode_opts *opts, pskv_stream_t stream) {
  if (!m || !l || !o || !out || rows < 1 || num_splits < 1 || num_splits > PSKV_MAX_SPLITS ||
      head_dim_v < 4 || head_dim_v % 4 != 0)
    return PSKV_ERR_INVALID_ARG;
  if (out_dtype != PSKV_DTYPE_F32 && out_dtype != PSKV_DTYPE_BF16) return PSKV_ERR_INVALID_ARG;
  if (!aligned(o, 16) || !aligned(out, 16) || !aligned(m, 4) || !aligned(l, 4))
    return PSKV_ERR_INVALID_ARG;
  int group = 0, rc;
  if ((rc = merge_group_of(opts, &group))) return rc;
  WorkspacePlan w;
  if ((rc = plan_workspace(1, rows, head_dim_v, num_splits, group, &w))) return rc;
  if (w.groups > kMaxGroups) return PSKV_ERR_INVALID_ARG;
  (void)workspace;  // the group states stay on chip: no scratch is needed
  (void)workspace_bytes;
  MergeArgs a;
  a.m = m;
  a.l = l;
  a.o = o;
  a.rows = rows;
  a.count = num_splits;
  a.dv = head_dim_v;
  a.group = group;
  a.out = out;
  a.out_dtype = out_dtype;
  a.status = status;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (opts && opts->partial_begin) {
    e = cudaEventRecord(reinterpret_cast<cudaEvent_t>(opts->partial_begin), s);
    if (e != cudaSuccess) return cuda_fail(e);
  }
  int launched = 0;
  e = launch_merge(a, s, &launched);
  g_launches.fetch_add((uint64_t)launched, std::memory_order_relaxed);
  if (e != cudaSuccess) return cuda_fail(e);
  if (opts && opts->partial_end) {
    e = cudaEventRecord(reinterpret_cast<cudaEvent_t>(opts->partial_end), s);
    if (e != cudaSuccess) return cuda_fail(e);
  }
  return PSKV_OK;
}

int decode_attn_workspace_bytes(int32_t batch, int32_t num_q_heads, int32_t head_dim_v,
                                int32_t num_splits, size_t *bytes) {
  if (!bytes || num_splits < 0 || num_splits > PSKV_MAX_SPLITS) return PSKV_ERR_INVALID_ARG;
  const int64_t p = num_splits == 0 ? PSKV_AUTO_MAX_SPLITS : num_splits;
  WorkspacePlan w;
  const int rc = plan_workspace(batch, num_q_heads, head_dim_v, p, PSKV_MERGE_GROUP, &w);
  if (rc) return rc;
  *bytes = w.total;
  return PSKV_OK;
}

int merge_partials_workspace_bytes(int32_t rows, int32_t num_splits, int32_t head_dim_v,
                                   size_t *bytes) {
  if (!bytes || num_splits < 1 || num_splits > PSKV_MAX_SPLITS) return PSKV_ERR_INVALID_ARG;
  WorkspacePlan w;
  const int rc = plan_workspace(1, rows, head_dim_v, num_splits, PSKV_MERGE_GROUP, &w);
  if (rc) return rc;
  *bytes = 0;  // the group states stay on chip
  return PSKV_OK;
}

int pskv_partial_scratch_bytes(int64_t batch, int64_t num_q_heads, int64_t head_dim_v,
                               int64_t num_splits, size_t *maxima, size_t *denominators,
                               size_t *numerators, size_t *total) {
  if (batch < 1 || num_q_heads < 1 || head_dim_v < 1 || num_splits < 1)
    return PSKV_ERR_INVALID_ARG;
  size_t states, nums, sum;
  if (__builtin_mul_overflow((size_t)batch, (size_t)num_q_heads, &states) ||
      __builtin_mul_overflow(states, (size_t)num_splits, &states) ||
      __builtin_mul_overflow(states, (size_t)4, &states) ||
      __builtin_mul_overflow(states, (size_t)head_dim_v, &nums) ||
      __builtin_add_overflow(states, states, &sum) || __builtin_add_overflow(sum, nums, &sum))
    return PSKV_ERR_OVERFLOW;
  if (maxima) *maxima = states;
  if (denominators) *denominators = states;
  if (numerators) *numerators = nums;
  if (total) *total = sum;
  return PSKV_OK;
}

int pskv_plan_splits(const pskv_layout *layout, int32_t batch, int32_t num_q_heads,
                     const int32_t *seq_lens_host, int32_t *num_splits) {
  if (!layout || !seq_lens_host || !num_splits || batch < 1 || num_q_heads < 1)
    return PSKV_ERR_INVALID_ARG;
  if (num_q_heads % layout->d.num_kv_heads != 0) return PSKV_ERR_UNSUPPORTED;
  const int group = num_q_heads / layout->d.num_kv_heads;
  // single-token decode: one column per query head of the KV group
  int P = 0;
  const int rc = auto_partial_splits(layout->d, batch, group, group, seq_lens_host, &P);
  if (rc) return rc;
  *num_splits = P;
  return PSKV_OK;
}

const char *pskv_strerror(int status) {
  switch (status) {
    case PSKV_OK: return "ok";
    case PSKV_ERR_INVALID_ARG: return "invalid argument";
    case PSKV_ERR_UNSUPPORTED: return "unsupported shape or format";
    case PSKV_ERR_OVERFLOW: return "size overflow";
    case PSKV_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case PSKV_ERR_PAST_PAGES: return "position past the row's pages";
    case PSKV_ERR_CUDA: return "CUDA error";
    default: return "unknown status";
  }
}

const char *pskv_last_cuda_error(void) { return g_cuda_error; }

uint64_t pskv_kernel_launches(void) { return g_launches.load(std::memory_order_relaxed); }

int pskv_version(void) { return 102; }

int pskv_check_flags(const pskv_layout *layout, int32_t clear, pskv_stream_t stream,
                     uint32_t *flags) {
  if (!layout || !flags) return PSKV_ERR_INVALID_ARG;
  *flags = 0;
  int32_t *status = layout->d.status;
  if (!status) return PSKV_OK;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int32_t word = 0;
  cudaError_t e = cudaMemcpyAsync(&word, status, sizeof word, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess && clear) e = cudaMemsetAsync(status, 0, sizeof(int32_t), s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e);
  *flags = (uint32_t)word;
  return PSKV_OK;
}

}  // extern "C"
