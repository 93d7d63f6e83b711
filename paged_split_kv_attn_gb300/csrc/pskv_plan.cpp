// pskv_plan.cpp -- host-only planning and argument checks (no CUDA calls).
#include "pskv_plan.h"

#include <stdlib.h>

namespace pskv {

static bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_layout_desc(const pskv_layout_desc *d) {
  if (!d || !d->k_pool || !d->v_pool) return PSKV_ERR_INVALID_ARG;
  if (d->num_pages < 1 || d->page_size < 1 || d->num_kv_heads < 1 || d->head_dim_k < 1 ||
      d->head_dim_v < 1)
    return PSKV_ERR_INVALID_ARG;
  if (d->page_size % PSKV_KEY_TILE != 0) return PSKV_ERR_INVALID_ARG;
  if (d->kv_dtype != PSKV_DTYPE_F32 && d->kv_dtype != PSKV_DTYPE_BF16) return PSKV_ERR_INVALID_ARG;
  if (d->format != PSKV_FORMAT_SPLIT && d->format != PSKV_FORMAT_FOLDED) return PSKV_ERR_INVALID_ARG;
  if (d->head_dim_v != 256 && d->head_dim_v != 512) return PSKV_ERR_UNSUPPORTED;
  if (d->format == PSKV_FORMAT_SPLIT && d->head_dim_k != d->head_dim_v) return PSKV_ERR_UNSUPPORTED;
  if (d->format == PSKV_FORMAT_FOLDED &&
      (d->head_dim_k * 4 != d->head_dim_v || d->kv_dtype != PSKV_DTYPE_BF16))
    return PSKV_ERR_UNSUPPORTED;
  if (!aligned16(d->k_pool) || !aligned16(d->v_pool)) return PSKV_ERR_INVALID_ARG;
  if (d->status && (reinterpret_cast<uintptr_t>(d->status) & 3u)) return PSKV_ERR_INVALID_ARG;
  // every element index of a region must fit in size_t and every row index in int64
  size_t rows, elems;
  if (__builtin_mul_overflow((size_t)d->num_pages, (size_t)d->num_kv_heads, &rows) ||
      __builtin_mul_overflow(rows, (size_t)d->page_size, &rows) ||
      __builtin_mul_overflow(rows, (size_t)d->head_dim_v * 4, &elems))
    return PSKV_ERR_OVERFLOW;
  if (d->num_pages > 0x7fffffffLL) return PSKV_ERR_UNSUPPORTED;  // page ids are int32
  return PSKV_OK;
}

static size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

int plan_workspace(int64_t batch, int64_t num_q_heads, int64_t head_dim_v, int64_t splits,
                   int64_t group, WorkspacePlan *out) {
  if (!out || batch < 1 || num_q_heads < 1 || head_dim_v < 1 || splits < 1 || group < 1)
    return PSKV_ERR_INVALID_ARG;
  const int64_t ng = (splits + group - 1) / group;
  size_t rows, states, ostate;
  if (__builtin_mul_overflow((size_t)batch, (size_t)num_q_heads, &rows) ||
      __builtin_mul_overflow(rows, (size_t)splits * 4, &states) ||
      __builtin_mul_overflow(states, (size_t)head_dim_v, &ostate))
    return PSKV_ERR_OVERFLOW;
  if (states > ((size_t)1 << 60) || ostate > ((size_t)1 << 60))
    return PSKV_ERR_OVERFLOW;  // keeps the additions below from wrapping
  WorkspacePlan w;
  w.m_off = 0;
  w.l_off = align256(w.m_off + states);
  w.o_off = align256(w.l_off + states);
  w.total = align256(w.o_off + ostate);
  w.groups = (int)ng;
  *out = w;
  return PSKV_OK;
}

int check_lengths(const pskv_layout *layout, int32_t batch, int32_t table_stride,
                  const int32_t *seq_lens_host, int32_t min_len) {
  if (!layout || !seq_lens_host || batch < 1 || table_stride < 1 || min_len < 1)
    return PSKV_ERR_INVALID_ARG;
  const int64_t cap = (int64_t)table_stride * layout->d.page_size;
  for (int32_t b = 0; b < batch; ++b)
    if (seq_lens_host[b] < min_len || (int64_t)seq_lens_host[b] > cap) return PSKV_ERR_INVALID_ARG;
  return PSKV_OK;
}

int plan_splits(int slots, int32_t batch, int32_t num_kv_heads, const int32_t *seq_lens_host,
                int fill32) {
  if (slots < 1) slots = 1;
  int64_t total_tiles = 0, max_tiles = 0;
  for (int32_t b = 0; b < batch; ++b) {
    const int64_t len = seq_lens_host[b] > 0 ? seq_lens_host[b] : 0;
    const int64_t t = (len + PSKV_KEY_TILE - 1) / PSKV_KEY_TILE;
    total_tiles += t;
    if (t > max_tiles) max_tiles = t;
  }
  if (max_tiles == 0) return 1;
  // The longest row's pieces should carry about total_tiles * Hkv / slots tiles
  // each (one wave of CTAs when all rows are equal), filled to fill32 / 32 of
  // the slots (see pskv_plan.h).  For a batch, twice as many pieces, so that
  // short rows' CTAs fill the tail.  A piece keeps at least three tiles (short
  // windows are bound by each CTA's start, not by bytes).
  if (fill32 < 1 || fill32 > 32) fill32 = 32;
  int64_t p = (max_tiles * (int64_t)slots * fill32) / (total_tiles * (int64_t)num_kv_heads * 32);
  if (batch > 1) p *= 2;
  if (p > max_tiles / 3) p = max_tiles / 3;
  if (p < 1) p = 1;
  if (p > max_tiles) p = max_tiles;
  if (p > PSKV_AUTO_MAX_SPLITS) p = PSKV_AUTO_MAX_SPLITS;
  return (int)p;
}

int check_append_host(const pskv_layout *layout, int32_t n, int32_t table_stride, int32_t batch,
                      const int32_t *row_of, const int32_t *pos_of, const int32_t *pages_of_row) {
  if (!layout || !row_of || !pos_of || !pages_of_row) return PSKV_ERR_INVALID_ARG;
  for (int32_t r = 0; r < n; ++r) {
    const int32_t b = row_of[r], pos = pos_of[r];
    if (b < 0 || b >= batch || pos < 0) return PSKV_ERR_INVALID_ARG;
    const int32_t lease = pages_of_row[b];
    if (lease < 0 || lease > table_stride) return PSKV_ERR_INVALID_ARG;
    if ((int64_t)pos >= (int64_t)lease * layout->d.page_size) return PSKV_ERR_PAST_PAGES;
  }
  return PSKV_OK;
}

int pick_kernel(int kv_dtype, int head_dim, int group, int format) {
  const bool mma_group = group == 1 || group == 2 || group == 4 || group == 8;
  if (kv_dtype == PSKV_DTYPE_BF16 && mma_group && (head_dim == 256 || head_dim == 512))
    return kKernelMma;
  if (format == PSKV_FORMAT_FOLDED) return -1;  // folded pools run on the tensor-core consumer only
  const bool g_ok = group == 1 || group == 2 || group == 4 || group == 8 ||
                    (group == 16 && head_dim == 256);
  if ((head_dim == 256 || head_dim == 512) && g_ok) return kKernelSimt;
  return -1;
}

int plan_tc_splits(int64_t units, int slots, int64_t max_tiles) {
  if (units < 1 || slots < 1 || units >= slots) return 1;
  int64_t cap = max_tiles / 4;
  if (cap > 32) cap = 32;
  if (cap < 1) cap = 1;
  const int64_t p = (slots + units - 1) / units;  // one wave at least
  return (int)(p < cap ? p : cap);
}

int plan_verify_splits(int64_t units, int slots, int64_t max_tiles) {
  if (units < 1 || slots < 1 || units >= slots) return 1;
  int64_t p = slots / units;
  const int64_t cap = max_tiles / 2 < PSKV_MAX_SPLITS ? max_tiles / 2 : PSKV_MAX_SPLITS;
  if (p > cap) p = cap;
  return p < 1 ? 1 : (int)p;
}

}  // namespace pskv
