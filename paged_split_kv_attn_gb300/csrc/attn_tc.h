// attn_tc.h -- arguments and launcher of the tensor-memory (tcgen05) attention
// kernel (not installed).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace pskv {

// Arguments of the tensor-memory (tcgen05) attention kernel: paged prefill at
// head dim 256 or 512 over bf16 split pools; grid (qblocks * P, Hkv, B), one CTA
// (head dim 512: a pair of CTAs) per block of 128 query columns (tokens x the
// KV group's heads) and partition.
struct TcArgs {
  const void *q;               // bf16 [rows][Hq][D]
  const int32_t *page_tables;  // [B][table_stride]
  const int32_t *seq_lens;     // [B]
  const int32_t *cu_q;         // [B + 1] first query row of each table row, or null:
  int num_tokens;              //   then num_tokens rows per table row (a verify window)
  int32_t *status;
  float *ws_m, *ws_l, *ws_o;   // partials [rows][Hq][P] (o: x D) when not direct
  void *out;                   // [rows][Hq][D] of out_dtype when direct
  int out_dtype;
  int direct;
  long long num_pages;
  int table_stride, page_size, num_kv_heads, num_q_heads;
  int group_shift;             // log2 of the query heads per KV head
  int num_splits, qblocks, total_rows, window;
  int box_rows;                // rows per tensor copy: 64 when a page holds whole tiles, else 16
  float scale_log2;
  const unsigned long long *tree_mask;  // [rows] drafted-tree ancestor masks (key-major kernel), or null
};

// Encodes the pools' tensor maps (rows = num_pages * Hkv * page_size < 2^31) and launches:
// head dim 256 one CTA per (query block, partition) of `grid`, head dim 512 a pair of CTAs.
cudaError_t launch_attn_tc(const TcArgs &a, const void *k_pool, const void *v_pool, int head_dim,
                           dim3 grid, cudaStream_t s);

// Verify windows of 17 to 64 query columns per KV head (num_tokens rows per
// table row, qblocks 1, no offsets, no window): the key-major kernel, one CTA
// per (partition, KV head, row) of `grid`; partitions of whole 16-key groups.
cudaError_t launch_attn_verify(const TcArgs &a, const void *k_pool, const void *v_pool,
                               int head_dim, dim3 grid, cudaStream_t s);

}  // namespace pskv
