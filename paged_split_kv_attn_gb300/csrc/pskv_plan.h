// pskv_plan.h -- host-only planning and argument checks (no CUDA calls).
//
// Kept free of CUDA so it can be compiled and tested on any host, including
// under the address and undefined-behaviour sanitizers.
#pragma once

#include <stddef.h>
#include <stdint.h>

#include "pskv.h"

struct pskv_layout {
  pskv_layout_desc d;
  int elem_size;    // bytes per element
  int k_row_bytes;  // bytes of one stored key row of one head
  int v_row_bytes;  // bytes of one value row of one head
};

namespace pskv {

// Byte offsets of the workspace sections (each 256-byte aligned): the
// partials only (the merge keeps its group states on chip).
struct WorkspacePlan {
  size_t m_off, l_off, o_off;  // partials: m, l [rows][P], o [rows][P][dv]
  size_t total;
  int groups;  // ng = ceil(P / group)
};

int check_layout_desc(const pskv_layout_desc *d);

// Sizes of the decode workspace for `splits` partitions (merged in groups of `group`).
int plan_workspace(int64_t batch, int64_t num_q_heads, int64_t head_dim_v, int64_t splits,
                   int64_t group, WorkspacePlan *out);

// Checks the host lengths: each in [min_len, table_stride * page_size].
int check_lengths(const pskv_layout *layout, int32_t batch, int32_t table_stride,
                  const int32_t *seq_lens_host, int32_t min_len = 1);

// Automatic split count for `slots` CTA slots (SMs x CTAs per SM), filling
// fill32 / 32 of them.  Byte-bound calls (the split-format single-token decode
// on the tensor-core kernel) fill 27/32: with a few SMs running one CTA
// instead of two the stream still saturates HBM, and fewer, longer pieces
// spend less on each CTA's start and on the merge (measured on GB300 over
// 10.6K-163K keys: 64 pieces of a 304-slot grid beat 76 by 1-3.5 % per call).
// Calls with more arithmetic per byte (folded rows, verify windows, prefill)
// fill every slot.
constexpr int kFillBytes32 = 27;
// Key partitions for the tensor-memory prefill kernel: `units` blocks of 128
// query columns (x KV heads x rows) over `slots` concurrent units (SMs, or SM
// pairs at head dim 512), each block holding up to max_tiles 64-key tiles.
// Splits the keys only when the blocks alone leave slots idle: P = ceil(slots /
// units), at most 32 and at least 4 tiles per partition; with a wave or more
// of blocks, P = 1 (a block's fixed costs and the merge outweigh balancing the
// last wave).
int plan_tc_splits(int64_t units, int slots, int64_t max_tiles);
// Partitions per (row, KV head) for the key-major verify kernel: `units`
// (KV heads x rows) CTAs per partition over `slots` SMs, rows of at most
// max_tiles 128-key tiles.  One wave: P = floor(slots / units), at least 1,
// at most max_tiles / 2 (two tiles per partition) and PSKV_MAX_SPLITS.
int plan_verify_splits(int64_t units, int slots, int64_t max_tiles);
int plan_splits(int slots, int32_t batch, int32_t num_kv_heads, const int32_t *seq_lens_host,
                int fill32 = 32);

// Checks host copies of an append's rows against the leases.
int check_append_host(const pskv_layout *layout, int32_t n, int32_t table_stride, int32_t batch,
                      const int32_t *row_of, const int32_t *pos_of, const int32_t *pages_of_row);

// Which partial kernel family serves (dtype, head_dim_v, group, format); -1 if none.
enum { kKernelMma = 0, kKernelSimt = 1 };
int pick_kernel(int kv_dtype, int head_dim, int group, int format = PSKV_FORMAT_SPLIT);

}  // namespace pskv
