// append.cu -- copy new K/V rows into their pages, bit for bit.
//
// TensorFold #1619 ("gemma4 CUDA: the global layers' caches in pages of the
// core pool..."), description "Writes": the rows a forward produced are copied
// into the pages so the cache holds the same bits a linear cache would;
// "Leasing": a row past its slot's pages is refused (PastPages).
// One warp moves one (new row, KV head) pair with 16-byte vector loads and
// stores.  Every index is checked on the device; a bad row is skipped and a
// fault bit set, never trapped.
#include "pskv_internal.cuh"

namespace pskv {

constexpr int kAppendWarps = 4;

// Longest row handled: 2048 bytes (head dim 512 in f32) = 4 vectors of 16 bytes per lane.
// (K rows of a folded pool are a quarter of that.)
constexpr int kMaxVecsPerLane = 4;

__global__ void __launch_bounds__(kAppendWarps * 32) pskv_append_rows(const AppendArgs a) {
  const long long item = (long long)blockIdx.x * kAppendWarps + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  pdl_wait();
  pdl_launch_dependents();
  if (item >= (long long)a.n * a.num_kv_heads) return;
  const int r = (int)(item / a.num_kv_heads), h = (int)(item % a.num_kv_heads);
  const size_t src_row = (size_t)r * a.num_kv_heads + h;
  const uint4 *ks = reinterpret_cast<const uint4 *>(static_cast<const char *>(a.k_new) +
                                                    src_row * a.k_row_bytes);
  const uint4 *vs = reinterpret_cast<const uint4 *>(static_cast<const char *>(a.v_new) +
                                                    src_row * a.v_row_bytes);
  const int kvecs = a.k_row_bytes / 16, vvecs = a.v_row_bytes / 16;
  // the row's bytes and its indices are independent: load them all before any check
  uint4 kb[kMaxVecsPerLane], vb[kMaxVecsPerLane];
#pragma unroll
  for (int i = 0; i < kMaxVecsPerLane; ++i) {
    const int v = lane + 32 * i;
    if (v < kvecs) kb[i] = ks[v];
    if (v < vvecs) vb[i] = vs[v];
  }
  const int b = a.row_of[r], pos = a.pos_of[r];
  if (b < 0 || b >= a.batch || pos < 0) {
    if (lane == 0 && h == 0) raise_fault(a.status, PSKV_FAULT_PAST_PAGES);
    return;
  }
  const int lease = a.pages_of_row[b];
  const long long slot = pos / a.page_size;
  const int page = slot < a.table_stride ? a.page_tables[(size_t)b * a.table_stride + slot] : -1;
  if (lease < 0 || lease > a.table_stride || (long long)pos >= (long long)lease * a.page_size) {
    if (lane == 0 && h == 0) raise_fault(a.status, PSKV_FAULT_PAST_PAGES);
    return;
  }
  if (page < 0 || (long long)page >= a.num_pages) {
    if (lane == 0 && h == 0) raise_fault(a.status, PSKV_FAULT_BAD_PAGE);
    return;
  }
  const size_t dst_row = ((size_t)page * a.num_kv_heads + h) * a.page_size + pos % a.page_size;
  uint4 *kd = reinterpret_cast<uint4 *>(static_cast<char *>(a.k_pool) + dst_row * a.k_row_bytes);
  uint4 *vd = reinterpret_cast<uint4 *>(static_cast<char *>(a.v_pool) + dst_row * a.v_row_bytes);
#pragma unroll
  for (int i = 0; i < kMaxVecsPerLane; ++i) {
    const int v = lane + 32 * i;
    if (v < kvecs) kd[v] = kb[i];
    if (v < vvecs) vd[v] = vb[i];
  }
}

cudaError_t launch_append(const AppendArgs &a, cudaStream_t s) {
  const long long items = (long long)a.n * a.num_kv_heads;
  const long long blocks = (items + kAppendWarps - 1) / kAppendWarps;
  if (blocks <= 0) return cudaSuccess;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
  return launch_pdl(pskv_append_rows, dim3((unsigned)blocks), dim3(kAppendWarps * 32), 0, s, a);
}

}  // namespace pskv
