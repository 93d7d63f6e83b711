// pskv_internal.cuh -- shared declarations of the CUDA library (not installed).
//
// Device helpers wrap the sm_90+/sm_100 PTX the kernels use: mbarriers, the
// bulk async copy engine (cp.async.bulk, "TMA" without a tensor map),
// ldmatrix / movmatrix and the bf16 mma.  Every wait on an mbarrier is
// bounded; a wait that expires reports failure instead of spinning forever.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "pskv.h"

namespace pskv {

constexpr int kKeyTile = PSKV_KEY_TILE;  // keys per tile
constexpr uint32_t kWaitPolls = 1u << 22;            // try_wait polls before giving up
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

constexpr int kLenHints = 8;  // rows whose host length rides in the kernel arguments

// Arguments of the split-KV partial kernels (one launch, grid (P, Hkv, B)).
struct PartialArgs {
  const void *q;             // [B][Hq][D]
  const void *k_pool;        // [num_pages][Hkv][ps][D]
  const void *v_pool;
  const int32_t *page_tables;  // [B][table_stride]
  const int32_t *seq_lens;     // [B]
  const int32_t *first_pos;    // [B] or null
  const int32_t *window_lo;    // [B] or null
  int32_t *status;             // fault word or null
  float *ws_m;                 // [B][Hq][P]
  float *ws_l;                 // [B][Hq][P]
  float *ws_o;                 // [B][Hq][P][D]
  long long num_pages;
  int table_stride;
  int page_size;
  int num_kv_heads;
  int num_q_heads;
  int num_splits;
  int num_tokens;    // query tokens per row (1, or a verify window's length) when cu_q is null
  int col_blocks;    // CTAs per (row, KV head, partition): query columns in blocks
  float scale_log2;  // scale * log2(e)
  const int32_t *cu_q;  // [B + 1] first query row of each table row (varlen prefill), or null
  int total_rows;       // query rows in all (checks cu_q)
  int window;           // per-token window in keys (prefill), 0 = none
  void *out;            // [rows][Hq][D] of out_dtype: written directly when `direct`
  int out_dtype;
  int direct;           // one partition: write o / l to `out`, no partials, no merge
  const void *append_k;  // [B][Hkv][Dk]: the new row of key len - 1 written by its CTA, or null
  const void *append_v;  // [B][Hkv][Dv]
  const int32_t *append_pages;  // [B] pages leased per row
  int k_row_bytes, v_row_bytes;  // bytes of one stored K / V row of one head
  // [rows] ancestor mask of each query token of a drafted tree (bit j: the
  // window's token j is visible), or null for causal windows
  const unsigned long long *tree_mask;
  // Host copies of the first rows' lengths (-1: none): the producer warp
  // fetches the page ids its partition starts with while the device length
  // is still on its way, and keeps them only when the device length gives
  // the same first table slot and slot count (plain uniform rows only).
  int len_hint[kLenHints];
};

// Arguments of the merge kernel: level 1 folds groups of `group` partials of
// each row into group states (on chip), level 2 folds a row's group states
// and writes the normalised output.
struct MergeArgs {
  const float *m;  // [rows][count]
  const float *l;
  const float *o;  // [rows][count][dv]
  int rows;
  int count;
  int dv;
  int group;
  void *out;  // [rows][dv]
  int out_dtype;
  int32_t *status;
};

struct AppendArgs {
  const void *k_new;  // [n][Hkv][D]
  const void *v_new;
  const int32_t *row_of;
  const int32_t *pos_of;
  int n;
  const int32_t *page_tables;
  int table_stride;
  const int32_t *pages_of_row;
  int batch;
  void *k_pool;
  void *v_pool;
  long long num_pages;
  int page_size;
  int num_kv_heads;
  int k_row_bytes;  // head_dim_k * element size, a multiple of 16
  int v_row_bytes;  // head_dim_v * element size, a multiple of 16
  int32_t *status;
};

struct PrepArgs {
  const void *x;          // bf16 projection rows [n][x_stride]
  long long x_stride;     // elements per projection row
  int q_col, k_col, v_col;  // first column of the q, K and V bands
  int n;                  // tokens
  int num_q_heads;
  int num_kv_heads;
  int d;                  // head dim
  int rot;                // leading columns rotated (even)
  float eps;
  const float *w_q;       // [d] or null (1)
  const float *w_k;       // [d] or null (1)
  const float *rope_cos;  // [max_pos][rot / 2]
  const float *rope_sin;
  int max_pos;
  const int32_t *row_of;  // [n] table row of each token
  const int32_t *pos_of;  // [n] key index of each token in its row
  const int32_t *first_pos;  // [batch] position of key 0 of each row, or null (0)
  const int32_t *page_tables;
  int table_stride;
  const int32_t *pages_of_row;
  int batch;
  void *k_pool;
  void *v_pool;
  long long num_pages;
  int page_size;
  int k_cols;             // stored K columns: d (split) or rot (folded)
  int folded;             // fold K's multiplier into q past rot
  void *q_out;            // bf16 [n][num_q_heads][d]
  int32_t *status;
};


// Host-side launchers (one per kernel family).  They return a CUDA error code.
// The tensor-core family takes `nt` n-tiles of 8 query columns (group x tokens <= 8 nt).
cudaError_t launch_partial_mma(const PartialArgs &a, int head_dim, int group, bool folded, int nt,
                               dim3 grid, cudaStream_t s);
cudaError_t launch_partial_simt_f32(const PartialArgs &a, int head_dim, int group, dim3 grid,
                                    cudaStream_t s);
cudaError_t launch_partial_simt_bf16(const PartialArgs &a, int head_dim, int group, dim3 grid,
                                     cudaStream_t s);
cudaError_t occupancy_partial_mma(int head_dim, int group, bool folded, int nt, int *ctas);
cudaError_t occupancy_partial_simt_f32(int head_dim, int group, int *ctas);
cudaError_t occupancy_partial_simt_bf16(int head_dim, int group, int *ctas);
cudaError_t launch_merge(const MergeArgs &a, cudaStream_t s, int *launches);
cudaError_t launch_append(const AppendArgs &a, cudaStream_t s);
cudaError_t launch_prep(const PrepArgs &a, cudaStream_t s);

// Launch `kernel` with programmatic dependent launch allowed: it may start
// while the previous kernel on the stream is still running, and must execute
// pdl_wait() before touching memory that kernel (or any earlier one) uses.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args &&...args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

#ifdef __CUDACC__

// Wait until the previous grid on the stream has completed and its writes are
// visible (a no-op when the kernel was not launched with PDL).  Every kernel of
// this library executes it before its first global access that could conflict
// and before it exits, so stream order holds transitively across a chain.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Allow the next kernel on the stream to begin launching.
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void raise_fault(int32_t *status, uint32_t bits) {
  if (status) atomicOr(reinterpret_cast<unsigned int *>(status), bits);
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(
          smem_u32(bar)),
      "r"(bytes)
      : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait for the phase of `bar` with the given parity to complete.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  for (uint32_t i = 0; i < kWaitPolls; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}

// One bulk copy global -> shared; completion is counted in bytes on `bar`.
// Both addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes,
                                         uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// The same copy with an L2 eviction policy (from make_evict_first_policy):
// streamed K/V bytes are read once per call, so they are marked first to go
// and the small, reused data (tables, lengths, queries, partials) stays.
__device__ __forceinline__ void bulk_g2s_hint(void *dst, const void *src, uint32_t bytes,
                                              uint64_t *bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

__device__ __forceinline__ uint64_t make_evict_first_policy() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// Partials (m, l, o) are read back by the merge right after the kernel that
// writes them; stored with an L2 evict-last policy they stay in L2 while the
// rest of the K/V stream passes (written plainly, most of them were written
// back to DRAM before the merge ran, and the merge read them from DRAM).
__device__ __forceinline__ uint64_t make_evict_last_policy() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ void st_keep(float *p, float v, uint64_t policy) {
  asm volatile("st.global.L2::cache_hint.f32 [%0], %1, %2;" ::"l"(p), "f"(v), "l"(policy)
               : "memory");
}
__device__ __forceinline__ void st_keep(float4 *p, float4 v, uint64_t policy) {
  asm volatile("st.global.L2::cache_hint.v4.f32 [%0], {%1, %2, %3, %4}, %5;" ::"l"(p), "f"(v.x),
               "f"(v.y), "f"(v.z), "f"(v.w), "l"(policy)
               : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &a0, uint32_t &a1, uint32_t &a2,
                                        uint32_t &a3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(a0), "=r"(a1), "=r"(a2), "=r"(a3)
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &a0, uint32_t &a1, uint32_t &a2,
                                          uint32_t &a3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(a0), "=r"(a1), "=r"(a2), "=r"(a3)
               : "r"(addr));
}

__device__ __forceinline__ uint32_t movmatrix_t(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

// c += A(16x16, row) * B(16x8, col), bf16 inputs, f32 accumulate.
__device__ __forceinline__ void mma_bf16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Two floats -> packed bf16x2 (round to nearest even); `lo` in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&v);
}

__device__ __forceinline__ float bf16_lo(uint32_t x) { return __uint_as_float(x << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t x) { return __uint_as_float(x & 0xffff0000u); }

#endif  // __CUDACC__

}  // namespace pskv
