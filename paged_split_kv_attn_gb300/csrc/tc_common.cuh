// tc_common.cuh -- pieces shared by the tensor-memory attention kernels:
// bounded barrier waits with a CTA-wide abort flag, the elected issuing lane,
// 2^x on the special-function unit, the copy warp's page-id cache and the
// tensor maps over a pool region.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pskv_internal.cuh"

namespace pskv {
namespace tc {

// Bounded wait that gives up at once when another thread of the CTA already has.
__device__ __forceinline__ bool tc_wait(uint64_t *bar, uint32_t parity, volatile int *abort_flag,
                                        int32_t *status) {
  if (*abort_flag) return false;
  if (mbar_wait(bar, parity)) return true;
  *abort_flag = 1;
  raise_fault(status, PSKV_FAULT_WAIT_TIMEOUT);
  return false;
}

// The same wait taken by a whole warp: one answer for all lanes.
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, volatile int *abort_flag,
                                          int32_t *status) {
  const bool ok = tc_wait(bar, parity, abort_flag, status);
  return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ bool elect_one() {
  uint32_t pred;
  asm volatile(
      "{\n\t.reg .pred p;\n\telect.sync _|p, 0xffffffff;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(pred));
  return pred != 0;
}

// 2^x by the special-function unit (inputs of -inf give 0; results below the
// smallest normal flush to 0, far below what a weight can contribute).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Page ids of 32 consecutive table slots held across the copy warp's lanes.
struct PageCache {
  int base = -1, val = -1;
  __device__ int get(const int32_t *tbl, int slot, int n_slots, int lane) {
    if (base < 0 || slot < base || slot >= base + 32) {
      base = slot;
      val = slot + lane < n_slots ? __ldg(tbl + slot + lane) : -1;
    }
    return __shfl_sync(0xffffffffu, val, slot - base);
  }
};

// The pool's tensor-map encoder, looked up once from the driver.
inline PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      p = nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }();
  return fn;
}

// The pool region as a 2-D tensor of `rows` rows of `dt` bf16, read in boxes
// of 64 columns x box_rows rows in the 128-byte swizzled layout.
inline bool make_map(CUtensorMap *m, const void *region, long long rows, int dt, int box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)dt, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)dt * 2};
  const cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  const cuuint32_t elem[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(region), dims, strides,
             box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Queries [rows][heads][dt] bf16 as a 3-D tensor read in boxes of 64 columns x
// `heads_box` heads x `rows_box` rows (128-byte swizzled): a box holds the
// query columns (row, head) of one KV group in row-major order.
inline bool make_q_map(CUtensorMap *m, const void *q, long long rows, int heads, int dt,
                       int heads_box, int rows_box) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)dt, (cuuint64_t)heads, (cuuint64_t)rows};
  const cuuint64_t strides[2] = {(cuuint64_t)dt * 2, (cuuint64_t)heads * dt * 2};
  const cuuint32_t box[3] = {64, (cuuint32_t)heads_box, (cuuint32_t)rows_box};
  const cuuint32_t elem[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(q), dims, strides, box,
             elem, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace tc
}  // namespace pskv
