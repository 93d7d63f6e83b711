// pskv_static.cu -- split-KV decode for callers that cannot allocate device memory.
//
// decode_attn_splitkv needs a caller-supplied workspace for the split-KV
// partials and the merge's group results.  Some callers have no way to get
// one: code running where cudaMalloc is off limits (for example inside a
// host callback, a signal-safe or real-time path that must not enter the
// allocator, or a plugin whose host framework owns all device allocations
// and exposes no scratch API).  decode_attn_splitkv_static serves them from a
// fixed scratch array compiled into this library instead.
//
// The array is a file-scope __device__ variable, so every GPU that loads the
// library holds PSKV_STATIC_SCRATCH_BYTES of it until the process exits.  Its
// name is only meaningful in device code; host code needs the device address,
// which cudaGetSymbolAddress returns per device.  This file looks that address
// up the first time the entry point runs on a device (with that device
// current) and caches it; that first call should therefore happen before any
// stream capture begins on that device.  The cached address belongs to the
// device's primary context as it was then: after cudaDeviceReset on that
// device the module is loaded again and the address may change, so calling
// this entry point after a reset is not supported.
//
// Every call uses the same array and the array keeps whatever the previous
// call left in it.  Nothing in it has to start at zero: each decode writes
// every partial and group result before reading it.  Two calls whose work
// overlaps on the GPU (different streams, or different host threads, without
// ordering between them) would write the same bytes at the same time: callers
// must order them.
#include <mutex>

#include "pskv_internal.cuh"
#include "pskv_plan.h"

namespace {

__device__ __align__(256) unsigned char g_static_scratch[PSKV_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
void *g_scratch_addr[kMaxDevices] = {};
std::mutex g_scratch_mutex;

// Device address of the scratch array on the current device (looked up once per device).
int scratch_address(void **out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PSKV_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (!g_scratch_addr[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || !p) return PSKV_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return PSKV_OK;
}

}  // namespace

extern "C" int decode_attn_splitkv_static(const pskv_layout *layout, const void *q,
                                          const int32_t *page_tables, int32_t table_stride,
                                          const int32_t *seq_lens_host, const int32_t *seq_lens,
                                          int32_t batch, int32_t num_q_heads, float scale,
                                          int32_t num_splits, void *out, int32_t out_dtype,
                                          pskv_stream_t stream) {
  if (!layout || !seq_lens_host || batch < 1 || num_q_heads < 1) return PSKV_ERR_INVALID_ARG;
  if (num_splits < 0 || num_splits > PSKV_MAX_SPLITS) return PSKV_ERR_INVALID_ARG;
  int P = num_splits;
  if (P == 0) {
    // the automatic plan, lowered if needed to the most splits the array can hold
    int rc = pskv_plan_splits(layout, batch, num_q_heads, seq_lens_host, &P);
    if (rc) return rc;
    while (P > 1) {
      size_t need = 0;
      rc = decode_attn_workspace_bytes(batch, num_q_heads, layout->d.head_dim_v, P, &need);
      if (rc == PSKV_OK && need <= (size_t)PSKV_STATIC_SCRATCH_BYTES) break;
      --P;
    }
  }
  size_t need = 0;
  int rc = decode_attn_workspace_bytes(batch, num_q_heads, layout->d.head_dim_v, P, &need);
  if (rc) return rc;
  if (need > (size_t)PSKV_STATIC_SCRATCH_BYTES) return PSKV_ERR_WORKSPACE_TOO_SMALL;
  void *scratch = nullptr;
  if ((rc = scratch_address(&scratch))) return rc;
  return decode_attn_splitkv(layout, q, page_tables, table_stride, seq_lens_host, seq_lens, batch,
                             num_q_heads, scale, P, scratch, PSKV_STATIC_SCRATCH_BYTES, out,
                             out_dtype, nullptr, stream);
}
