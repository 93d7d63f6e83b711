// prep.cu -- the K/V prep with the page write fused in.
//
// pegainfer #1055, Description: the hd512 prep writes the split or the folded
// row, and folds K's norm weight into the query.  pegainfer #1057,
// Description: the preps are elementwise, one RMS reduction per head row.
// TensorFold #1619, description "Writes": the rows go into the pages with the
// bits a linear cache would hold; "Leasing": a row past its slot's pages is
// refused.  Here one kernel does both: it normalises and rotates each new
// token's q, K and V head rows and stores K and V straight into their pages
// (no staging buffer, no separate copy launch) and the prepared q into q_out.
//
// One warp per (token, head row): the Hq query rows, then the Hkv key/value
// rows.  A row x of d columns becomes x / sqrt(mean(x^2) + eps) * w, then its
// first `rot` columns turn as pairs (i, i + rot/2) by the caller's cos/sin
// for the token's position; V is normalised only.  The sum of squares is
// formed in a fixed order (each lane over its columns in order, then a
// butterfly), so the result is deterministic.
#include "pskv_internal.cuh"

namespace pskv {

constexpr int kPrepWarps = 8;
constexpr int kPrepMaxD = 512;

__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) {
  return __uint_as_float(((uint32_t)b) << 16);
}

// Round-to-nearest-even float -> bf16 bits (NaN kept quiet).
__device__ __forceinline__ uint16_t float_to_bf16_bits(float f) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}

constexpr int kPrepChunks = kPrepMaxD / 8 / 32;  // 16-byte chunks of a head row per lane
constexpr int kPrepPairs = kPrepMaxD / 2 / 32;   // rotated pairs per lane at most

// One head row in flight: lane l holds columns [8v, 8v + 8) for v = l, l + 32, ...
struct RowRegs {
  uint4 x[kPrepChunks];
};

// A per-column multiplier for the same columns.
struct MulRegs {
  float4 m[kPrepChunks][2];
};

__device__ __forceinline__ void load_mul_regs(MulRegs &r, const float *w, int d, int lane) {
#pragma unroll
  for (int k = 0; k < kPrepChunks; ++k) {
    const int v = lane + 32 * k;
    if (v < d / 8) {
      r.m[k][0] = reinterpret_cast<const float4 *>(w)[2 * v];
      r.m[k][1] = reinterpret_cast<const float4 *>(w)[2 * v + 1];
    }
  }
}

__device__ __forceinline__ float mul_at(const MulRegs &r, int k, int e) {
  const float4 q = r.m[k][e >> 2];
  const int i = e & 3;
  return i == 0 ? q.x : (i == 1 ? q.y : (i == 2 ? q.z : q.w));
}

__device__ __forceinline__ void load_row_regs(RowRegs &r, const uint16_t *src, int d, int lane) {
#pragma unroll
  for (int k = 0; k < kPrepChunks; ++k) {
    const int v = lane + 32 * k;
    if (v < d / 8) r.x[k] = reinterpret_cast<const uint4 *>(src)[v];
  }
}

// y[0..d) = row / sqrt(mean(row^2) + eps) * w (w null: 1), in this warp's shared buffer.
__device__ void normalise_row(float *y, const RowRegs &r, int d, float eps, const MulRegs *w,
                              int lane) {
  float f[kPrepChunks][8];
  float ss = 0.f;
#pragma unroll
  for (int k = 0; k < kPrepChunks; ++k) {
    const int v = lane + 32 * k;
    if (v >= d / 8) continue;
    const uint32_t u[4] = {r.x[k].x, r.x[k].y, r.x[k].z, r.x[k].w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      f[k][2 * e] = bf16_bits_to_float((uint16_t)(u[e] & 0xffffu));
      f[k][2 * e + 1] = bf16_bits_to_float((uint16_t)(u[e] >> 16));
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) ss = fmaf(f[k][e], f[k][e], ss);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
  const float inv = 1.f / sqrtf(ss / (float)d + eps);
#pragma unroll
  for (int k = 0; k < kPrepChunks; ++k) {
    const int v = lane + 32 * k;
    if (v >= d / 8) continue;
#pragma unroll
    for (int e = 0; e < 8; ++e) y[8 * v + e] = w ? f[k][e] * inv * mul_at(*w, k, e) : f[k][e] * inv;
  }
  __syncwarp();
}

// The rotation angles of this lane's pairs i = lane, lane + 32, ... (< rot / 2).
struct PairAngles {
  float c[kPrepPairs], s[kPrepPairs];
};

__device__ __forceinline__ void load_angles(PairAngles &g, const PrepArgs &a, int pos, int lane) {
  const int half = a.rot / 2;
#pragma unroll
  for (int k = 0; k < kPrepPairs; ++k) {
    const int i = lane + 32 * k;
    if (i < half) {
      g.c[k] = a.rope_cos[(size_t)pos * half + i];
      g.s[k] = a.rope_sin[(size_t)pos * half + i];
    }
  }
}

// Turn the first rot columns of y as pairs (i, i + rot/2).
__device__ void rotate_row(float *y, const PairAngles &g, int rot, int lane) {
  const int half = rot / 2;
#pragma unroll
  for (int k = 0; k < kPrepPairs; ++k) {
    const int i = lane + 32 * k;
    if (i < half) {
      const float x0 = y[i], x1 = y[i + half];
      y[i] = x0 * g.c[k] - x1 * g.s[k];
      y[i + half] = x1 * g.c[k] + x0 * g.s[k];
    }
  }
  __syncwarp();
}

// Store y[0..cols) as bf16 at dst (16-byte vectors); scale columns >= from by mul if given.
__device__ void store_row(uint16_t *dst, const float *y, int cols, const MulRegs *mul, int from,
                          int lane) {
#pragma unroll
  for (int k = 0; k < kPrepChunks; ++k) {
    const int v = lane + 32 * k;
    if (v >= cols / 8) continue;
    uint32_t w[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int i0 = 8 * v + 2 * e, i1 = i0 + 1;
      const float f0 = (mul && i0 >= from) ? y[i0] * mul_at(*mul, k, 2 * e) : y[i0];
      const float f1 = (mul && i1 >= from) ? y[i1] * mul_at(*mul, k, 2 * e + 1) : y[i1];
      w[e] = (uint32_t)float_to_bf16_bits(f0) | ((uint32_t)float_to_bf16_bits(f1) << 16);
    }
    reinterpret_cast<uint4 *>(dst)[v] = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

// Every global load that does not depend on another is issued before the first
// use: the row's bytes and the token's (row, key) together, then the position
// (and the page), then the angles, so a token costs two or three memory round
// trips rather than one per step.
__global__ void __launch_bounds__(kPrepWarps * 32) pskv_prep_append(const PrepArgs a) {
  __shared__ float rows[kPrepWarps][kPrepMaxD];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int slots = a.num_q_heads + a.num_kv_heads;
  const long long item = (long long)blockIdx.x * kPrepWarps + warp;
  pdl_wait();
  pdl_launch_dependents();
  if (item >= (long long)a.n * slots) return;
  const int t = (int)(item / slots), s = (int)(item % slots);
  const bool is_q = s < a.num_q_heads;
  const int h = is_q ? s : s - a.num_q_heads;
  float *y = rows[warp];
  const uint16_t *xrow = static_cast<const uint16_t *>(a.x) + (size_t)t * (size_t)a.x_stride;
  RowRegs xr, vr;
  MulRegs wr, fold;  // the row's norm multiplier; K's, for a folded query's columns past rot
  load_row_regs(xr, xrow + (is_q ? a.q_col : a.k_col) + (size_t)h * a.d, a.d, lane);
  if (!is_q) load_row_regs(vr, xrow + a.v_col + (size_t)h * a.d, a.d, lane);
  const float *w = is_q ? a.w_q : a.w_k;
  if (w) load_mul_regs(wr, w, a.d, lane);
  const bool fold_q = is_q && a.folded;
  if (fold_q) load_mul_regs(fold, a.w_k, a.d, lane);
  const int b = a.row_of[t], key = a.pos_of[t];
  const bool row_ok = b >= 0 && b < a.batch && key >= 0;
  // the token's page slot (key rows only), checked like an append
  int lease = 0, page = -1;
  if (!is_q && row_ok) {
    lease = a.pages_of_row[b];
    const long long slot = key / a.page_size;
    page = slot < a.table_stride ? a.page_tables[(size_t)b * a.table_stride + slot] : -1;
  }
  const long long pos_ll =
      (long long)key + ((a.first_pos != nullptr && row_ok) ? a.first_pos[b] : 0);
  if (!row_ok || pos_ll < 0 || pos_ll >= a.max_pos) {
    if (lane == 0 && s == 0)
      raise_fault(a.status, row_ok ? PSKV_FAULT_BAD_POSITION : PSKV_FAULT_PAST_PAGES);
    return;
  }
  const int pos = (int)pos_ll;
  PairAngles ang;
  if (a.rot > 0) load_angles(ang, a, pos, lane);
  if (is_q) {
    normalise_row(y, xr, a.d, a.eps, w ? &wr : nullptr, lane);
    if (a.rot > 0) rotate_row(y, ang, a.rot, lane);
    uint16_t *dst = static_cast<uint16_t *>(a.q_out) + ((size_t)t * a.num_q_heads + h) * a.d;
    store_row(dst, y, a.d, fold_q ? &fold : nullptr, a.rot, lane);
    return;
  }
  if (lease < 0 || lease > a.table_stride || (long long)key >= (long long)lease * a.page_size) {
    if (lane == 0 && h == 0) raise_fault(a.status, PSKV_FAULT_PAST_PAGES);
    return;
  }
  if (page < 0 || (long long)page >= a.num_pages) {
    if (lane == 0 && h == 0) raise_fault(a.status, PSKV_FAULT_BAD_PAGE);
    return;
  }
  const size_t dst_row = ((size_t)page * a.num_kv_heads + h) * a.page_size + key % a.page_size;
  normalise_row(y, xr, a.d, a.eps, w ? &wr : nullptr, lane);
  if (a.rot > 0) rotate_row(y, ang, a.rot, lane);
  store_row(static_cast<uint16_t *>(a.k_pool) + dst_row * a.k_cols, y, a.k_cols, nullptr, 0, lane);
  __syncwarp();
  normalise_row(y, vr, a.d, a.eps, nullptr, lane);
  store_row(static_cast<uint16_t *>(a.v_pool) + dst_row * a.d, y, a.d, nullptr, 0, lane);
}

cudaError_t launch_prep(const PrepArgs &a, cudaStream_t s) {
  if (a.d > kPrepMaxD) return cudaErrorInvalidValue;
  const long long items = (long long)a.n * (a.num_q_heads + a.num_kv_heads);
  const long long blocks = (items + kPrepWarps - 1) / kPrepWarps;
  if (blocks <= 0) return cudaSuccess;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
  return launch_pdl(pskv_prep_append, dim3((unsigned)blocks), dim3(kPrepWarps * 32), 0, s, a);
}

}  // namespace pskv
