// merge.cu -- the two-level merge of split-KV partials.
//
// Each partial is an online-softmax state (m, l, o[dv]) in units of the scaled
// score.  States are combined by the exact rescaling identity (gem "Parked
// D512 fused split-KV decode design", "Candidate ownership and storage"):
//   M = max_i m_i,  l = sum_i l_i e^(m_i - M),  o = sum_i o_i e^(m_i - M),
// which is the pairwise identity applied to all states of a set at once.
// Level 1 folds groups of up to PSKV_MERGE_GROUP partials of a row into
// separate group states (pegainfer #1055 folded a group into its own first
// slot and needed a barrier between the group reads and the store; here the
// group states live in shared memory apart from the partials, so that race
// cannot occur).  Level 2 folds the group states of a row and writes
// out = o / l.  Folding order is fixed (index order), so the result is
// deterministic.  An empty state (m = -inf) contributes nothing and its o is
// never used; an empty state that carries l != 0 (or a NaN m) is flagged
// PSKV_FAULT_BAD_STATE and treated as empty.
#include <math_constants.h>

#include "pskv_internal.cuh"

namespace pskv {

constexpr int kMergeThreads = 128;
constexpr int kMaxStates = 64;  // states one warp weighs: groups of a row, or partials of a group
constexpr int kChunk = 16;      // states whose o is loaded together (all loads in flight at once)

// One warp reads n <= 64 states' (m, l) in parallel and computes the weights
// w_i = e^(m_i - M) (-1 marks an empty state, whose o is skipped), M and l.
// Every lane returns M and L; the weights go to w_s[0..n).
template <bool kCoherent = false>
__device__ __forceinline__ void warp_state_weights(const float *m, const float *l, int n,
                                                   float *w_s, float &M_out, float &L_out,
                                                   int32_t *status, int lane) {
  float mi[kMaxStates / 32], li[kMaxStates / 32];
  bool bad = false;
  float M = -CUDART_INF_F;
#pragma unroll
  for (int k = 0; k < kMaxStates / 32; ++k) {
    const int i = lane + 32 * k;
    mi[k] = i < n ? (kCoherent ? __ldcg(m + i) : m[i]) : -CUDART_INF_F;
    li[k] = i < n ? (kCoherent ? __ldcg(l + i) : l[i]) : 0.f;
    if (isnan(mi[k]) || (mi[k] == -CUDART_INF_F && li[k] != 0.f)) {
      bad = true;
      mi[k] = -CUDART_INF_F;  // an invalid state counts as empty
    }
    M = fmaxf(M, mi[k]);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  float L = 0.f;
#pragma unroll
  for (int k = 0; k < kMaxStates / 32; ++k) {
    const int i = lane + 32 * k;
    const bool empty = mi[k] == -CUDART_INF_F;
    const float w = empty ? 0.f : exp2f((mi[k] - M) * kLog2e);
    if (i < n) w_s[i] = empty ? -1.f : w;
    // fixed-order sum: lane partials, then a butterfly (same bits every run)
    if (!empty) L = fmaf(li[k], w, L);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) L += __shfl_xor_sync(0xffffffffu, L, off);
  if (__any_sync(0xffffffffu, bad) && lane == 0) raise_fault(status, PSKV_FAULT_BAD_STATE);
  M_out = M;
  L_out = L;
}

// Load o_i[d4] of states [i0, i0 + kChunk) (those below n), all in flight at once.
// The values of empty states are loaded too but never used (their o may be
// uninitialised); loading them keeps the loads independent of the weights, so
// they overlap the (m, l) loads.  kCoherent reads through L2 only (for data
// other blocks of this grid just wrote).
template <bool kCoherent>
__device__ __forceinline__ void load_chunk(const float *o, int n, int dv, int d4, int i0,
                                           float4 (&v)[kChunk]) {
#pragma unroll
  for (int k = 0; k < kChunk; ++k)
    if (i0 + k < n) {
      const float4 *src = reinterpret_cast<const float4 *>(o + (size_t)(i0 + k) * dv) + d4;
      v[k] = kCoherent ? __ldcg(src) : __ldg(src);
    }
}

// acc += w_i v[i - i0] over the chunk's states, in index order; empty states
// (w < 0) are skipped by selection, so whatever their o holds never reaches acc.
__device__ __forceinline__ void combine_chunk(float4 &acc, const float4 (&v)[kChunk], int n,
                                              int i0, const float *w_s) {
#pragma unroll
  for (int k = 0; k < kChunk; ++k) {
    if (i0 + k < n) {
      const float w = w_s[i0 + k];
      if (w >= 0.f) {
        acc.x = fmaf(v[k].x, w, acc.x);
        acc.y = fmaf(v[k].y, w, acc.y);
        acc.z = fmaf(v[k].z, w, acc.z);
        acc.w = fmaf(v[k].w, w, acc.w);
      }
    }
  }
}

// Both levels in one launch, one block per (row, 64 or 128 output columns).  Every
// block computes the row's level-1 weights (warp w takes groups w, w + 4, ...)
// and the level-2 weights over the group states; its threads fold, for their
// column, each group of partials in index order into a shared-memory group
// accumulator (level 1), then one thread per column folds the group results
// in index order and normalises (level 2).  The group results never leave the
// chip, and the arithmetic and its order are those of two separate levels.
// The first group's numerators are loaded before any weight is known.
// kCols float4 columns per block (16, or 32 when a row has at most 4 groups:
// then no thread of the block idles), kMergeThreads / kCols threads per column.
template <int kColsPerBlock>
__global__ void __launch_bounds__(kMergeThreads) pskv_merge_cols(const MergeArgs a) {
  constexpr int kGroupLanes = kMergeThreads / kColsPerBlock;  // threads per column
  __shared__ float w_s[PSKV_MAX_SPLITS];             // level-1 weights, by partial
  __shared__ float m_s[PSKV_MAX_SPLITS], l_s[PSKV_MAX_SPLITS];  // the row's partial (m, l)
  __shared__ float Mg_s[kMaxStates], Lg_s[kMaxStates], wg_s[kMaxStates];  // group states
  __shared__ float4 o1_s[kMaxStates][kColsPerBlock];  // group numerators of this block's columns
  __shared__ float M_s, L_s;
  const int row = blockIdx.x;
  const int c = threadIdx.x % kColsPerBlock, j = threadIdx.x / kColsPerBlock;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int dv4 = a.dv / 4, d4 = blockIdx.y * kColsPerBlock + c;
  const int P = a.count, G = a.group, ng = (P + G - 1) / G;
  const float *m = a.m + (size_t)row * P, *l = a.l + (size_t)row * P;
  const float *o = a.o + (size_t)row * P * a.dv;
  pdl_wait();
  pdl_launch_dependents();
  float4 v[kChunk];
  if (j < ng && d4 < dv4) load_chunk<false>(o, min(P, j * G + G), a.dv, d4, j * G, v);
  // every (m, l) of the row in one round trip, staged in shared memory
  for (int i = threadIdx.x; i < P; i += kMergeThreads) {
    m_s[i] = m[i];
    l_s[i] = l[i];
  }
  __syncthreads();
  // level-1 weights and group states
  for (int g = warp; g < ng; g += kMergeThreads / 32) {
    const int i0 = g * G, n = min(P, i0 + G) - i0;
    float Mg, Lg;
    warp_state_weights<false>(m_s + i0, l_s + i0, n, w_s + i0, Mg, Lg, a.status, lane);
    if (lane == 0) {
      Mg_s[g] = Mg;
      Lg_s[g] = Lg;
    }
  }
  __syncthreads();
  // level-2 weights (warp 0) while every thread folds its groups (level 1)
  if (warp == 0) {
    float M, L;
    warp_state_weights<false>(Mg_s, Lg_s, ng, wg_s, M, L, a.status, lane);
    if (lane == 0) {
      M_s = M;
      L_s = L;
    }
  }
  if (d4 < dv4) {
    for (int g = j; g < ng; g += kGroupLanes) {
      const int i0 = g * G, end = min(P, i0 + G);
      if (g != j) load_chunk<false>(o, end, a.dv, d4, i0, v);
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      combine_chunk(acc, v, end, i0, w_s);
      o1_s[g][c] = acc;
    }
  }
  __syncthreads();
  // level 2 and normalisation, one thread per column
  if (j == 0 && d4 < dv4) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int g = 0; g < ng; ++g) {
      const float w = wg_s[g];
      if (w >= 0.f) {
        const float4 x = o1_s[g][c];
        acc.x = fmaf(x.x, w, acc.x);
        acc.y = fmaf(x.y, w, acc.y);
        acc.z = fmaf(x.z, w, acc.z);
        acc.w = fmaf(x.w, w, acc.w);
      }
    }
    const bool empty_row = (M_s == -CUDART_INF_F);
    const float L = L_s;
    const float4 r = empty_row ? make_float4(0.f, 0.f, 0.f, 0.f)
                               : make_float4(acc.x / L, acc.y / L, acc.z / L, acc.w / L);
    if (a.out_dtype == PSKV_DTYPE_BF16) {
      uint2 packed;
      packed.x = pack_bf16x2(r.x, r.y);
      packed.y = pack_bf16x2(r.z, r.w);
      reinterpret_cast<uint2 *>(static_cast<char *>(a.out) + (size_t)row * a.dv * 2)[d4] = packed;
    } else {
      reinterpret_cast<float4 *>(static_cast<char *>(a.out) + (size_t)row * a.dv * 4)[d4] = r;
    }
    if (empty_row && d4 == 0) raise_fault(a.status, PSKV_FAULT_EMPTY_ROW);
  }
}

cudaError_t launch_merge(const MergeArgs &a, cudaStream_t s, int *launches) {
  *launches = 0;
  const int ng = (a.count + a.group - 1) / a.group;
  if (ng > kMaxStates || a.count > PSKV_MAX_SPLITS || a.group > kChunk) return cudaErrorInvalidValue;
  *launches = 1;
  if (ng <= kMergeThreads / 32) {  // every group lane busy with 32 columns per block
    const int chunks = (a.dv / 4 + 31) / 32;
    return launch_pdl(pskv_merge_cols<32>, dim3(a.rows, chunks), dim3(kMergeThreads), 0, s, a);
  }
  const int chunks = (a.dv / 4 + 15) / 16;
  return launch_pdl(pskv_merge_cols<16>, dim3(a.rows, chunks), dim3(kMergeThreads), 0, s, a);
}

}  // namespace pskv
