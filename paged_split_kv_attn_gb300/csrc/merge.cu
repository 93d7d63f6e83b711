// merge.cu -- the two-level merge of split-KV partials.
//
// Each partial is an online-softmax state (m, l, o[dv]) in units of the scaled
// score.  States are combined by the exact rescaling identity (gem "Parked
// D512 fused split-KV decode design", "Candidate ownership and storage"):
//   M = max_i m_i,  l = sum_i l_i e^(m_i - M),  o = sum_i o_i e^(m_i - M),
// which is the pairwise identity applied to all states of a set at once.
// Level 1 folds groups of up to PSKV_MERGE_GROUP partials of a row into a
// SEPARATE buffer (pegainfer #1055 folded a group into its own first slot and
// needed a barrier between the group reads and the store; writing elsewhere
// removes that race by construction).  Level 2 folds the group results of a
// row and writes out = o / l.  Folding order is fixed (index order), so the
// result is deterministic.  An empty state (m = -inf) contributes nothing and
// its o is never used; an empty state that carries l != 0 (or a NaN m) is
// flagged PSKV_FAULT_BAD_STATE and treated as empty.
#include <math_constants.h>

#include "pskv_internal.cuh"

namespace pskv {

constexpr int kMergeThreads = 128;
constexpr int kMaxStates = 64;  // states one level-2 block folds (PSKV_MAX_SPLITS / PSKV_MERGE_GROUP)
constexpr int kChunk = 16;      // states whose o is loaded together (all loads in flight at once)

// Warp 0 reads the n states' (m, l) in parallel and computes the weights
// w_i = e^(m_i - M) (-1 marks an empty state, whose o is skipped), M and l.
template <bool kCoherent = false>
__device__ void state_weights(const float *m, const float *l, int n, float *w_s, float *M_s,
                              float *L_s, int32_t *status) {
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
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
    if (lane == 0) {
      *M_s = M;
      *L_s = L;
    }
  }
  __syncthreads();
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

// Fold the n states of one row: (m, l) weights by warp 0, o by every thread,
// with the first chunk of each thread's first column loaded before the weights.
// Calls f(d4, acc) for every column d4 of the row.
template <bool kCoherent, class F>
__device__ __forceinline__ void fold_states(const float *m, const float *l, const float *o, int n,
                                            int dv, float *w_s, float *M_s, float *L_s,
                                            int32_t *status, F &&f) {
  const int dv4 = dv / 4;
  float4 v[kChunk];
  if ((int)threadIdx.x < dv4) load_chunk<kCoherent>(o, n, dv, threadIdx.x, 0, v);
  state_weights<kCoherent>(m, l, n, w_s, M_s, L_s, status);
  for (int d4 = threadIdx.x; d4 < dv4; d4 += blockDim.x) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int i0 = 0; i0 < n; i0 += kChunk) {
      if (d4 != (int)threadIdx.x || i0 != 0) load_chunk<kCoherent>(o, n, dv, d4, i0, v);
      combine_chunk(acc, v, n, i0, w_s);
    }
    f(d4, acc);
  }
}

// grid (groups, rows): fold partials [grp*group, min(count, (grp+1)*group)) of a row.
__global__ void __launch_bounds__(kMergeThreads) pskv_merge_level1(const MergeArgs a) {
  __shared__ float w_s[kMaxStates];
  __shared__ float M_s, L_s;
  const int grp = blockIdx.x, row = blockIdx.y;
  const int ng = (a.count + a.group - 1) / a.group;
  const int p0 = grp * a.group;
  const int n = min(a.count - p0, a.group);
  const size_t base = (size_t)row * a.count + p0;
  const size_t out_state = (size_t)row * ng + grp;
  pdl_wait();
  pdl_launch_dependents();
  fold_states<false>(a.m + base, a.l + base, a.o + base * a.dv, n, a.dv, w_s, &M_s, &L_s,
                     a.status, [&](int d4, float4 acc) {
                       reinterpret_cast<float4 *>(a.o1 + out_state * a.dv)[d4] = acc;
                     });
  if (threadIdx.x == 0) {
    a.m1[out_state] = M_s;
    a.l1[out_state] = L_s;
  }
}

// Fold all `n` states of `row` and write the normalised output row.
template <bool kCoherent>
__device__ void fold_and_finalize(const float *m, const float *l, const float *o, int n, int row,
                                  const MergeArgs &a, float *w_s, float &M_s, float &L_s) {
  const size_t base = (size_t)row * n;
  fold_states<kCoherent>(m + base, l + base, o + base * a.dv, n, a.dv, w_s, &M_s, &L_s, a.status,
                         [&](int d4, float4 acc) {
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
  });
  if (threadIdx.x == 0 && M_s == -CUDART_INF_F) raise_fault(a.status, PSKV_FAULT_EMPTY_ROW);
}

// grid (rows): fold all `n` states of a row and normalise.
__global__ void __launch_bounds__(kMergeThreads) pskv_merge_level2(const float *m, const float *l,
                                                                   const float *o, int n,
                                                                   const MergeArgs a) {
  __shared__ float w_s[kMaxStates];
  __shared__ float M_s, L_s;
  pdl_wait();
  pdl_launch_dependents();
  fold_and_finalize<false>(m, l, o, n, blockIdx.x, a, w_s, M_s, L_s);
}

// Both levels in one launch, grid (groups, rows): each block folds one group
// of partials (level 1) into the group buffer; the block that finishes a row's
// last group (counted on a per-row counter that the partial kernel zeroed)
// folds that row's group results (level 2).  The level-2 fold reads the group
// buffer in index order, so which block finishes last does not change a bit.
__global__ void __launch_bounds__(kMergeThreads) pskv_merge_two_level(const MergeArgs a) {
  __shared__ float w_s[kMaxStates];
  __shared__ float M_s, L_s;
  __shared__ bool last_s;
  const int grp = blockIdx.x, row = blockIdx.y;
  const int ng = (a.count + a.group - 1) / a.group;
  const int p0 = grp * a.group;
  const int n = min(a.count - p0, a.group);
  const size_t base = (size_t)row * a.count + p0;
  pdl_wait();
  pdl_launch_dependents();
  const size_t out_state = (size_t)row * ng + grp;
  fold_states<false>(a.m + base, a.l + base, a.o + base * a.dv, n, a.dv, w_s, &M_s, &L_s,
                     a.status, [&](int d4, float4 acc) {
                       reinterpret_cast<float4 *>(a.o1 + out_state * a.dv)[d4] = acc;
                     });
  if (threadIdx.x == 0) {
    a.m1[out_state] = M_s;
    a.l1[out_state] = L_s;
  }
  // publish this group's result, then count it
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) last_s = atomicAdd(a.counters + row, 1u) == (unsigned)(ng - 1);
  __syncthreads();
  if (!last_s) return;
  __threadfence();
  fold_and_finalize<true>(a.m1, a.l1, a.o1, ng, row, a, w_s, M_s, L_s);
}

cudaError_t launch_merge(const MergeArgs &a, cudaStream_t s, int *launches) {
  *launches = 0;
  if (a.count <= a.group) {  // one group: the second level reads the partials directly
    *launches = 1;
    return launch_pdl(pskv_merge_level2, dim3(a.rows), dim3(kMergeThreads), 0, s, a.m, a.l, a.o,
                      a.count, a);
  }
  const int ng = (a.count + a.group - 1) / a.group;
  if (a.counters != nullptr) {  // both levels in one launch
    *launches = 1;
    return launch_pdl(pskv_merge_two_level, dim3(ng, a.rows), dim3(kMergeThreads), 0, s, a);
  }
  cudaError_t e = launch_pdl(pskv_merge_level1, dim3(ng, a.rows), dim3(kMergeThreads), 0, s, a);
  if (e != cudaSuccess) return e;
  *launches = 2;
  return launch_pdl(pskv_merge_level2, dim3(a.rows), dim3(kMergeThreads), 0, s,
                    (const float *)a.m1, (const float *)a.l1, (const float *)a.o1, ng, a);
}

}  // namespace pskv
