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
// its o is never read; an empty state that carries l != 0 (or a NaN m) is
// flagged PSKV_FAULT_BAD_STATE and treated as empty.
#include <math_constants.h>

#include "pskv_internal.cuh"

namespace pskv {

constexpr int kMergeThreads = 128;
constexpr int kMaxStates = 64;  // states one level-2 block folds (PSKV_MAX_SPLITS / PSKV_MERGE_GROUP)

// Weights e^(m_i - M) of `n` states (thread 0 computes; the block reads them).
__device__ void state_weights(const float *m, const float *l, int n, float *w_s, float *M_s,
                              float *L_s, int32_t *status) {
  if (threadIdx.x == 0) {
    float M = -CUDART_INF_F;
    bool bad = false;
    for (int i = 0; i < n; ++i) {
      const float mi = m[i];
      if (isnan(mi) || (mi == -CUDART_INF_F && l[i] != 0.f)) bad = true;
      else M = fmaxf(M, mi);
    }
    float L = 0.f;
    for (int i = 0; i < n; ++i) {
      const float mi = m[i];
      const bool empty = isnan(mi) || mi == -CUDART_INF_F;
      const float w = empty ? 0.f : exp2f((mi - M) * kLog2e);
      w_s[i] = empty ? -1.f : w;  // -1 marks "skip this state's o"
      if (!empty) L = fmaf(l[i], w, L);
    }
    if (bad) raise_fault(status, PSKV_FAULT_BAD_STATE);
    *M_s = M;
    *L_s = L;
  }
  __syncthreads();
}

// grid (groups, rows): fold partials [grp*group, min(count, (grp+1)*group)) of a row.
__global__ void __launch_bounds__(kMergeThreads) pskv_merge_level1(const MergeArgs a) {
  __shared__ float w_s[PSKV_MERGE_GROUP];
  __shared__ float M_s, L_s;
  const int grp = blockIdx.x, row = blockIdx.y;
  const int ng = (a.count + a.group - 1) / a.group;
  const int p0 = grp * a.group;
  const int n = min(a.count - p0, a.group);
  const size_t base = (size_t)row * a.count + p0;
  state_weights(a.m + base, a.l + base, n, w_s, &M_s, &L_s, a.status);
  const size_t out_state = (size_t)row * ng + grp;
  if (threadIdx.x == 0) {
    a.m1[out_state] = M_s;
    a.l1[out_state] = L_s;
  }
  const int dv4 = a.dv / 4;
  for (int d4 = threadIdx.x; d4 < dv4; d4 += blockDim.x) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int i = 0; i < n; ++i) {
      const float w = w_s[i];
      if (w < 0.f) continue;
      const float4 v = reinterpret_cast<const float4 *>(a.o + (base + i) * a.dv)[d4];
      acc.x = fmaf(v.x, w, acc.x);
      acc.y = fmaf(v.y, w, acc.y);
      acc.z = fmaf(v.z, w, acc.z);
      acc.w = fmaf(v.w, w, acc.w);
    }
    reinterpret_cast<float4 *>(a.o1 + out_state * a.dv)[d4] = acc;
  }
}

// grid (rows): fold all `n` states of a row and normalise.
__global__ void __launch_bounds__(kMergeThreads) pskv_merge_level2(const float *m, const float *l,
                                                                   const float *o, int n,
                                                                   const MergeArgs a) {
  __shared__ float w_s[kMaxStates];
  __shared__ float M_s, L_s;
  const int row = blockIdx.x;
  const size_t base = (size_t)row * n;
  state_weights(m + base, l + base, n, w_s, &M_s, &L_s, a.status);
  const bool empty_row = (M_s == -CUDART_INF_F);
  if (empty_row && threadIdx.x == 0) raise_fault(a.status, PSKV_FAULT_EMPTY_ROW);
  const float L = L_s;
  const int dv4 = a.dv / 4;
  for (int d4 = threadIdx.x; d4 < dv4; d4 += blockDim.x) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int i = 0; i < n; ++i) {
      const float w = w_s[i];
      if (w < 0.f) continue;
      const float4 v = reinterpret_cast<const float4 *>(o + (base + i) * a.dv)[d4];
      acc.x = fmaf(v.x, w, acc.x);
      acc.y = fmaf(v.y, w, acc.y);
      acc.z = fmaf(v.z, w, acc.z);
      acc.w = fmaf(v.w, w, acc.w);
    }
    float4 r;
    if (empty_row) {
      r = make_float4(0.f, 0.f, 0.f, 0.f);
    } else {
      r = make_float4(acc.x / L, acc.y / L, acc.z / L, acc.w / L);
    }
    if (a.out_dtype == PSKV_DTYPE_BF16) {
      uint2 packed;
      packed.x = pack_bf16x2(r.x, r.y);
      packed.y = pack_bf16x2(r.z, r.w);
      reinterpret_cast<uint2 *>(static_cast<char *>(a.out) + (size_t)row * a.dv * 2)[d4] = packed;
    } else {
      reinterpret_cast<float4 *>(static_cast<char *>(a.out) + (size_t)row * a.dv * 4)[d4] = r;
    }
  }
}

cudaError_t launch_merge(const MergeArgs &a, cudaStream_t s, int *launches) {
  *launches = 0;
  if (a.count <= a.group) {  // one group: the second level reads the partials directly
    pskv_merge_level2<<<a.rows, kMergeThreads, 0, s>>>(a.m, a.l, a.o, a.count, a);
    *launches = 1;
    return cudaGetLastError();
  }
  const int ng = (a.count + a.group - 1) / a.group;
  pskv_merge_level1<<<dim3(ng, a.rows), kMergeThreads, 0, s>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  pskv_merge_level2<<<a.rows, kMergeThreads, 0, s>>>(a.m1, a.l1, a.o1, ng, a);
  *launches = 2;
  return cudaGetLastError();
}

}  // namespace pskv
