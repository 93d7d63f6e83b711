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
constexpr int kMaxStates = 64;  // group states of a row (level 2)
constexpr int kChunk = 16;      // partials of a group, loaded together (all loads in flight at once)

// Both levels in one launch, one block per (row, 64 or 128 output columns).
// Thread (c, j) of a block owns float4 column c of the block's columns and folds
// the groups j, j + L, ... of the row's partials (L = threads per column): it
// loads a group's (m, l) and its column's numerators all at once (one memory
// round trip; every thread of a group reads the same (m, l), which the
// hardware serves as one broadcast), computes the group's weights
// w_i = e^(m_i - M_g) itself and folds the group in index order (level 1) into
// a shared-memory group state.  One thread per column then folds the group
// states in index order and normalises (level 2).  The group states never
// leave the chip, every step's order is fixed, and the weights and sums are
// computed identically by every thread that needs them, so the result is
// deterministic.  An empty state's o is loaded but never used.
// Four blocks per SM (128 registers a thread, no spills): a call with many
// rows (a verify window's tokens x query heads) runs its blocks in fewer waves.
template <int kColsPerBlock>
__global__ void __launch_bounds__(kMergeThreads, 4) pskv_merge_cols(const MergeArgs a) {
  constexpr int kGroupLanes = kMergeThreads / kColsPerBlock;  // threads per column
  __shared__ float Mg_s[kMaxStates], Lg_s[kMaxStates];  // group states (m, l)
  __shared__ int bad_s;
  // the group numerators of the block's columns, [ng][kColsPerBlock]: sized by
  // the launch (2 KB for four groups), so that a merge block launched early fits
  // on an SM beside the partial kernel's CTAs
  extern __shared__ float4 o1_s[];
  const int row = blockIdx.x;
  const int c = threadIdx.x % kColsPerBlock, j = threadIdx.x / kColsPerBlock;
  const int dv4 = a.dv / 4, d4 = blockIdx.y * kColsPerBlock + c;
  const int d4c = d4 < dv4 ? d4 : dv4 - 1;  // columns past dv load a real column, never stored
  const int P = a.count, G = a.group, ng = (P + G - 1) / G;
  const float *m = a.m + (size_t)row * P, *l = a.l + (size_t)row * P;
  const float *o = a.o + (size_t)row * P * a.dv;
  if (threadIdx.x == 0) bad_s = 0;
  pdl_wait();
  pdl_launch_dependents();
  bool bad = false;
  // ---- level 1: this thread's groups, each in one round trip
  for (int g = j; g < ng; g += kGroupLanes) {
    const int i0 = g * G, n = min(P, i0 + G) - i0;
    float mi[kChunk], li[kChunk];
    float4 v[kChunk];
#pragma unroll
    for (int k = 0; k < kChunk; ++k)
      if (k < n) {
        mi[k] = m[i0 + k];
        li[k] = l[i0 + k];
        v[k] = __ldg(reinterpret_cast<const float4 *>(o + (size_t)(i0 + k) * a.dv) + d4c);
      }
    float M = -CUDART_INF_F;
#pragma unroll
    for (int k = 0; k < kChunk; ++k)
      if (k < n) {
        if (isnan(mi[k]) || (mi[k] == -CUDART_INF_F && li[k] != 0.f)) {
          bad = true;
          mi[k] = -CUDART_INF_F;  // an invalid state counts as empty
        }
        M = fmaxf(M, mi[k]);
      }
    float L = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int k = 0; k < kChunk; ++k)
      if (k < n && mi[k] != -CUDART_INF_F) {  // empty states: skipped by selection
        const float w = exp2f((mi[k] - M) * kLog2e);
        L = fmaf(li[k], w, L);
        acc.x = fmaf(v[k].x, w, acc.x);
        acc.y = fmaf(v[k].y, w, acc.y);
        acc.z = fmaf(v[k].z, w, acc.z);
        acc.w = fmaf(v[k].w, w, acc.w);
      }
    o1_s[g * kColsPerBlock + c] = acc;
    if (c == 0) {
      Mg_s[g] = M;
      Lg_s[g] = L;
    }
  }
  if (bad) bad_s = 1;
  __syncthreads();
  // ---- level 2 and normalisation, one thread per column
  if (j == 0 && d4 < dv4) {
    float M = -CUDART_INF_F;
    for (int g = 0; g < ng; ++g) M = fmaxf(M, Mg_s[g]);
    float L = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int g = 0; g < ng; ++g) {
      const float mg = Mg_s[g];
      if (mg != -CUDART_INF_F) {
        const float w = exp2f((mg - M) * kLog2e);
        const float4 x = o1_s[g * kColsPerBlock + c];
        L = fmaf(Lg_s[g], w, L);
        acc.x = fmaf(x.x, w, acc.x);
        acc.y = fmaf(x.y, w, acc.y);
        acc.z = fmaf(x.z, w, acc.z);
        acc.w = fmaf(x.w, w, acc.w);
      }
    }
    const bool empty_row = (M == -CUDART_INF_F);
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
  if (threadIdx.x == 0 && bad_s) raise_fault(a.status, PSKV_FAULT_BAD_STATE);
}

cudaError_t launch_merge(const MergeArgs &a, cudaStream_t s, int *launches) {
  *launches = 0;
  const int ng = (a.count + a.group - 1) / a.group;
  if (ng > kMaxStates || a.count > PSKV_MAX_SPLITS || a.group > kChunk) return cudaErrorInvalidValue;
  *launches = 1;
  if (ng <= kMergeThreads / 32) {  // every group lane busy with 32 columns per block
    const int chunks = (a.dv / 4 + 31) / 32;
    return launch_pdl(pskv_merge_cols<32>, dim3(a.rows, chunks), dim3(kMergeThreads),
                      (size_t)ng * 32 * sizeof(float4), s, a);
  }
  const int chunks = (a.dv / 4 + 15) / 16;
  return launch_pdl(pskv_merge_cols<16>, dim3(a.rows, chunks), dim3(kMergeThreads),
                    (size_t)ng * 16 * sizeof(float4), s, a);
}

}  // namespace pskv
