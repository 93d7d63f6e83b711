// partial_kernel.cuh -- the split-KV partial kernel (decode, verify windows, prefill).
//
// One CTA computes the online-softmax partial of one (row b, KV head g,
// partition p[, column block]): for the query columns it serves (the G query
// heads that share KV head g, times the row's query tokens in a verify window
// or a prefill chunk) it streams the partition's keys and values once and
// keeps, per column, the running max m, the running sum l and the
// unnormalised numerator o (gem "Parked D512 fused split-KV decode design",
// "Candidate ownership and storage": one first-pass worker per (kv_head,
// partition), each K/V row staged once for all query heads of the group).
//
// Structure (GB300):
//  * the last warp is the producer: per 16-key tile it reads the tile's page id
//    from the table (32 ids per warp-wide load, so one table read serves up to
//    32 pages; TensorFold #1619 measured a per-key page lookup at +5.8..7.9 %
//    and moved it to once per tile) and issues bulk async copies
//    (cp.async.bulk, L2 evict-first) of the tile's valid key rows into a ring
//    of shared-memory stages, counted on the stage's "full" mbarrier.  When the
//    call carries the step's new K/V row, the CTA whose partition holds it
//    first writes it into its page;
//  * the other warps are consumers.  On the tensor-core path (bf16) they all
//    take every tile together (MmaConsumer, below); on the CUDA-core path
//    (f32 pools, 16 query heads per KV head) warp w takes tiles w, w+CW, ...
//    with its own (m, l, o), and the warp states are merged in shared memory
//    at the end (SimtConsumer);
//  * the partition's (m, l, o) per column goes to the workspace for the merge
//    kernel, or, when the call has a single partition, the CTA normalises and
//    writes its output itself.
// Keys outside a column's visible range (past its token, below a window bound,
// past the row) are masked: rows outside the CTA's key range are never copied,
// scores are set to -inf by selection and values masked to zero, so stale
// shared memory can never reach the result.
//
// Copy granularity: the bulk copy engine's per-copy cost dominates below
// about 2 KB (1 KB copies streamed at ~4.6 TB/s on GB300, 2 KB copies at
// ~7.1 TB/s), so key rows are copied in groups of R consecutive rows, one copy
// per group.  In shared memory each group is followed by 16 bytes of padding:
// with R = 2 and 1 KB rows, the 8 even keys of a tile start in 8 distinct
// 16-byte bank groups, and so do the 8 odd keys, which the tensor-core
// consumer exploits by ordering its MMA rows even keys first.
#pragma once

#include <math_constants.h>

#include "pskv_internal.cuh"

namespace pskv {

#ifndef PSKV_STAGE_BUDGET
#define PSKV_STAGE_BUDGET 100000  // shared-memory bytes given to the stage ring
#endif

// Ring of stages for `kWarps` consumer warps.  Warp w owns stages w, w + kWarps, ...
// (the stage count is a multiple of kWarps), so every stage is always consumed
// by the same warp, in order: a consumer never waits on a phase more than one
// ahead of its barrier's current phase.  Rows are copied in groups of kRows.
// kFixedStages > 0 sets the stage count directly (the budget then does not apply).
template <int kRowBytesK, int kRowBytesV, int kRows, int kWarps, int kFixedStages = 0>
struct RingGeom {
  static constexpr int kRowsPerCopy = kRows;
  static constexpr int kGroupStrideK = kRows * kRowBytesK + 16;
  static constexpr int kGroupStrideV = kRows * kRowBytesV + 16;
  static constexpr int kTileBytesK = (kKeyTile / kRows) * kGroupStrideK;
  static constexpr int kTileBytesV = (kKeyTile / kRows) * kGroupStrideV;
  static constexpr int kStageBytes = kTileBytesK + kTileBytesV;  // K tile then V tile
  static constexpr int kPerWarpFit = PSKV_STAGE_BUDGET / (kWarps * kStageBytes);
  static constexpr int kPerWarpMax = 8 / kWarps > 0 ? 8 / kWarps : 1;
  static constexpr int kPerWarp =
      kPerWarpFit < 1 ? 1 : (kPerWarpFit > kPerWarpMax ? kPerWarpMax : kPerWarpFit);
  static constexpr int kStages = kFixedStages > 0 ? kFixedStages : kWarps * kPerWarp;
  static constexpr int kRingBytes = kStages * kStageBytes;
  // byte offset of key row t (0..15) in a K tile and in a V tile
  static __device__ __forceinline__ int row_off_k(int t) {
    return (t / kRows) * kGroupStrideK + (t % kRows) * kRowBytesK;
  }
  static __device__ __forceinline__ int row_off_v(int t) {
    return (t / kRows) * kGroupStrideV + (t % kRows) * kRowBytesV;
  }
  static_assert(kKeyTile % kRows == 0, "row groups must divide the tile");
};

// -------------------------------------------------------------------------------------------
// Tensor-core consumer: bf16 K/V, query columns in n-tiles of 8.
// A column is one (query token, query head of the KV group): 8 heads of one
// token per n-tile in single-token decode, up to 16 columns per CTA for verify
// windows.  The consumer warps work on every tile together (one warp alone
// issues mma.sync too slowly to keep up with HBM):
//  1. scores: the head dimension is cut into four quarters; warp w forms the
//     partial scores S^T[16 keys x 8 columns] = K[:, dq] Q^T[dq, :] of n-tile
//     w % NT over quarter dq = w / NT (mma m16n8k16, keys as M so no row is
//     wasted);
//  2. the four quarters' partials of each n-tile are summed through shared
//     memory in a fixed order, so every warp holds the same S^T of every
//     column and runs the same online-softmax update;
//  3. warp w accumulates O^T[dw x cols] += V^T[dw x 16] P^T[16 x cols] over its
//     own slice dw of the head dimension (D / warps wide), with P^T obtained
//     from the S^T accumulator by movmatrix.trans.  P is applied as a bf16
//     hi+lo pair (p = hi + lo to ~2^-17 relative), so the weights keep nearly
//     fp32 accuracy while V stays bf16.
// With one n-tile that is four warps, each on a quarter of D for both steps;
// with two, eight warps: each warp's products, accumulators and dependency
// chain per tile stay as short as with one n-tile, and the score exchange
// grows only with the number of n-tiles.
// MMA row m holds key 2m (m < 8) or key 2(m-8)+1 (m >= 8): with rows stored in
// padded pairs, each 8x8 ldmatrix phase then reads 8 distinct bank groups.
// -------------------------------------------------------------------------------------------

// Stages per CTA of the tensor-core consumer.  Three stages per CTA, with as
// many CTAs per SM as shared memory allows (2 for split hd512 rows, 3 for
// folded ones), measured best on GB300: more stages per CTA left fewer CTAs
// to overlap their start-up and tail, fewer left too few bytes in flight.
#ifndef PSKV_MMA_STAGES
#define PSKV_MMA_STAGES 3
#endif

// bar.sync on a named barrier shared by the `n` threads of the consumer warps.
__device__ __forceinline__ void consumers_sync(int n) {
  asm volatile("bar.sync 1, %0;" ::"r"(n) : "memory");
}

// The same barrier with an AND vote: true iff `pred` holds in every consumer thread.
__device__ __forceinline__ bool consumers_all(int n, bool pred) {
  uint32_t out;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, 1, %2, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(out)
      : "r"((uint32_t)pred), "r"(n)
      : "memory");
  return out != 0;
}

// The step's new K/V row of table row b, KV head g (key `key`), copied into
// its page by one warp exactly as kv_append_rows would: the lease and the
// page id are checked first, a bad one flags the fault word and skips the
// copy.  The copy is made visible to the bulk-copy (async) proxy before the
// same warp loads any tile.
static __device__ void append_new_row(const PartialArgs &a, int b, int g, int key, int lane) {
  const int lease = a.append_pages[b];
  if (lease < 0 || lease > a.table_stride || (long long)key >= (long long)lease * a.page_size) {
    if (lane == 0) raise_fault(a.status, PSKV_FAULT_PAST_PAGES);
    return;
  }
  const int page = a.page_tables[(size_t)b * a.table_stride + key / a.page_size];
  if (page < 0 || (long long)page >= a.num_pages) {
    if (lane == 0) raise_fault(a.status, PSKV_FAULT_BAD_PAGE);
    return;
  }
  const size_t src = (size_t)b * a.num_kv_heads + g;
  const size_t dst = ((size_t)page * a.num_kv_heads + g) * a.page_size + key % a.page_size;
  const uint4 *ks = reinterpret_cast<const uint4 *>(static_cast<const char *>(a.append_k) +
                                                    src * a.k_row_bytes);
  const uint4 *vs = reinterpret_cast<const uint4 *>(static_cast<const char *>(a.append_v) +
                                                    src * a.v_row_bytes);
  uint4 *kd = reinterpret_cast<uint4 *>(static_cast<char *>(const_cast<void *>(a.k_pool)) +
                                        dst * a.k_row_bytes);
  uint4 *vd = reinterpret_cast<uint4 *>(static_cast<char *>(const_cast<void *>(a.v_pool)) +
                                        dst * a.v_row_bytes);
  for (int v = lane; v < a.k_row_bytes / 16; v += 32) kd[v] = ks[v];
  for (int v = lane; v < a.v_row_bytes / 16; v += 32) vd[v] = vs[v];
  asm volatile("fence.proxy.async.global;" ::: "memory");
  __syncwarp();
}

// The query tokens and keys one CTA serves: row b's tokens are query/output
// rows r0 .. r0 + T - 1; token t sits at key len - T + t and sees keys up to
// itself, from lo_fixed (a windowed decode's bound, else 0) or, with a
// per-token window, from its own key - window + 1.
struct RowPlan {
  int b, T, r0, len;
  int lo_fixed;
  int window;
};

// Columns past the window's tokens x G (G < 8 query heads per KV head, or a
// window that does not fill its last n-tile) have zero queries and are never
// written back.
// kFolded: the pool keeps only the first D/4 columns of K (the rotated quarter)
// and the folded query's other columns meet V's (pegainfer #1055, Description:
// the folded row holds K only where the rotation touches it, V in full, with
// K's norm weight folded into the query).  The warps scoring quarter 0 read
// their operands from the K tile, the others from the V tile.
// kTree: the query columns are tokens of a drafted tree; window keys are
// visible to a column by its token's ancestor mask (held in shared memory).
template <int kD, int kG = 8, bool kFolded = false, int kNT = 1, bool kTree = false>
struct MmaConsumer {
  using Elem = __nv_bfloat16;
  static constexpr int D = kD;
  static constexpr int G = kG;
  static_assert(kG == 1 || kG == 2 || kG == 4 || kG == 8, "query heads per KV head");
  // Window column j (of tokens x G) serves query token j / G, head j % G of the
  // KV group; CTA column block cb takes columns [cb * kCols, (cb + 1) * kCols).
  static constexpr int NT = kNT;
  static constexpr int kCols = 8 * kNT;
  static constexpr int kQuarters = 4;              // score partials per n-tile
  static constexpr int kWarps = kQuarters * kNT;
  // registers sized for two CTAs per SM (the compiler accounts for how the
  // warps spread over the SM's four register files: 96 per thread at 9 warps)
  static constexpr int kMinBlocks = 2;
  static constexpr bool kCooperative = true;       // every warp takes part in every tile
  static constexpr int DQ = D / kQuarters;         // score columns per warp
  static constexpr int KSQ = DQ / 16;              // k-steps of a warp's score product
  static constexpr int DW = D / kWarps;            // output columns per warp
  static constexpr int KSP = DW / 16;              // m-tiles of a warp's PV product
  // score accumulator chains (two when the second n-tile's state needs the registers)
  static constexpr int CH = (KSQ % 4 == 0 && kNT == 1) ? 4 : 2;
  static constexpr int kXchgBytes = 2 * kQuarters * NT * 32 * 16;  // double-buffered exchange
  static constexpr int kExtraSmem = kXchgBytes + (kTree ? kCols * 8 : 0);  // + tree masks
  static constexpr int kRowBytesK = (kFolded ? D / 4 : D) * 2;     // bytes of one stored K row
  static constexpr int kRowBytesV = D * 2;
  using Geom = RingGeom<kRowBytesK, kRowBytesV, 2, 1, PSKV_MMA_STAGES>;
  static constexpr int RBK = kRowBytesK, RBV = kRowBytesV;
  static constexpr int GSK = Geom::kGroupStrideK;  // bytes of a padded pair of K rows
  static constexpr int GSV = Geom::kGroupStrideV;  // bytes of a padded pair of V rows
  static_assert(KSQ % CH == 0 && KSP >= 1, "warp shares of the head dimension");

  uint32_t qf[KSQ][2];     // Q^T B-fragments of this warp's n-tile and quarter:
                           //   (d = dq0 + 16k + 2c + {0,1} [+8], column 8 nts + r)
  float o[NT][KSP][4];     // O^T accumulators: (d = dw0 + 16j + r [+8], columns 8nt + 2c, +1)
  float m0[NT], m1[NT];    // reference max (log2 units) of columns 8nt + 2c, +1: the same in every warp
  float l0[NT], l1[NT];    // this lane's share of the sums of those columns
  int lim0[NT], lim1[NT];  // keys below lim are visible to those columns (causal in a window)
  int lo_fixed, window;    // and keys from lo_fixed on, or from lim - window on with a window
  float scale_log2;
  float4 *xchg;            // [2][kQuarters][NT][32] partial scores
  const unsigned long long *tmask;  // [kCols] tree masks of the block's columns (kTree)
  int win0;                // the window's first key (len - tokens)
  int r, c, warp, tokens, cbase, r0;

  __device__ int nt_scored() const { return warp % NT; }  // the n-tile this warp scores
  __device__ int quarter() const { return warp / NT; }     // the quarter of D it scores over

  static __device__ void prologue(const PartialArgs &, int, int, unsigned char *) {}

  __device__ void init(const PartialArgs &a, const RowPlan &rp, int h0, int lane,
                       unsigned char *extra, int cb) {
    r = lane >> 2;
    c = lane & 3;
    warp = threadIdx.x >> 5;
    tokens = rp.T;
    r0 = rp.r0;
    lo_fixed = rp.lo_fixed;
    window = rp.window;
    cbase = cb * kCols;
    scale_log2 = a.scale_log2;
    xchg = reinterpret_cast<float4 *>(extra);
    win0 = rp.len - rp.T;
    if constexpr (kTree) {
      unsigned long long *tm = reinterpret_cast<unsigned long long *>(extra + kXchgBytes);
      tmask = tm;
      // Column i of the block takes its token's mask, cut to the tokens up to
      // itself; a mask without its own bit or with a later one is flagged.  The
      // first tile's consumer barrier orders these stores before any read.
      if (threadIdx.x < kCols) {
        const int t = (cbase + (int)threadIdx.x) / G;
        unsigned long long m = 0;
        if (t < tokens) {
          m = a.tree_mask[r0 + t];
          const unsigned long long upto = t >= 63 ? ~0ull : (2ull << t) - 1;
          if (!((m >> t) & 1ull) || (m & ~upto)) raise_fault(a.status, PSKV_FAULT_BAD_MASK);
          m &= upto;
        }
        tm[threadIdx.x] = m;
      }
    }
    {
      const int jq = cbase + 8 * nt_scored() + r, tq = jq / G;  // the column this lane feeds
      const bool real = tq < tokens;
      const uint16_t *q =
          static_cast<const uint16_t *>(a.q) +
          (((size_t)r0 + (real ? tq : 0)) * a.num_q_heads + h0 + jq % G) * D + quarter() * DQ;
#pragma unroll
      for (int k = 0; k < KSQ; ++k) {
        qf[k][0] = real ? *reinterpret_cast<const uint32_t *>(q + 16 * k + 2 * c) : 0u;
        qf[k][1] = real ? *reinterpret_cast<const uint32_t *>(q + 16 * k + 8 + 2 * c) : 0u;
      }
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      // token t of the row sits at key len - tokens + t and sees keys up to itself
      const int j0 = cbase + 8 * nt + 2 * c, t0 = j0 / G, t1 = (j0 + 1) / G;
      const int own0 = rp.len - tokens + t0, own1 = rp.len - tokens + t1;
      lim0[nt] = t0 < tokens ? own0 + 1 : 0;
      lim1[nt] = t1 < tokens ? own1 + 1 : 0;

#pragma unroll
      for (int j = 0; j < KSP; ++j) o[nt][j][0] = o[nt][j][1] = o[nt][j][2] = o[nt][j][3] = 0.f;
      m0[nt] = m1[nt] = -CUDART_INF_F;
      l0[nt] = l1[nt] = 0.f;
    }
  }

  __device__ void tile(const unsigned char *ks, const unsigned char *vs, int key0, int i0, int len,
                       bool skip, int lane, int j_tile) {
    const int mi = lane >> 3, rr = lane & 7;
    // ---- partial scores of this warp's n-tile over its quarter of D
    float acc[CH][4];
#pragma unroll
    for (int ch = 0; ch < CH; ++ch) acc[ch][0] = acc[ch][1] = acc[ch][2] = acc[ch][3] = 0.f;
    // A rows m = (mi&1)*8 + rr hold key 2*rr + (mi&1): pair rr, row (mi&1) of the pair
    const int dq = quarter();
    const bool from_v = kFolded && dq > 0;  // a folded key's columns past D/4 live in V
    const uint32_t kaddr =
        from_v ? smem_u32(vs) + rr * GSV + (mi & 1) * RBV + (mi >> 1) * 16 + dq * DQ * 2
               : smem_u32(ks) + rr * GSK + (mi & 1) * RBK + (mi >> 1) * 16 +
                     (kFolded ? 0 : dq * DQ * 2);
#pragma unroll
    for (int k = 0; k < KSQ; ++k) {
      uint32_t a0, a1, a2, a3;
      ldsm_x4(kaddr + k * 32, a0, a1, a2, a3);
      mma_bf16(acc[k % CH], a0, a1, a2, a3, qf[k][0], qf[k][1]);
    }
    // ---- sum the four quarters' partials of each n-tile (fixed order: every warp gets the same bits)
    float4 *slot = xchg + (j_tile & 1) * kQuarters * NT * 32;
    {
      float4 part = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int ch = 0; ch < CH; ++ch) {
        part.x += acc[ch][0];
        part.y += acc[ch][1];
        part.z += acc[ch][2];
        part.w += acc[ch][3];
      }
      slot[(dq * NT + nt_scored()) * 32 + lane] = part;
    }
    consumers_sync(kWarps * 32);
    float s00[NT], s01[NT], s10[NT], s11[NT];
    const int tA = key0 + 2 * r, tB = tA + 1;  // keys of MMA rows r and r + 8
    bool need = false;
    // The reference max only moves when some score exceeds it by more than
    // kSlack (log2 units): below that, exp2(s - m) <= 2^8 is exact in float and
    // in the hi+lo weights, and (m, l, o) stays an exact state for any reference
    // m, so most tiles skip the cross-lane max and the rescale.  The decision
    // depends only on the scores, which every warp holds identically.
    constexpr float kSlack = 8.f;
    float x0[NT], x1[NT];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      float4 st = slot[nt * 32 + lane];
#pragma unroll
      for (int q = 1; q < kQuarters; ++q) {
        const float4 x = slot[(q * NT + nt) * 32 + lane];
        st.x += x.x;
        st.y += x.y;
        st.z += x.z;
        st.w += x.w;
      }
      // a token's first visible key: lo_fixed, or (own + 1) - window with a window
      const int lo0 = window > 0 ? max(0, lim0[nt] - window) : lo_fixed;
      const int lo1 = window > 0 ? max(0, lim1[nt] - window) : lo_fixed;
      // in a drafted tree, a window key (t >= win0) is visible to a column iff
      // its bit is set in the column's mask (only tiles reaching the window look)
      const bool in_tree = kTree && key0 + kKeyTile > win0;
      auto vis = [&](int t, int lo, int lim, int col) {
        const int dt = t - win0;
        return !skip && t >= lo && t < lim &&
               (!in_tree || dt < 0 || (dt < 64 && ((tmask[col] >> dt) & 1ull)));
      };
      const int ca = 8 * nt + 2 * c, cb1 = ca + 1;  // the block's columns of this lane
      s00[nt] = vis(tA, lo0, lim0[nt], ca) ? st.x * scale_log2 : -CUDART_INF_F;   // key tA, col 8nt+2c
      s01[nt] = vis(tA, lo1, lim1[nt], cb1) ? st.y * scale_log2 : -CUDART_INF_F;  // key tA, col 8nt+2c+1
      s10[nt] = vis(tB, lo0, lim0[nt], ca) ? st.z * scale_log2 : -CUDART_INF_F;   // key tB, col 8nt+2c
      s11[nt] = vis(tB, lo1, lim1[nt], cb1) ? st.w * scale_log2 : -CUDART_INF_F;  // key tB, col 8nt+2c+1
      x0[nt] = fmaxf(s00[nt], s10[nt]);
      x1[nt] = fmaxf(s01[nt], s11[nt]);
      need |= x0[nt] > m0[nt] + kSlack || x1[nt] > m1[nt] + kSlack;
    }

    // ---- online softmax update
    if (__any_sync(0xffffffffu, need)) {
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {  // max over the 16 keys: lanes sharing c
          x0[nt] = fmaxf(x0[nt], __shfl_xor_sync(0xffffffffu, x0[nt], off));
          x1[nt] = fmaxf(x1[nt], __shfl_xor_sync(0xffffffffu, x1[nt], off));
        }
        const float n0 = fmaxf(m0[nt], x0[nt]), n1 = fmaxf(m1[nt], x1[nt]);
        const float al0 = (m0[nt] == -CUDART_INF_F) ? 0.f : exp2f(m0[nt] - n0);
        const float al1 = (m1[nt] == -CUDART_INF_F) ? 0.f : exp2f(m1[nt] - n1);
        l0[nt] *= al0;
        l1[nt] *= al1;
#pragma unroll
        for (int j = 0; j < KSP; ++j) {
          o[nt][j][0] *= al0;
          o[nt][j][1] *= al1;
          o[nt][j][2] *= al0;
          o[nt][j][3] *= al1;
        }
        m0[nt] = n0;
        m1[nt] = n1;
      }
    }
    uint32_t bh0[NT], bh1[NT], bl0[NT], bl1[NT];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const float u0 = (m0[nt] == -CUDART_INF_F) ? 0.f : m0[nt];  // nothing visible yet: weights 0
      const float u1 = (m1[nt] == -CUDART_INF_F) ? 0.f : m1[nt];
      const float p00 = exp2f(s00[nt] - u0), p01 = exp2f(s01[nt] - u1);
      const float p10 = exp2f(s10[nt] - u0), p11 = exp2f(s11[nt] - u1);
      l0[nt] += p00 + p10;
      l1[nt] += p01 + p11;
      // P^T fragments (hi + lo bf16 pairs), transposed in registers
      const uint32_t hA = pack_bf16x2(p00, p01), hB = pack_bf16x2(p10, p11);
      const uint32_t lA = pack_bf16x2(p00 - bf16_lo(hA), p01 - bf16_hi(hA));
      const uint32_t lB = pack_bf16x2(p10 - bf16_lo(hB), p11 - bf16_hi(hB));
      bh0[nt] = movmatrix_t(hA);
      bh1[nt] = movmatrix_t(hB);
      bl0[nt] = movmatrix_t(lA);
      bl1[nt] = movmatrix_t(lB);
    }

    // ---- O^T += V^T P^T over this warp's d slice; values of keys outside [i0, len) masked to zero
    const bool full = !skip && key0 >= i0 && key0 + kKeyTile <= len;
    uint32_t mlo = 0xffffffffu, mhi = 0xffffffffu;
    if (!full) {
      // B rows k = 2c, 2c+1 hold keys 4c, 4c+2; k = 2c+8, 2c+9 hold keys 4c+1, 4c+3
      const int t0 = key0 + 4 * c;
      auto ok = [&](int t) { return !skip && t >= i0 && t < len; };
      mlo = (ok(t0) ? 0x0000ffffu : 0u) | (ok(t0 + 2) ? 0xffff0000u : 0u);
      mhi = (ok(t0 + 1) ? 0x0000ffffu : 0u) | (ok(t0 + 3) ? 0xffff0000u : 0u);
    }
    // V^T A-fragment: source row k = rr + 8*(mi>>1) holds key 2*rr + (mi>>1)
    const uint32_t vaddr =
        smem_u32(vs) + rr * GSV + (mi >> 1) * RBV + (mi & 1) * 16 + warp * DW * 2;
#pragma unroll
    for (int j = 0; j < KSP; ++j) {
      uint32_t a0, a1, a2, a3;
      ldsm_x4_t(vaddr + j * 32, a0, a1, a2, a3);
      a0 &= mlo;
      a1 &= mlo;
      a2 &= mhi;
      a3 &= mhi;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        mma_bf16(o[nt][j], a0, a1, a2, a3, bh0[nt], bh1[nt]);
        mma_bf16(o[nt][j], a0, a1, a2, a3, bl0[nt], bl1[nt]);
      }
    }
  }

  // Sum this warp's per-lane l over the 8 lanes that share a column pair.
  __device__ void finish() {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {
        l0[nt] += __shfl_xor_sync(0xffffffffu, l0[nt], off);
        l1[nt] += __shfl_xor_sync(0xffffffffu, l1[nt], off);
      }
  }

  // Write this partition's (m, l, o) of every real column: every warp writes
  // its d slice; warp 0 the scalars.  Column j -> query row r0 + j / G, head
  // h0 + j % G.  With one partition (`direct`) the normalised output o / l goes
  // straight to `out` (zeros and PSKV_FAULT_EMPTY_ROW where no key was seen).
  __device__ void write_partial(const PartialArgs &a, const RowPlan &, int h0, int p) const {
    const int P = a.num_splits, d0 = warp * DW;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int jc = cbase + 8 * nt + 2 * c + e, t = jc / G;
        if (t >= tokens) continue;
        const size_t qrow = ((size_t)r0 + t) * a.num_q_heads + h0 + jc % G;
        if (a.direct) {
          const float mm = e ? m1[nt] : m0[nt];
          const float inv = mm == -CUDART_INF_F ? 0.f : 1.f / (e ? l1[nt] : l0[nt]);
          if (a.out_dtype == PSKV_DTYPE_BF16) {
            __nv_bfloat16 *dst = static_cast<__nv_bfloat16 *>(a.out) + qrow * D + d0 + r;
#pragma unroll
            for (int j = 0; j < KSP; ++j) {
              dst[16 * j] = __float2bfloat16_rn(o[nt][j][e] * inv);
              dst[16 * j + 8] = __float2bfloat16_rn(o[nt][j][2 + e] * inv);
            }
          } else {
            float *dst = static_cast<float *>(a.out) + qrow * D + d0 + r;
#pragma unroll
            for (int j = 0; j < KSP; ++j) {
              dst[16 * j] = o[nt][j][e] * inv;
              dst[16 * j + 8] = o[nt][j][2 + e] * inv;
            }
          }
          if (mm == -CUDART_INF_F && warp == 0 && r == 0) raise_fault(a.status, PSKV_FAULT_EMPTY_ROW);
          continue;
        }
        const size_t row = qrow * P + p;
        float *dst = a.ws_o + row * D + d0 + r;
        const uint64_t keep = make_evict_last_policy();
#pragma unroll
        for (int j = 0; j < KSP; ++j) {
          st_keep(dst + 16 * j, o[nt][j][e], keep);
          st_keep(dst + 16 * j + 8, o[nt][j][2 + e], keep);
        }
        if (warp == 0 && r == 0) {
          const float mm = e ? m1[nt] : m0[nt];
          st_keep(a.ws_m + row, mm == -CUDART_INF_F ? -CUDART_INF_F : mm * kLn2, keep);
          st_keep(a.ws_l + row, e ? l1[nt] : l0[nt], keep);
        }
      }
    }
  }
};

// -------------------------------------------------------------------------------------------
// CUDA-core consumer for any supported (element type, D, G): f32 pools, bf16
// pools with G != 8, or windowed rows with few query heads per KV head.
// Lane owns E = D/32 elements of every row, in 16-byte chunks k at
// d = (lane + 32k) * VE, so a warp reads each row as contiguous 512-byte runs.
// Scores are reduced across the warp by butterfly shuffles; keys are processed
// four at a time so the softmax rescale is paid once per four keys.
// -------------------------------------------------------------------------------------------
template <typename T, int kD, int kG>
struct SimtConsumer {
  using Elem = T;
  static constexpr int D = kD;
  static constexpr int G = kG;
  static constexpr int kCols = kG;  // one query token: a column per head of the group
  static constexpr int E = D / 32;
  static constexpr int VE = 16 / (int)sizeof(T);
  static constexpr int NC = E / VE;
  static constexpr bool kQInRegs = G * E <= 64;
  static constexpr int kExtraSmem = kQInRegs ? 0 : G * D * 4;
  // four consumer warps, two when a stage is too big for four of them
  static constexpr int kWarps = (D * (int)sizeof(T) > 1024) ? 2 : 4;
  static constexpr bool kCooperative = false;  // warp w takes tiles w, w + kWarps, ...
  static constexpr int kMinBlocks = 1;
  static constexpr int kRowBytesK = D * (int)sizeof(T), kRowBytesV = D * (int)sizeof(T);
  using Geom = RingGeom<kRowBytesK, kRowBytesV, kKeyTile, kWarps>;  // one copy per tile

  float q[kQInRegs ? G : 1][kQInRegs ? E : 1];
  float o[G][E];
  float m[G], l[G];
  float scale_log2;
  const float *q_s;
  int lane_;

  static __device__ float to_f32(float x) { return x; }
  static __device__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

  // Load the lane's E elements of a row (global or shared) as f32.
  static __device__ void load_row(const T *row, int lane, float (&dst)[E]) {
#pragma unroll
    for (int k = 0; k < NC; ++k) {
      const uint4 raw = *reinterpret_cast<const uint4 *>(row + (lane + 32 * k) * VE);
      if constexpr (sizeof(T) == 4) {
        dst[k * VE + 0] = __uint_as_float(raw.x);
        dst[k * VE + 1] = __uint_as_float(raw.y);
        dst[k * VE + 2] = __uint_as_float(raw.z);
        dst[k * VE + 3] = __uint_as_float(raw.w);
      } else {
        const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          dst[k * VE + 2 * i] = bf16_lo(w[i]);
          dst[k * VE + 2 * i + 1] = bf16_hi(w[i]);
        }
      }
    }
  }

  // All threads: stage Q of the group as f32 when it does not fit in registers.
  static __device__ void prologue(const PartialArgs &a, int b, int h0, unsigned char *extra) {
    if constexpr (!kQInRegs) {
      float *qs = reinterpret_cast<float *>(extra);
      const T *q = static_cast<const T *>(a.q) + ((size_t)b * a.num_q_heads + h0) * D;
      for (int i = threadIdx.x; i < G * D; i += blockDim.x) qs[i] = to_f32(q[i]);
    }
  }

  __device__ void init(const PartialArgs &a, const RowPlan &rp, int h0, int lane,
                       unsigned char *extra, int) {
    const int b = rp.b;
    lane_ = lane;
    scale_log2 = a.scale_log2;
    q_s = reinterpret_cast<const float *>(extra);
    if constexpr (kQInRegs) {
      const T *qb = static_cast<const T *>(a.q) + ((size_t)b * a.num_q_heads + h0) * D;
#pragma unroll
      for (int g = 0; g < G; ++g) load_row(qb + (size_t)g * D, lane, q[g]);
    }
#pragma unroll
    for (int g = 0; g < G; ++g) {
      m[g] = -CUDART_INF_F;
      l[g] = 0.f;
#pragma unroll
      for (int e = 0; e < E; ++e) o[g][e] = 0.f;
    }
  }

  __device__ float qval(int g, int e) const {
    if constexpr (kQInRegs) {
      return q[g][e];
    } else {
      const int k = e / VE, v = e % VE;
      return q_s[g * D + (lane_ + 32 * k) * VE + v];
    }
  }

  __device__ void tile(const unsigned char *ks, const unsigned char *vs, int key0, int i0, int len,
                       bool skip, int lane, int) {
#pragma unroll 1
    for (int t0 = 0; t0 < kKeyTile; t0 += 4) {
      float s[4][G];
      bool valid[4];
      bool any = false;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int t = key0 + t0 + u;
        valid[u] = !skip && t >= i0 && t < len;
        any |= valid[u];
#pragma unroll
        for (int g = 0; g < G; ++g) s[u][g] = -CUDART_INF_F;
        if (valid[u]) {
          float kf[E];
          load_row(reinterpret_cast<const T *>(ks + Geom::row_off_k(t0 + u)), lane, kf);
#pragma unroll
          for (int g = 0; g < G; ++g) {
            float acc = 0.f;
#pragma unroll
            for (int e = 0; e < E; ++e) acc = fmaf(qval(g, e), kf[e], acc);
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
            s[u][g] = acc * scale_log2;
          }
        }
      }
      if (!any) continue;
      bool rescale = false;
      float al[G];
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const float x = fmaxf(fmaxf(s[0][g], s[1][g]), fmaxf(s[2][g], s[3][g]));
        const float n = fmaxf(m[g], x);
        const float u = (n == -CUDART_INF_F) ? 0.f : n;
        al[g] = exp2f(m[g] - u);
        rescale |= (al[g] != 1.f);
        float sum = 0.f;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          s[k][g] = exp2f(s[k][g] - u);
          sum += s[k][g];
        }
        l[g] = l[g] * al[g] + sum;
        m[g] = n;
      }
      if (rescale) {
#pragma unroll
        for (int g = 0; g < G; ++g)
#pragma unroll
          for (int e = 0; e < E; ++e) o[g][e] *= al[g];
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        if (!valid[u]) continue;
        float vf[E];
        load_row(reinterpret_cast<const T *>(vs + Geom::row_off_v(t0 + u)), lane, vf);
#pragma unroll
        for (int g = 0; g < G; ++g)
#pragma unroll
          for (int e = 0; e < E; ++e) o[g][e] = fmaf(s[u][g], vf[e], o[g][e]);
      }
    }
  }

  __device__ void finish() {}

  __device__ void store(float *o_s, float *m_s, float *l_s) const {
#pragma unroll
    for (int g = 0; g < G; ++g) {
#pragma unroll
      for (int e = 0; e < E; ++e) {
        const int k = e / VE, v = e % VE;
        o_s[g * D + (lane_ + 32 * k) * VE + v] = o[g][e];
      }
      if (lane_ == 0) {
        m_s[g] = m[g];
        l_s[g] = l[g];
      }
    }
  }
};

// -------------------------------------------------------------------------------------------
// The kernel skeleton shared by both consumers.
// -------------------------------------------------------------------------------------------
template <class C>
struct PartialSmem {
  using Geom = typename C::Geom;
  static constexpr int kRing = Geom::kRingBytes;
  static constexpr int kExtraOff = kRing;
  static constexpr int kBarOff = (kExtraOff + C::kExtraSmem + 15) / 16 * 16;
  static constexpr int kSkipOff = kBarOff + 2 * Geom::kStages * 8;
  static constexpr int kRedOff = kSkipOff + 4 * Geom::kStages;
  static constexpr int kWeightOff = kRedOff + 2 * C::kWarps * C::G * 4;
  static constexpr int kAbortOff = kWeightOff + C::kWarps * C::G * 4;
  static constexpr int kBytes = kAbortOff + 16;
  // the warp states alias the ring once every stage has been consumed
  static_assert(C::kCooperative || C::kWarps * C::G * C::D * 4 <= kRing,
                "merge area must fit in the ring");
  static_assert(kBytes <= 227 * 1024, "shared memory budget");
  static_assert(C::kCooperative || Geom::kStages % C::kWarps == 0,
                "stages must divide among the consumer warps");
};

// Merge the independent warps' states (the ring is free now) and write the partial.
template <class C>
__device__ __forceinline__ void merge_warp_states(const C &cons, const PartialArgs &a,
                                                  unsigned char *ring, float *red_m, float *red_l,
                                                  float *weight, size_t row0, int P, int warp) {
  constexpr int D = C::D, G = C::G, CW = C::kWarps, NT = (CW + 1) * 32;
  float *o_s = reinterpret_cast<float *>(ring);  // [warps][G][D]
  if (warp < CW) cons.store(o_s + (size_t)warp * G * D, red_m + warp * G, red_l + warp * G);
  __syncthreads();
  if (threadIdx.x < G) {
    const int h = threadIdx.x;
    float M = -CUDART_INF_F;
    for (int w = 0; w < CW; ++w) M = fmaxf(M, red_m[w * G + h]);
    float L = 0.f;
    for (int w = 0; w < CW; ++w) {
      const float mw = red_m[w * G + h];
      const float wt = (mw == -CUDART_INF_F) ? 0.f : exp2f(mw - M);
      weight[w * G + h] = wt;
      L += wt * red_l[w * G + h];
    }
    const uint64_t keep = make_evict_last_policy();
    st_keep(a.ws_m + row0 + (size_t)h * P, (M == -CUDART_INF_F) ? -CUDART_INF_F : M * kLn2, keep);
    st_keep(a.ws_l + row0 + (size_t)h * P, L, keep);
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < G * D; idx += NT) {
    const int h = idx / D, d = idx - h * D;
    float acc = 0.f;
#pragma unroll
    for (int w = 0; w < CW; ++w) {
      const float wt = weight[w * G + h];
      if (wt != 0.f) acc = fmaf(o_s[(w * G + h) * D + d], wt, acc);
    }
    st_keep(a.ws_o + (row0 + (size_t)h * P) * D + d, acc, make_evict_last_policy());
  }
}

template <class C>
__global__ void __launch_bounds__((C::kWarps + 1) * 32, C::kMinBlocks)
    pskv_partial_kernel(const PartialArgs a) {
  extern __shared__ __align__(128) unsigned char smem[];
  using Geom = typename C::Geom;
  using S = PartialSmem<C>;
  constexpr int D = C::D, G = C::G, NS = Geom::kStages;
  constexpr int RBK = C::kRowBytesK, RBV = C::kRowBytesV;  // bytes of a K row, a V row
  constexpr int TBK = Geom::kTileBytesK;
  constexpr int R = Geom::kRowsPerCopy;
  constexpr int CW = C::kWarps;  // consumer warps; warp CW is the producer

  unsigned char *ring = smem;
  unsigned char *extra = smem + S::kExtraOff;
  uint64_t *full_bar = reinterpret_cast<uint64_t *>(smem + S::kBarOff);
  uint64_t *empty_bar = full_bar + NS;
  int *stage_skip = reinterpret_cast<int *>(smem + S::kSkipOff);
  float *red_m = reinterpret_cast<float *>(smem + S::kRedOff);  // [warps][G] (log2 units)
  float *red_l = red_m + CW * G;                                   // [warps][G]
  float *weight = reinterpret_cast<float *>(smem + S::kWeightOff); // [warps][G]
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + S::kAbortOff);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // x = partition x column block (the blocks of one partition launch together
  // and share its keys in L2), y = KV head, z = row
  const int cb = (int)(blockIdx.x % (unsigned)a.col_blocks);
  const int p = (int)(blockIdx.x / (unsigned)a.col_blocks), g = blockIdx.y, b = blockIdx.z;
  const int P = a.num_splits;
  const int h0 = g * G;

  // Only set-up that touches no global memory overlaps the previous kernel;
  // every read of caller memory (lengths, window bounds, tables, queries,
  // pools) and every write comes after pdl_wait().
  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], C::kCooperative ? CW : 1);  // released by every warp that reads it
    }
    *abort_flag = 0;
    mbar_fence_init();
  }
  pdl_wait();
  pdl_launch_dependents();

  // ---- the page ids of the partition's first tiles, fetched by the producer
  // from the host's copy of the length while the device length is read (plain
  // rows: uniform tokens, no window, one column block); kept below only if the
  // device length gives the same first slot and slot count
  int hint_slot = -1, hint_slots = -1, hint_ids = -1;
  if (warp == C::kWarps && b < kLenHints && a.len_hint[b] >= a.num_tokens && a.cu_q == nullptr &&
      a.window_lo == nullptr && a.window == 0 && a.col_blocks == 1) {
    const int hl = a.len_hint[b];
    const int tiles = (hl + kKeyTile - 1) / kKeyTile, per = (tiles + P - 1) / P;
    const int tb = p * per < tiles ? p * per : tiles;
    hint_slot = tb * kKeyTile / a.page_size;
    hint_slots = (hl + a.page_size - 1) / a.page_size;
    const int sl = hint_slot + lane;
    hint_ids = sl < hint_slots ? __ldg(a.page_tables + (size_t)b * a.table_stride + sl) : -1;
  }

  // ---- this CTA's query tokens (row b's are query rows r0 .. r0 + T - 1)
  RowPlan rp;
  rp.b = b;
  rp.T = a.num_tokens;
  rp.r0 = b * a.num_tokens;
  rp.window = a.window;
  if (a.cu_q != nullptr) {
    const int c0 = a.cu_q[b], c1 = a.cu_q[b + 1];
    if (c0 < 0 || c1 < c0 || c1 > a.total_rows) {  // never address rows outside the arrays
      if (threadIdx.x == 0 && p == 0 && g == 0 && cb == 0) raise_fault(a.status, PSKV_FAULT_BAD_LENGTH);
      rp.T = 0;
      rp.r0 = 0;
    } else {
      rp.T = c1 - c0;
      rp.r0 = c0;
    }
  }
  const int T = rp.T;
  if (cb * C::kCols >= T * G) return;  // no real column in this block
  // ---- and its keys: a token at key len - T + t sees keys up to itself
  const long long cap = (long long)a.table_stride * a.page_size;
  long long len_ll = a.seq_lens[b];
  if (len_ll < T || len_ll < 1 || len_ll > cap) {  // a row holds at least its query tokens
    if (threadIdx.x == 0 && p == 0 && g == 0 && cb == 0) raise_fault(a.status, PSKV_FAULT_BAD_LENGTH);
    len_ll = len_ll < 0 ? 0 : (len_ll > cap ? cap : len_ll);
  }
  const int len = (int)len_ll;
  rp.len = len;
  rp.lo_fixed = 0;
  if (a.window_lo != nullptr) {
    long long d = (long long)a.window_lo[b] - (long long)a.first_pos[b];
    rp.lo_fixed = (int)(d < 0 ? 0 : (d > len ? len : d));
  }
  const int t_first = cb * C::kCols / G, t_last = min(T - 1, ((cb + 1) * C::kCols - 1) / G);
  const int k_hi = max(0, min(len, len - T + t_last + 1));  // keys [k_lo, k_hi) serve this block
  const int k_lo = min(k_hi, a.window > 0 ? max(0, len - T + t_first - a.window + 1) : rp.lo_fixed);
  const int i0 = k_lo;
  const int n_tiles = (k_hi + kKeyTile - 1) / kKeyTile;
  const int t_lo = k_lo < k_hi ? k_lo / kKeyTile : n_tiles;
  const long long total = n_tiles - t_lo;
  const long long per = (total + P - 1) / P;
  const long long lo_ll = (long long)p * per < total ? (long long)p * per : total;
  const long long hi_ll = (long long)(p + 1) * per < total ? (long long)(p + 1) * per : total;
  const int t_begin = t_lo + (int)lo_ll;
  const int n_my = (int)(hi_ll - lo_ll);

  const size_t row0 = ((size_t)b * a.num_q_heads + h0) * P + p;  // workspace state of head h0 (T = 1)
  // The step's new row (key len - 1, single-token decode) is written by the
  // CTA whose partition holds it; when no partition does (a window past the
  // row's keys), by partition 0.
  const bool append_here =
      a.append_k != nullptr && cb == 0 &&
      (k_lo < k_hi ? (len - 1 >= (t_begin) * kKeyTile && len - 1 < (t_begin + n_my) * kKeyTile)
                   : p == 0);
  if (n_my <= 0) {  // empty partition: m = -inf, l = 0 (o is not written)
    if (append_here && warp == 0) append_new_row(a, b, g, len - 1, lane);
    const int c0 = cb * C::kCols, c1 = min(c0 + C::kCols, T * G);  // this block's columns
    if (a.direct) {  // one partition and no key: zeros, flagged
      for (int i = c0 * D + threadIdx.x; i < c1 * D; i += blockDim.x) {
        const size_t qrow = ((size_t)rp.r0 + i / D / G) * a.num_q_heads + h0 + (i / D) % G;
        if (a.out_dtype == PSKV_DTYPE_BF16)
          static_cast<__nv_bfloat16 *>(a.out)[qrow * D + i % D] = __float2bfloat16_rn(0.f);
        else
          static_cast<float *>(a.out)[qrow * D + i % D] = 0.f;
      }
      if (threadIdx.x == 0 && c0 < c1) raise_fault(a.status, PSKV_FAULT_EMPTY_ROW);
      return;
    }
    for (int i = c0 + threadIdx.x; i < c1; i += blockDim.x) {
      const size_t row = (((size_t)rp.r0 + i / G) * a.num_q_heads + h0 + i % G) * P + p;
      const uint64_t keep = make_evict_last_policy();
      st_keep(a.ws_m + row, -CUDART_INF_F, keep);
      st_keep(a.ws_l + row, 0.f, keep);
    }
    return;
  }
  C::prologue(a, b, h0, extra);
  __syncthreads();

  C cons;
  if (warp == CW) {
    // ---------------- producer warp
    const int32_t *tbl = a.page_tables + (size_t)b * a.table_stride;
    const int n_slots = (k_hi + a.page_size - 1) / a.page_size;  // table entries in use
    int cache_base = -1, cached = -1;
    if (hint_slots == n_slots && hint_slot == t_begin * kKeyTile / a.page_size) {
      cache_base = hint_slot;  // the fetched ids are the ones this partition starts with
      cached = hint_ids;
    }
    int issued = 0;
    const uint64_t stream_policy = make_evict_first_policy();
    if (append_here) {
      append_new_row(a, b, g, len - 1, lane);
      asm volatile("fence.proxy.async.global;" ::: "memory");  // the issuing lane's own order
    }
    for (int j = 0; j < n_my; ++j) {
      const int s = j % NS;
      if (__shfl_sync(0xffffffffu, *abort_flag, 0)) break;  // one decision for the whole warp
      if (j >= NS) {
        const bool freed = mbar_wait(&empty_bar[s], ((j / NS) - 1) & 1);
        if (!__all_sync(0xffffffffu, freed)) {
          if (lane == 0) {
            raise_fault(a.status, PSKV_FAULT_WAIT_TIMEOUT);
            *abort_flag = 1;
          }
          break;
        }
      }
      const int key0 = (t_begin + j) * kKeyTile;
      const int slot = key0 / a.page_size;
      if (cache_base < 0 || slot >= cache_base + 32) {
        cache_base = slot;
        const int sl = slot + lane;
        cached = sl < n_slots ? __ldg(tbl + sl) : -1;
      }
      const int page = __shfl_sync(0xffffffffu, cached, slot - cache_base);
      const bool ok = page >= 0 && (long long)page < a.num_pages;
      const int r_lo = i0 > key0 ? i0 - key0 : 0;
      const int r_hi = k_hi - key0 < kKeyTile ? k_hi - key0 : kKeyTile;
      unsigned char *kdst = ring + s * Geom::kStageBytes;
      unsigned char *vdst = kdst + TBK;
      if (lane == 0) {
        stage_skip[s] = ok ? 0 : 1;
        if (!ok) raise_fault(a.status, PSKV_FAULT_BAD_PAGE);
        mbar_arrive_expect_tx(&full_bar[s], ok ? (uint32_t)((r_hi - r_lo) * (RBK + RBV)) : 0u);
      }
      __syncwarp();
      // one copy per group of R rows (clipped to the valid rows); lane i copies
      // K group i, lane 16 + i V group i
      const int grp = lane & 15;
      const int g_lo = max(grp * R, r_lo), g_hi = min(grp * R + R, r_hi);
      if (ok && grp < kKeyTile / R && g_lo < g_hi) {
        const size_t grow = ((size_t)page * a.num_kv_heads + g) * a.page_size +
                            (size_t)(key0 % a.page_size) + g_lo;
        const bool is_k = lane < 16;
        const int rb = is_k ? RBK : RBV;
        const unsigned char *src =
            static_cast<const unsigned char *>(is_k ? a.k_pool : a.v_pool) + grow * rb;
        bulk_g2s_hint(is_k ? kdst + Geom::row_off_k(g_lo) : vdst + Geom::row_off_v(g_lo), src,
                      (uint32_t)((g_hi - g_lo) * rb), &full_bar[s], stream_policy);
      }
      issued = j + 1;
    }
    if (*abort_flag) {
      // never leave a copy in flight into shared memory this CTA gives up
      const int first = issued > NS ? issued - NS : 0;
      for (int j = first; j < issued; ++j) mbar_wait(&full_bar[j % NS], (j / NS) & 1);
    }
  } else {
    // ---------------- consumer warps
    // cooperative consumers all take every tile; the others take every CW-th
    cons.init(a, rp, h0, lane, extra, cb);
    const int j0 = C::kCooperative ? 0 : warp, dj = C::kCooperative ? 1 : CW;
    for (int j = j0; j < n_my; j += dj) {
      const int s = j % NS;
      const bool landed = mbar_wait(&full_bar[s], (j / NS) & 1) && !*abort_flag;
      // one decision for every thread that will meet at the consumers' barrier
      bool go;
      if constexpr (C::kCooperative)
        go = consumers_all(CW * 32, landed);
      else
        go = __all_sync(0xffffffffu, landed);
      if (!go) {
        if (lane == 0) {
          raise_fault(a.status, PSKV_FAULT_WAIT_TIMEOUT);
          *abort_flag = 1;
        }
        break;
      }
      const unsigned char *kst = ring + s * Geom::kStageBytes;
      cons.tile(kst, kst + TBK, (t_begin + j) * kKeyTile, i0, k_hi, stage_skip[s] != 0, lane, j);
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty_bar[s]);
    }
    cons.finish();
  }
  __syncthreads();
  if (*abort_flag) return;

  if constexpr (C::kCooperative) {
    if (warp < CW) cons.write_partial(a, rp, h0, p);
    return;
  } else {
    merge_warp_states<C>(cons, a, ring, red_m, red_l, weight, row0, P, warp);
  }
}

template <class C>
cudaError_t set_partial_smem_attr() {
  constexpr int bytes = PartialSmem<C>::kBytes;
  static bool attr_set[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 64 && attr_set[dev]) return cudaSuccess;
  e = cudaFuncSetAttribute(pskv_partial_kernel<C>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           bytes);
  if (e == cudaSuccess && dev >= 0 && dev < 64) attr_set[dev] = true;
  return e;
}

template <class C>
cudaError_t launch_partial_kernel(const PartialArgs &a, dim3 grid, cudaStream_t stream) {
  cudaError_t e = set_partial_smem_attr<C>();
  if (e != cudaSuccess) return e;
  return launch_pdl(pskv_partial_kernel<C>, grid, dim3((C::kWarps + 1) * 32),
                    PartialSmem<C>::kBytes, stream, a);
}

// CTAs of this kernel that fit on one SM at once.
template <class C>
cudaError_t partial_kernel_occupancy(int *ctas) {
  cudaError_t e = set_partial_smem_attr<C>();
  if (e != cudaSuccess) return e;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas, pskv_partial_kernel<C>,
                                                       (C::kWarps + 1) * 32,
                                                       PartialSmem<C>::kBytes);
}

}  // namespace pskv
