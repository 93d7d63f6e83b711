// attn_tc.cu -- paged attention of many query rows per KV head on the fifth-
// generation tensor cores (tcgen05, tensor memory, tensor copies).
//
// Serves paged prefill (pegainfer #1057, Description: the sliding family's
// prompt rows read through a windowed varlen kernel with a window lower bound)
// at head dim 256, bf16 pools in the split format.  One CTA takes a block of
// 128 query rows of one (row, KV head): row i of the block is query column
// qb * 128 + i of the row's chunk (token column / G, head column % G), and a
// partition of the keys those tokens can see.  Per tile of 64 keys:
//   S  = Q K^T    M = 128 rows, N = 64 keys, K = 256 (16 MMAs; S in tensor memory)
//   softmax       one thread per query row reads its 64 scores from tensor
//                 memory, masks them (causal, window, keys outside the
//                 CTA's range), keeps the row's reference max and sum (exp2
//                 units; the max moves only past a slack of 8, as in the
//                 decode kernels) and writes P as a bf16 hi + lo pair into
//                 shared memory
//   O += P V      M = 128, N = 256, K = 64 keys, hi then lo (8 MMAs; O in tensor memory)
// Q (64 KB) and the K and V tiles (two stages each) arrive by tensor copies in
// the 128-byte swizzled layout the MMA descriptors read.  Warp 0 issues the
// MMAs, warp 1 the copies; warps 2-5 run the softmax and the epilogue (warp w
// owns tensor-memory lanes 32 (w % 4) .. + 31).  The two issuing warps are the
// oldest of their schedulers, so the softmax's long instruction streams do not
// hold them back.  Every wait is bounded; on expiry the CTA flags
// PSKV_FAULT_WAIT_TIMEOUT, lets what it issued finish and frees its tensor
// memory.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <math_constants.h>

#include "pskv_internal.cuh"
#include "tc_ops.cuh"

namespace pskv {

namespace {

constexpr int kD = 256;                     // head dim served
constexpr int kRows = 128;                  // query rows per CTA (MMA M)
constexpr int kKeys = 64;                   // keys per tile (MMA N of S, K of PV)
constexpr int kQSlab = kRows * 128;         // bytes of one 64-column slab of Q
constexpr int kKVSlab = kKeys * 128;        // bytes of one 64-column slab of a K or V tile
constexpr int kQBytes = 4 * kQSlab;         // 64 KB
constexpr int kKVBytes = 4 * kKVSlab;       // 32 KB
constexpr int kPBytes = kRows * kKeys * 2;  // 16 KB per P buffer (hi, lo)
constexpr int kThreads = 192;               // MMA warp, copy warp, 4 softmax warps
constexpr int kTmemCols = 512;              // S at columns [0, 64), O at [64, 320)
constexpr int kOCol = 64;
constexpr float kSlack = 8.f;               // reference-max slack (log2 units)

// shared memory (offsets from a 1,024-byte aligned base)
constexpr int kOffQ = 0;
constexpr int kOffK = kOffQ + kQBytes;       // K stage s at kOffK + s * kKVBytes
constexpr int kOffV = kOffK + 2 * kKVBytes;  // V stage s at kOffV + s * kKVBytes
constexpr int kOffP = kOffV + 2 * kKVBytes;  // P hi, then P lo
constexpr int kOffBar = kOffP + 2 * kPBytes;
// barriers: fullK[2], fullV[2], emptyK[2], emptyV[2], s_full, s_free, p_full, pv_done, drain,
// q_full, info_free[2]
constexpr int kNumBars = 16;
constexpr int kOffInfo = kOffBar + kNumBars * 8;  // StageInfo[2]
constexpr int kOffSlot = kOffInfo + 2 * 16;       // tensor-memory address
constexpr int kOffAbort = kOffSlot + 4;
constexpr int kSmemUsed = kOffAbort + 4;
constexpr int kSmemBytes = kSmemUsed + 1024;      // + alignment of the dynamic base
static_assert(kSmemBytes <= 232448, "shared memory per CTA");

constexpr uint32_t kIdescS = tc::instr_desc(kRows, kKeys, false, false);
constexpr uint32_t kIdescPV = tc::instr_desc(kRows, kD, false, true);

// What the copy warp loaded into a stage: the tile's rows [vlo, vhi) lie in
// the CTA's key range; `bad` marks 16-row chunks whose page id was outside
// the pool (not loaded).  Written before the stage's K barrier is armed, read
// by the softmax warps after that barrier completes.
struct StageInfo {
  int vlo, vhi;
  uint32_t bad;
  int pad;
};

}  // namespace


namespace {

// The CTA's share of the work, the same in every thread.
struct TcPlan {
  int b, g, qb, p;
  int T, r0, len;
  int k_lo, k_hi;    // keys the block's tokens can see
  int t_begin, n;    // this partition's tiles: [t_begin, t_begin + n) of 64 keys
  bool ok;           // the row's offsets and length are usable
};

__device__ __forceinline__ TcPlan make_plan(const TcArgs &a) {
  TcPlan pl;
  const int x = blockIdx.x;
  // heavier (later) query blocks first: under causality they see more keys
  pl.qb = a.qblocks - 1 - x % a.qblocks;
  pl.p = x / a.qblocks;
  pl.g = blockIdx.y;
  pl.b = blockIdx.z;
  pl.ok = true;
  const int c0 = a.cu_q[pl.b], c1 = a.cu_q[pl.b + 1];
  if (c0 < 0 || c1 < c0 || c1 > a.total_rows) {  // never address rows outside the arrays
    pl.ok = false;
    pl.T = 0;
    pl.r0 = 0;
  } else {
    pl.T = c1 - c0;
    pl.r0 = c0;
  }
  const long long cap = (long long)a.table_stride * a.page_size;
  long long len = a.seq_lens[pl.b];
  if (len < pl.T || len < 1 || len > cap) {
    pl.ok = false;
    len = len < 0 ? 0 : (len > cap ? cap : len);
  }
  pl.len = (int)len;
  const int G = 1 << a.group_shift;
  const int col0 = pl.qb * kRows, cols = pl.T * G;
  pl.k_lo = pl.k_hi = 0;
  pl.t_begin = 0;
  pl.n = 0;
  if (col0 >= cols) return pl;  // no query row in this block
  const int t_first = col0 >> a.group_shift;
  const int t_last = min(pl.T - 1, (col0 + kRows - 1) >> a.group_shift);
  pl.k_hi = max(0, min(pl.len, pl.len - pl.T + t_last + 1));
  pl.k_lo = min(pl.k_hi, a.window > 0 ? max(0, pl.len - pl.T + t_first - a.window + 1) : 0);
  const int t_lo = pl.k_lo / kKeys, t_hi = (pl.k_hi + kKeys - 1) / kKeys;
  const int total = pl.k_lo < pl.k_hi ? t_hi - t_lo : 0;
  const int P = a.num_splits;
  const int per = (total + P - 1) / P;
  const int lo = min(pl.p * per, total), hi = min(pl.p * per + per, total);
  pl.t_begin = t_lo + lo;
  pl.n = hi - lo;
  return pl;
}

// Bounded wait that gives up at once when another thread of the CTA already has.
__device__ __forceinline__ bool tc_wait(uint64_t *bar, uint32_t parity, volatile int *abort_flag,
                                        int32_t *status) {
  if (*abort_flag) return false;
  if (mbar_wait(bar, parity)) return true;
  *abort_flag = 1;
  raise_fault(status, PSKV_FAULT_WAIT_TIMEOUT);
  return false;
}

__device__ __forceinline__ bool elect_one() {
  uint32_t pred;
  asm volatile(
      "{\n\t.reg .pred p;\n\telect.sync _|p, 0xffffffff;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(pred));
  return pred != 0;
}

// Page ids of 32 consecutive table slots held across the control warp's lanes.
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

// Barrier slots.
enum : int {
  kFullK = 0, kFullV = 2, kEmptyK = 4, kEmptyV = 6,
  kSFull = 8, kSFree = 9, kPFull = 10, kPvDone = 11, kDrain = 12, kQFull = 13, kInfoFree = 14
};

__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, volatile int *abort_flag,
                                          int32_t *status) {
  const bool ok = tc_wait(bar, parity, abort_flag, status);
  return __all_sync(0xffffffffu, ok);
}

// The copy warp (all lanes converged; one elected lane issues).  Tile j's K
// and V go to stage j % 2:
//   K(j) once S(j - 2) has released the stage and the softmax warps have
//        read the stage's record of tile j - 2;
//   V(j) once PV(j - 2) has released the stage.
// Q (four 64-column slabs of the 128-row block) is requested first.
struct Loader {
  const TcArgs &a;
  const TcPlan &pl;
  const CUtensorMap *qmap, *kmap, *vmap;
  unsigned char *sm;
  uint64_t *bars;
  StageInfo *info;
  volatile int *abort_flag;
  int lane;
  int n_slots;  // table slots the CTA's keys use
  PageCache kpages, vpages;
  int k_issued = 0, v_issued = 0;

  __device__ Loader(const TcArgs &a_, const TcPlan &pl_, const CUtensorMap *qm,
                    const CUtensorMap *km, const CUtensorMap *vm, unsigned char *sm_,
                    uint64_t *bars_, StageInfo *info_, volatile int *ab)
      : a(a_), pl(pl_), qmap(qm), kmap(km), vmap(vm), sm(sm_), bars(bars_), info(info_),
        abort_flag(ab) {
    lane = threadIdx.x & 31;
    n_slots = (pl.k_hi + a.page_size - 1) / a.page_size;
  }

  // Issue the tensor copies of tile j into its K or V stage: 16- or 64-row
  // chunks, each in four 64-column slabs; chunks with no row in the CTA's key
  // range are not loaded, nor are chunks whose page id lies outside the pool
  // (bit c of the bad mask per 16 rows).  The K copy writes the stage's record
  // before the barrier is armed (the arrive releases it).
  __device__ void load(int j, bool is_v) {
    const int key0 = (pl.t_begin + j) * kKeys;
    const int vlo = max(0, pl.k_lo - key0), vhi = min(kKeys, pl.k_hi - key0);
    const int32_t *tbl = a.page_tables + (size_t)pl.b * a.table_stride;
    const int br = a.box_rows;
    PageCache &pc = is_v ? vpages : kpages;
    uint32_t bad = 0, bytes = 0;
    int pages[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      pages[c] = -1;
      if (c * br >= kKeys) continue;
      if ((c + 1) * br <= vlo || c * br >= vhi) continue;  // no row of the chunk is in range
      const int page = pc.get(tbl, (key0 + c * br) / a.page_size, n_slots, lane);
      if (page < 0 || (long long)page >= a.num_pages) {
        bad |= (br == kKeys ? 0xFu : 1u << c);
        continue;
      }
      pages[c] = page;
      bytes += (uint32_t)(br * 128 * 4);
    }
    unsigned char *dst = sm + (is_v ? kOffV : kOffK) + (j & 1) * kKVBytes;
    uint64_t *bar = bars + (is_v ? kFullV : kFullK) + (j & 1);
    if (elect_one()) {
      if (bad) raise_fault(a.status, PSKV_FAULT_BAD_PAGE);
      if (!is_v) {
        info[j & 1].vlo = vlo;
        info[j & 1].vhi = vhi;
        info[j & 1].bad = bad;
      }
      mbar_arrive_expect_tx(bar, bytes);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        if (pages[c] < 0) continue;
        const int key = key0 + c * br;
        const int y = (pages[c] * a.num_kv_heads + pl.g) * a.page_size + key % a.page_size;
#pragma unroll
        for (int sl = 0; sl < 4; ++sl)
          tc::tma_load_2d(dst + sl * kKVSlab + c * br * 128, is_v ? vmap : kmap, sl * 64, y, bar);
      }
    }
    __syncwarp();
    (is_v ? v_issued : k_issued) = j + 1;
  }

  // Q block: box (64 columns, the G heads, 128 / G tokens) from the chunk's
  // first token of the block; rows past the packed query rows read zeros.
  __device__ void load_q() {
    if (elect_one()) {
      uint64_t *bar = bars + kQFull;
      mbar_arrive_expect_tx(bar, (uint32_t)kQBytes);
      const int t0 = pl.r0 + ((pl.qb * kRows) >> a.group_shift);
      const int h0 = pl.g << a.group_shift;
#pragma unroll
      for (int sl = 0; sl < 4; ++sl) tc::tma_load_3d(sm + kOffQ + sl * kQSlab, qmap, sl * 64, h0, t0, bar);
    }
    __syncwarp();
  }

  __device__ bool wait(int slot, uint32_t parity) {
    return warp_wait(bars + slot, parity, abort_flag, a.status);
  }

  __device__ void prologue() {
    load_q();
    load(0, false);
    load(0, true);
    if (pl.n > 1) {
      load(1, false);
      load(1, true);
    }
  }

  __device__ bool run() {
    for (int j = 2; j < pl.n; ++j) {
      const int s = j & 1;
      const uint32_t ph = ((j - 2) >> 1) & 1;  // completion (j - 2) / 2 of the stage's barriers
      if (!wait(kEmptyK + s, ph) || !wait(kInfoFree + s, ph)) return false;
      load(j, false);
      if (!wait(kEmptyV + s, ph)) return false;
      load(j, true);
    }
    return true;
  }

  // Wait (bounded) for the last copy issued into each stage (and Q).
  __device__ void drain() {
    mbar_wait(bars + kQFull, 0);
    for (int s = 0; s < 2; ++s) {
      const int jk = k_issued - 1 - ((k_issued - 1 - s) & 1);  // last K tile of stage s
      if (jk >= 0) mbar_wait(bars + kFullK + s, (jk >> 1) & 1);
      const int jv = v_issued - 1 - ((v_issued - 1 - s) & 1);
      if (jv >= 0) mbar_wait(bars + kFullV + s, (jv >> 1) & 1);
    }
  }
};

// The MMA warp (all lanes converged; one elected lane issues).  Per tile j:
//   S(j) = Q K(j)^T once K(j) has landed and the softmax has read S(j - 1);
//   O += P(j - 1) V(j - 1) once P(j - 1) is written and V(j - 1) has landed.
struct Issuer {
  const TcArgs &a;
  const TcPlan &pl;
  unsigned char *sm;
  uint64_t *bars;
  volatile int *abort_flag;

  __device__ bool wait(int slot, uint32_t parity) {
    return warp_wait(bars + slot, parity, abort_flag, a.status);
  }

  __device__ bool run(uint32_t tmem) {
    const uint32_t q_addr = smem_u32(sm + kOffQ);
    const uint32_t p_addr = smem_u32(sm + kOffP);
    // descriptors at the operands' first k-step; a k-step adds its byte offset / 16
    const uint64_t dq = tc::smem_desc(q_addr, 16, 1024);
    const uint64_t dp = tc::smem_desc(p_addr, 16, 1024);
    const int n = pl.n;
    if (!wait(kQFull, 0)) return false;
    for (int j = 0; j <= n; ++j) {
      if (j < n) {
        const int s = j & 1;
        if (!wait(kFullK + s, (j >> 1) & 1)) return false;
        if (j >= 1 && !wait(kSFree, (j - 1) & 1)) return false;
        tc::fence_after_sync();
        const uint64_t dk = tc::smem_desc(smem_u32(sm + kOffK + s * kKVBytes), 16, 1024);
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < kD / 16; ++kk)
            tc::mma(tmem, dq + (uint64_t)(((kk >> 2) * kQSlab + (kk & 3) * 32) >> 4),
                    dk + (uint64_t)(((kk >> 2) * kKVSlab + (kk & 3) * 32) >> 4), kIdescS, kk > 0);
          tc::commit(bars + kSFull);
          tc::commit(bars + kEmptyK + s);
        }
        __syncwarp();
      }
      if (j >= 1) {
        const int jp = j - 1, sp = jp & 1;
        if (!wait(kPFull, jp & 1)) return false;
        if (!wait(kFullV + sp, (jp >> 1) & 1)) return false;
        tc::fence_after_sync();
        const uint64_t dv = tc::smem_desc(smem_u32(sm + kOffV + sp * kKVBytes), 8192, 1024);
        if (elect_one()) {
#pragma unroll
          for (int part = 0; part < 2; ++part)
#pragma unroll
            for (int kk = 0; kk < kKeys / 16; ++kk)
              tc::mma(tmem + kOCol, dp + (uint64_t)((part * kPBytes + kk * 32) >> 4),
                      dv + (uint64_t)((kk * 2048) >> 4), kIdescPV, jp > 0 || part > 0 || kk > 0);
          tc::commit(bars + kPvDone);
          tc::commit(bars + kEmptyV + sp);
        }
        __syncwarp();
      }
    }
    return true;
  }

  // Wait (bounded) for every MMA issued.
  __device__ void drain() {
    if (elect_one()) tc::commit(bars + kDrain);
    __syncwarp();
    if (!mbar_wait(bars + kDrain, 0) && (threadIdx.x & 31) == 0)
      raise_fault(a.status, PSKV_FAULT_WAIT_TIMEOUT);
  }
};

// One softmax thread per query row (thread i = tensor-memory lane i).
struct RowState {
  float m;  // reference max (log2 units), -inf until a key is seen
  float l;  // sum of exp2(score - m)
};

// Multiply this warp's 128 x 256 O rows in tensor memory by alpha (1 keeps a row).
__device__ __forceinline__ void rescale_o(uint32_t lane_base, float alpha) {
#pragma unroll 1
  for (int c = 0; c < kD / 32; ++c) {
    uint32_t v[32];
    tc::ld32(lane_base + kOCol + 32 * c, v);
    tc::wait_ld();
    tc::reg_fence(v);
#pragma unroll
    for (int k = 0; k < 32; ++k) v[k] = __float_as_uint(__uint_as_float(v[k]) * alpha);
    tc::st32(lane_base + kOCol + 32 * c, v);
    tc::wait_st();
  }
}

// The softmax warps' loop over the partition's tiles.  Returns false on an abort.
__device__ __forceinline__ bool softmax_loop(const TcArgs &a, const TcPlan &pl, unsigned char *sm,
                                             uint64_t *bars, const StageInfo *info, uint32_t tmem,
                                             volatile int *abort_flag, RowState &st) {
  uint64_t *fullK = bars, *fullV = bars + 2;
  uint64_t *s_full = bars + 8, *s_free = bars + 9, *p_full = bars + 10, *pv_done = bars + 11;
  const int lane = threadIdx.x & 31, w = (threadIdx.x >> 5) & 3, i = 32 * w + lane;
  const int col = pl.qb * kRows + i, t = col >> a.group_shift;
  const bool real = t < pl.T;
  const int own = pl.len - pl.T + t;
  const int lim = real ? own + 1 : 0;  // keys below lim, from lo on, are visible
  const int lo = a.window > 0 ? max(0, own - a.window + 1) : 0;
  const uint32_t lane_base = tmem + ((uint32_t)(w * 32) << 16);
  unsigned char *p_hi = sm + kOffP + i * 128, *p_lo = p_hi + kPBytes;
  const float sc = a.scale_log2;
  auto wait_all = [&](uint64_t *bar, uint32_t parity) {
    const bool ok = tc_wait(bar, parity, abort_flag, a.status);
    return __all_sync(0xffffffffu, ok);
  };
  for (int j = 0; j < pl.n; ++j) {
    const int s = j & 1, key0 = (pl.t_begin + j) * kKeys;
    if (!wait_all(s_full, j & 1)) return false;
    if (!wait_all(&fullK[s], (j >> 1) & 1)) return false;  // complete: publishes the record
    const StageInfo inf = info[s];
    __syncwarp();
    if (lane == 0) mbar_arrive(bars + kInfoFree + s);  // the record may be rewritten
    tc::fence_after_sync();
    uint32_t va[32], vb[32];
    tc::ld32(lane_base, va);
    tc::ld32(lane_base + 32, vb);
    tc::wait_ld();
    tc::reg_fence(va);
    tc::reg_fence(vb);
    tc::fence_before_sync();
    __syncwarp();
    if (lane == 0) mbar_arrive(s_free);

    // ---- mask (by selection: scores of keys never loaded may be anything) and tile max
    float x[kKeys];
#pragma unroll
    for (int c = 0; c < 32; ++c) {
      x[c] = __uint_as_float(va[c]) * sc;
      x[32 + c] = __uint_as_float(vb[c]) * sc;
    }
    const bool whole = key0 >= lo && key0 + kKeys <= lim && inf.bad == 0;
    if (!whole) {
#pragma unroll
      for (int c = 0; c < kKeys; ++c) {
        const int k = key0 + c;
        const bool vis = k >= lo && k < lim && !((inf.bad >> (c >> 4)) & 1u);
        x[c] = vis ? x[c] : -CUDART_INF_F;
      }
    }
    float mt = x[0];
#pragma unroll
    for (int c = 1; c < kKeys; ++c) mt = fmaxf(mt, x[c]);
    // The reference max moves only when a score passes it by more than the
    // slack: below that, exp2(score - m) <= 2^8 is exact in float and in the
    // hi + lo weights, so (m, l, O) stays an exact state for any reference.
    float alpha = 1.f;
    bool rescale = false;
    if (mt > st.m + kSlack) {
      rescale = st.m != -CUDART_INF_F;  // with m = -inf the row's O and l are still 0
      alpha = rescale ? exp2f(st.m - mt) : 1.f;
      st.l *= alpha;
      st.m = mt;
    }
    // ---- P = exp2(x - m) as hi + lo bf16 pairs, built in registers while PV(j - 1) runs
    const float u = st.m == -CUDART_INF_F ? 0.f : st.m;
    uint32_t h[kKeys / 2], lw[kKeys / 2];
    float sum = 0.f;
#pragma unroll
    for (int e = 0; e < kKeys / 2; ++e) {
      const float p0 = exp2f(x[2 * e] - u), p1 = exp2f(x[2 * e + 1] - u);
      sum += p0 + p1;
      h[e] = pack_bf16x2(p0, p1);
      lw[e] = pack_bf16x2(p0 - bf16_lo(h[e]), p1 - bf16_hi(h[e]));
    }
    st.l += sum;

    // ---- V rows outside the CTA's keys or in skipped chunks: zero (they meet P = 0)
    if (inf.vlo > 0 || inf.vhi < kKeys || inf.bad != 0) {
      if (!wait_all(&fullV[s], (j >> 1) & 1)) return false;
      const int r = i >> 1;
      if (r < inf.vlo || r >= inf.vhi || ((inf.bad >> (r >> 4)) & 1u)) {
        unsigned char *vrow = sm + kOffV + s * kKVBytes + r * 128 + (i & 1) * 2 * kKVSlab;
#pragma unroll
        for (int sl = 0; sl < 2; ++sl)
#pragma unroll
          for (int q = 0; q < 8; ++q)
            *reinterpret_cast<uint4 *>(vrow + sl * kKVSlab + q * 16) = make_uint4(0, 0, 0, 0);
      }
    }

    // PV(j - 1) must be done before O is rescaled and before P is rewritten
    if (j >= 1 && !wait_all(pv_done, (j - 1) & 1)) return false;
    tc::fence_after_sync();
    if (__any_sync(0xffffffffu, rescale)) rescale_o(lane_base, alpha);
    // rows in the 128-byte swizzled layout: 16-byte chunk cc of row i at cc ^ (i % 8)
#pragma unroll
    for (int cc = 0; cc < kKeys / 8; ++cc) {
      const int off = ((cc ^ (i & 7)) * 16);
      *reinterpret_cast<uint4 *>(p_hi + off) =
          make_uint4(h[4 * cc], h[4 * cc + 1], h[4 * cc + 2], h[4 * cc + 3]);
      *reinterpret_cast<uint4 *>(p_lo + off) =
          make_uint4(lw[4 * cc], lw[4 * cc + 1], lw[4 * cc + 2], lw[4 * cc + 3]);
    }
    tc::fence_smem_for_async();
    tc::fence_before_sync();
    __syncwarp();
    if (lane == 0) mbar_arrive(p_full);
  }
  return true;
}

// Query row of block row i (output / partial row index without the partition).
__device__ __forceinline__ size_t query_row(const TcArgs &a, const TcPlan &pl, int i, bool *real) {
  const int col = pl.qb * kRows + i, t = col >> a.group_shift;
  *real = t < pl.T;
  const int h = (pl.g << a.group_shift) + (col & ((1 << a.group_shift) - 1));
  return ((size_t)pl.r0 + (*real ? t : 0)) * a.num_q_heads + h;
}

// Write row i's result: o / l to `out` (direct) or the partial (m, l, o).
__device__ __forceinline__ void write_rows(const TcArgs &a, const TcPlan &pl, uint32_t tmem,
                                           const RowState &st) {
  const int w = (threadIdx.x >> 5) & 3, i = 32 * w + (threadIdx.x & 31);
  const uint32_t lane_base = tmem + ((uint32_t)(w * 32) << 16);
  bool real;
  const size_t qrow = query_row(a, pl, i, &real);
  const bool empty = st.m == -CUDART_INF_F;
  const float inv = empty ? 0.f : 1.f / st.l;
  const size_t prow = qrow * a.num_splits + pl.p;
#pragma unroll 1
  for (int c = 0; c < kD / 32; ++c) {
    uint32_t v[32];
    tc::ld32(lane_base + kOCol + 32 * c, v);
    tc::wait_ld();
    tc::reg_fence(v);
    if (!real) continue;
    if (a.direct) {
      if (a.out_dtype == PSKV_DTYPE_BF16) {
        uint4 *dst = reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(a.out) + qrow * kD +
                                               32 * c);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint32_t wd[4];
#pragma unroll
          for (int e = 0; e < 4; ++e)
            wd[e] = pack_bf16x2(__uint_as_float(v[8 * q + 2 * e]) * inv,
                                __uint_as_float(v[8 * q + 2 * e + 1]) * inv);
          dst[q] = make_uint4(wd[0], wd[1], wd[2], wd[3]);
        }
      } else {
        float4 *dst = reinterpret_cast<float4 *>(static_cast<float *>(a.out) + qrow * kD + 32 * c);
#pragma unroll
        for (int q = 0; q < 8; ++q)
          dst[q] = make_float4(__uint_as_float(v[4 * q]) * inv, __uint_as_float(v[4 * q + 1]) * inv,
                               __uint_as_float(v[4 * q + 2]) * inv,
                               __uint_as_float(v[4 * q + 3]) * inv);
      }
    } else {
      float4 *dst = reinterpret_cast<float4 *>(a.ws_o + prow * kD + 32 * c);
#pragma unroll
      for (int q = 0; q < 8; ++q)
        dst[q] = make_float4(__uint_as_float(v[4 * q]), __uint_as_float(v[4 * q + 1]),
                             __uint_as_float(v[4 * q + 2]), __uint_as_float(v[4 * q + 3]));
    }
  }
  if (!real) return;
  if (a.direct) {
    if (empty) raise_fault(a.status, PSKV_FAULT_EMPTY_ROW);
  } else {
    a.ws_m[prow] = empty ? -CUDART_INF_F : st.m * kLn2;
    a.ws_l[prow] = st.l;
  }
}

// A block whose partition holds no tile: empty partial states, or (one
// partition) zeros flagged as empty rows.
__device__ __forceinline__ void write_empty(const TcArgs &a, const TcPlan &pl) {
  for (int i = threadIdx.x; i < kRows; i += blockDim.x) {
    bool real;
    const size_t qrow = query_row(a, pl, i, &real);
    if (!real) continue;
    if (a.direct) {
      for (int d = 0; d < kD; ++d) {
        if (a.out_dtype == PSKV_DTYPE_BF16)
          static_cast<__nv_bfloat16 *>(a.out)[qrow * kD + d] = __float2bfloat16_rn(0.f);
        else
          static_cast<float *>(a.out)[qrow * kD + d] = 0.f;
      }
      raise_fault(a.status, PSKV_FAULT_EMPTY_ROW);
    } else {
      const size_t prow = qrow * a.num_splits + pl.p;
      a.ws_m[prow] = -CUDART_INF_F;
      a.ws_l[prow] = 0.f;
    }
  }
}

}  // namespace

__global__ void __launch_bounds__(kThreads, 1)
    pskv_attn_tc_kernel(const TcArgs a, const __grid_constant__ CUtensorMap qmap,
                        const __grid_constant__ CUtensorMap kmap,
                        const __grid_constant__ CUtensorMap vmap) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char *sm = reinterpret_cast<unsigned char *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  uint64_t *bars = reinterpret_cast<uint64_t *>(sm + kOffBar);
  StageInfo *info = reinterpret_cast<StageInfo *>(sm + kOffInfo);
  uint32_t *slot = reinterpret_cast<uint32_t *>(sm + kOffSlot);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + kOffAbort);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // every read of caller memory comes after the previous kernel's writes
  pdl_wait();
  pdl_launch_dependents();
  const TcPlan pl = make_plan(a);
  if (!pl.ok && threadIdx.x == 0 && blockIdx.x == 0 && blockIdx.y == 0)
    raise_fault(a.status, PSKV_FAULT_BAD_LENGTH);
  if (pl.qb * kRows >= (pl.T << a.group_shift)) return;  // no query row in this block
  if (pl.n <= 0) {
    write_empty(a, pl);
    return;
  }

  Loader ld(a, pl, &qmap, &kmap, &vmap, sm, bars, info, abort_flag);
  if (warp == 1) {
    // the copy warp sets up the barriers and requests Q and the first tiles at once
    if (lane == 0) {
      for (int k = 0; k < 8; ++k) mbar_init(&bars[k], 1);  // fullK, fullV, emptyK, emptyV
      mbar_init(&bars[kSFull], 1);   // MMA commit
      mbar_init(&bars[kSFree], 4);   // one arrive per softmax warp
      mbar_init(&bars[kPFull], 4);   // one arrive per softmax warp
      mbar_init(&bars[kPvDone], 1);  // MMA commit
      mbar_init(&bars[kDrain], 1);   // MMA commit
      mbar_init(&bars[kQFull], 1);
      mbar_init(&bars[kInfoFree], 4);      // one arrive per softmax warp
      mbar_init(&bars[kInfoFree + 1], 4);
      *abort_flag = 0;
      mbar_fence_init();
    }
    __syncwarp();
    ld.prologue();
  } else if (warp == 0) {
    tc::alloc(slot, kTmemCols);
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *slot;

  if (warp == 0) {
    Issuer is{a, pl, sm, bars, abort_flag};
    is.run(tmem);
    is.drain();  // every MMA done before the memory is released
  } else if (warp == 1) {
    ld.run();
    ld.drain();  // every copy landed before the CTA leaves
  } else {
    RowState st;
    st.m = -CUDART_INF_F;
    st.l = 0.f;
    if (softmax_loop(a, pl, sm, bars, info, tmem, abort_flag, st)) {
      const bool ok = tc_wait(bars + kPvDone, (pl.n - 1) & 1, abort_flag, a.status);
      if (__all_sync(0xffffffffu, ok)) {
        tc::fence_after_sync();
        write_rows(a, pl, tmem, st);
      }
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    tc::fence_after_sync();
    tc::dealloc(tmem, kTmemCols);
  }
}

namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
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

// The pool region as a 2-D tensor of `rows` rows of 256 bf16, read in boxes
// of 64 columns x box_rows rows in the 128-byte swizzled layout.
bool make_map(CUtensorMap *m, const void *region, long long rows, int box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)kD, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)kD * 2};
  const cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  const cuuint32_t elem[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(region), dims, strides,
             box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The packed queries [rows][Hq][256] as a 3-D tensor (columns, heads, rows),
// read in boxes of 64 columns x G heads x 128 / G rows.
bool make_qmap(CUtensorMap *m, const void *q, int rows, int heads, int group) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)kD, (cuuint64_t)heads, (cuuint64_t)rows};
  const cuuint64_t strides[2] = {(cuuint64_t)kD * 2, (cuuint64_t)kD * 2 * heads};
  const cuuint32_t box[3] = {64, (cuuint32_t)group, (cuuint32_t)(kRows / group)};
  const cuuint32_t elem[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(q), dims, strides, box,
             elem, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_attn_tc(const TcArgs &a, const void *k_pool, const void *v_pool, dim3 grid,
                           cudaStream_t stream) {
  static bool attr_set[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (!(dev >= 0 && dev < 64 && attr_set[dev])) {
    e = cudaFuncSetAttribute(pskv_attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kSmemBytes);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_set[dev] = true;
  }
  const long long rows = a.num_pages * a.num_kv_heads * a.page_size;
  CUtensorMap qm, km, vm;
  if (!make_qmap(&qm, a.q, a.total_rows, a.num_q_heads, 1 << a.group_shift) ||
      !make_map(&km, k_pool, rows, a.box_rows) || !make_map(&vm, v_pool, rows, a.box_rows))
    return cudaErrorInvalidValue;
  return launch_pdl(pskv_attn_tc_kernel, grid, dim3(kThreads), (size_t)kSmemBytes, stream, a, qm,
                    km, vm);
}

}  // namespace pskv
