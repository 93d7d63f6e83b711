// attn_tc.cu -- paged attention of many query rows per KV head on the fifth-
// generation tensor cores (tcgen05, tensor memory, tensor copies).
//
// Serves paged prefill (pegainfer #1057, Description: the sliding family's
// prompt rows read through a windowed varlen kernel with a window lower bound)
// at head dim 256, bf16 pools in the split format.  One CTA takes a block of
// 128 query rows of one (row, KV head): row i of the block is query column
// qb * 128 + i of the row's chunk (token column / G, head column % G), and a
// partition of the keys those tokens can see.  Per tile j of 64 keys:
//   S  = Q K^T    M = 128 rows, N = 64 keys, K = 256 (16 MMAs)
//   softmax       one thread per query row reads its 64 scores, masks them
//                 (causal, window, keys outside the CTA's range), keeps the
//                 row's reference max and sum (exp2 units; the max moves only
//                 past a slack of 8, as in the decode kernels) and writes P
//                 as a bf16 hi + lo pair over the scores it read
//   O += P V      M = 128, N = 256, K = 64 keys, hi then lo (8 MMAs)
// Tensor memory (512 columns): Q (bf16 pairs) at [0, 128), two score / P
// regions at [128, 192) and [192, 256) (tile j uses region j % 2), O (f32) at
// [256, 512).  Q and P feed the MMAs from tensor memory; K and V tiles arrive
// by tensor copies in the 128-byte swizzled layout, three stages each.  Warp 0
// issues the MMAs, warp 1 the K copies and warp 6 the V copies (so that a K
// tile is requested three tiles ahead whatever the V side waits for); warps
// 2-5 stage Q and run the softmax and the epilogue (warp w owns tensor-memory
// lanes 32 (w % 4) .. + 31).  The issuing warps are the oldest of their
// schedulers, so the softmax's long instruction streams do not hold them
// back.  Every wait is bounded; on expiry the CTA flags
// PSKV_FAULT_WAIT_TIMEOUT, lets what it issued finish and frees its tensor
// memory.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <math_constants.h>

#include "attn_tc.h"
#include "pskv_internal.cuh"
#include "tc_common.cuh"
#include "tc_ops.cuh"

namespace pskv {

namespace {

using tc::elect_one;
using tc::ex2;
using tc::make_map;
using tc::PageCache;
using tc::tc_wait;
using tc::warp_wait;

constexpr int kD = 256;                     // head-dim columns per CTA
constexpr int kRows = 128;                  // query rows per CTA (MMA M)
constexpr int kKeys = 64;                   // keys per tile (MMA N of S, K of PV)
constexpr int kKVSlab = kKeys * 128;        // bytes of one 64-column slab of a K or V tile
constexpr int kKVBytes = 4 * kKVSlab;       // 32 KB
constexpr int kStages = 3;                  // most K or V stages (barrier and record slots)
constexpr int kXBytes = kRows * kKeys * 4;  // one block of partial scores (32 KB)
constexpr int kQSlab = kRows * 128;         // 64 columns of Q's 128 rows (16 KB)
constexpr int kTmemCols = 512;
constexpr int kQCol = 0;                    // Q: 256 bf16 = 128 columns
constexpr int kSCol = 128;                  // score / P region r at kSCol + 64 r
constexpr int kOCol = 256;                  // O: 256 f32 columns
constexpr float kSlack = 8.f;               // reference-max slack (log2 units)

// shared memory (offsets from a 1,024-byte aligned base): K stages, V stages,
// (CTA pair) two blocks of the peer's partial scores, barriers, stage records
constexpr int kOffK = 0;  // K stage s at kOffK + s * kKVBytes

// barrier slots
enum : int {
  kFullK = 0,                   // [3] K tile landed (copy bytes)
  kFullV = kFullK + kStages,    // [3] V tile landed
  kEmptyK = kFullV + kStages,   // [3] S of the stage's tile done (MMA commit)
  kEmptyV = kEmptyK + kStages,  // [3] PV of the stage's tile done (MMA commit)
  kInfoFree = kEmptyV + kStages,  // [3] the softmax warps read the stage's record
  kSFull = kInfoFree + kStages,   // [2] S of region r done (MMA commit)
  kPFull = kSFull + 2,            // [2] P of region r written (softmax warps)
  kPvDone = kPFull + 2,           // [2] PV of region r's tile done (MMA commit)
  kDrain = kPvDone + 2,           // every MMA done (MMA commit)
  kQReady = kDrain + 1,           // Q written to tensor memory (softmax warps)
  kXFull = kQReady + 1,           // [2] the peer's partial scores arrived (CTA pair)
  kXFree = kXFull + 2,            // [2] the peer read the partial scores sent to it
  kSReady = kXFree + 2,           // [2] the full scores of region r are in place (CTA pair)
  kQFull = kSReady + 2,           // Q's tensor copy landed
  kNumBars = kQFull + 1
};

// Head dim 256: one CTA.  Head dim 512: a cluster of two CTAs, rank c holding
// columns [256 c, 256 c + 256) of Q, K, V and O (two V stages, to make room
// for the block of partial scores received from the peer and the block staged
// for sending to it).
template <bool kPair>
struct Lay {
  static constexpr int kDT = kPair ? 2 * kD : kD;  // the pool's head dim
  // warps: 0 MMA, 1 K copies, 2-5 softmax, 6 V copies, (pair) 7-10 score exchange
  static constexpr int kThreads = kPair ? 352 : 224;
  static constexpr int kStagesK = kPair ? 2 : 3;
  static constexpr int kStagesV = kPair ? 2 : 3;
  static constexpr int kOffV = kOffK + kStagesK * kKVBytes;  // V stage s at kOffV + s * kKVBytes
  // the first of the two V stages that take Q's tensor copy at the start (the
  // pair's V stages are all it has; head dim 256 keeps stage 0 for V(0))
  static constexpr int kQStage = kPair ? 0 : 1;
  static constexpr int kOffX = kOffV + kStagesV * kKVBytes;  // received partial scores [2]
  static constexpr int kOffXs = kOffX + (kPair ? 2 * kXBytes : 0);  // partial scores to send
  static constexpr int kOffBar = kOffXs + (kPair ? kXBytes : 0);
  static constexpr int kOffInfo = kOffBar + kNumBars * 8;   // StageInfo[3]
  static constexpr int kOffSlot = kOffInfo + kStages * 16;  // tensor-memory address
  static constexpr int kOffAbort = kOffSlot + 4;
  static constexpr int kSmemBytes = kOffAbort + 4 + 1024;  // + alignment of the dynamic base
  static_assert(kSmemBytes <= 232448, "shared memory per CTA");
};

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

__device__ __forceinline__ TcPlan make_plan(const TcArgs &a, int x) {
  TcPlan pl;
  // heavier (later) query blocks first: under causality they see more keys
  pl.qb = a.qblocks - 1 - x % a.qblocks;
  pl.p = x / a.qblocks;
  pl.g = blockIdx.y;
  pl.b = blockIdx.z;
  pl.ok = true;
  // a verify window (no offsets): num_tokens query rows per table row
  const int c0 = a.cu_q ? a.cu_q[pl.b] : pl.b * a.num_tokens;
  const int c1 = a.cu_q ? a.cu_q[pl.b + 1] : c0 + a.num_tokens;
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


// ---- the CTA pair: distributed shared memory and cluster-scope barriers
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// The same shared-memory offset in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_to(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}
// Arrive on a barrier of another CTA, releasing this thread's writes at cluster scope.
__device__ __forceinline__ void arrive_cluster(uint32_t remote_bar) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(remote_bar)
               : "memory");
}
__device__ __forceinline__ bool try_wait_cluster(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], "
      "%2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait with cluster-scope acquire, one answer for the whole warp.
__device__ __forceinline__ bool warp_wait_cluster(uint64_t *bar, uint32_t parity,
                                                  volatile int *abort_flag, int32_t *status) {
  bool ok = !*abort_flag;
  if (ok && !try_wait_cluster(bar, parity)) {
    ok = false;
    for (uint32_t i = 0; i < kWaitPolls; ++i)
      if (try_wait_cluster(bar, parity)) {
        ok = true;
        break;
      }
    if (!ok) {
      *abort_flag = 1;
      raise_fault(status, PSKV_FAULT_WAIT_TIMEOUT);
    }
  }
  return __all_sync(0xffffffffu, ok);
}
// Bulk copy of this CTA's shared memory into the peer's (both addresses
// 16-byte aligned, bytes a multiple of 16), completion counted on the peer's
// barrier `remote_bar`; the copy's reads are tracked by this thread's bulk group.
__device__ __forceinline__ void bulk_s2peer(uint32_t remote_dst, uint32_t local_src, uint32_t bytes,
                                            uint32_t remote_bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, "
      "[%3];\n\tcp.async.bulk.commit_group;" ::"r"(remote_dst),
      "r"(local_src), "r"(bytes), "r"(remote_bar)
      : "memory");
}
// Wait until every bulk copy this thread committed has read its source.
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;"
               ::: "memory");
}

// A copy warp (all lanes converged; one elected lane issues), for K or for V.
// Tile j's K and V go to stage j % 3:
//   K(j) once S(j - 3) has released the stage and the softmax warps have read
//        the stage's record of tile j - 3;
//   V(j) once PV(j - 3) has released the stage.
// The first three K tiles are requested before the CTA's first barrier.
template <bool kPair>
struct Loader {
  using L = Lay<kPair>;
  const TcArgs &a;
  const TcPlan &pl;
  const CUtensorMap *kmap, *vmap;
  unsigned char *sm;
  uint64_t *bars;
  StageInfo *info;
  volatile int *abort_flag;
  int lane;
  int n_slots;  // table slots the CTA's keys use
  PageCache pages;  // each copy warp's own
  int issued = 0;
  int col0;         // first head-dim column this CTA holds

  __device__ Loader(const TcArgs &a_, const TcPlan &pl_, const CUtensorMap *km,
                    const CUtensorMap *vm, unsigned char *sm_, uint64_t *bars_, StageInfo *info_,
                    volatile int *ab, int col0_)
      : a(a_), pl(pl_), kmap(km), vmap(vm), sm(sm_), bars(bars_), info(info_), abort_flag(ab),
        col0(col0_) {
    lane = threadIdx.x & 31;
    n_slots = (pl.k_hi + a.page_size - 1) / a.page_size;
  }

  // Issue the tensor copies of tile j into its K or V stage: 16- or 64-row
  // chunks, each in four 64-column slabs; chunks with no row in the CTA's key
  // range are not loaded, nor are chunks whose page id lies outside the pool
  // (bit c of the bad mask per 16 rows).  The K copy writes the stage's record
  // before the barrier is armed (the arrive releases it).
  __device__ void load(int j, bool is_v) {
    const int st = j % (is_v ? L::kStagesV : L::kStagesK);
    const int key0 = (pl.t_begin + j) * kKeys;
    const int vlo = max(0, pl.k_lo - key0), vhi = min(kKeys, pl.k_hi - key0);
    const int32_t *tbl = a.page_tables + (size_t)pl.b * a.table_stride;
    const int br = a.box_rows;
    uint32_t bad = 0, bytes = 0;
    int pg[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      pg[c] = -1;
      if (c * br >= kKeys) continue;
      if ((c + 1) * br <= vlo || c * br >= vhi) continue;  // no row of the chunk is in range
      const int page = pages.get(tbl, (key0 + c * br) / a.page_size, n_slots, lane);
      if (page < 0 || (long long)page >= a.num_pages) {
        bad |= (br == kKeys ? 0xFu : 1u << c);
        continue;
      }
      pg[c] = page;
      bytes += (uint32_t)(br * 128 * 4);
    }
    unsigned char *dst = sm + (is_v ? L::kOffV : kOffK) + st * kKVBytes;
    uint64_t *bar = bars + (is_v ? kFullV : kFullK) + st;
    if (elect_one()) {
      if (bad) raise_fault(a.status, PSKV_FAULT_BAD_PAGE);
      if (!is_v) {
        info[st].vlo = vlo;
        info[st].vhi = vhi;
        info[st].bad = bad;
      }
      mbar_arrive_expect_tx(bar, bytes);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        if (pg[c] < 0) continue;
        const int key = key0 + c * br;
        const int y = (pg[c] * a.num_kv_heads + pl.g) * a.page_size + key % a.page_size;
#pragma unroll
        for (int sl = 0; sl < 4; ++sl)
          tc::tma_load_2d(dst + sl * kKVSlab + c * br * 128, is_v ? vmap : kmap, col0 + sl * 64, y,
                          bar);
      }
    }
    __syncwarp();
    issued = j + 1;
  }

  __device__ bool prologue(bool is_v) {
    for (int j = 0; j < (is_v ? L::kStagesV : L::kStagesK) && j < pl.n; ++j) {
      // (V stages kQStage and on hold Q's tensor copy until Q is in tensor memory)
      if (is_v && j == L::kQStage && !wait(kQReady, 0)) return false;
      load(j, is_v);
    }
    return true;
  }

  __device__ bool run(bool is_v) {
    const int S = is_v ? L::kStagesV : L::kStagesK;
    for (int j = S; j < pl.n; ++j) {
      const int st = j % S;
      const uint32_t ph = ((j - S) / S) & 1;  // the stage's previous use
      if (is_v) {
        if (!wait(kEmptyV + st, ph)) return false;
      } else {
        if (!wait(kEmptyK + st, ph) || !wait(kInfoFree + st, ph)) return false;
      }
      load(j, is_v);
    }
    return true;
  }

  __device__ bool wait(int slot, uint32_t parity) {
    return warp_wait(bars + slot, parity, abort_flag, a.status);
  }

  // Wait (bounded) for the last copy issued into each stage.
  __device__ void drain(bool is_v) {
    const int S = is_v ? L::kStagesV : L::kStagesK;
    for (int j = max(0, issued - S); j < issued; ++j)
      mbar_wait(bars + (is_v ? kFullV : kFullK) + j % S, (j / S) & 1);
  }
};

// The MMA warp (all lanes converged; one elected lane issues).  Per tile j:
//   S(j) = Q K(j)^T into region j % 2 once K(j) has landed and PV(j - 2) has
//        consumed the P that region held;
//   O += P(j - 1) V(j - 1) once P(j - 1) is written and V(j - 1) has landed.
template <bool kPair>
struct Issuer {
  using L = Lay<kPair>;
  const TcArgs &a;
  const TcPlan &pl;
  unsigned char *sm;
  uint64_t *bars;
  volatile int *abort_flag;

  __device__ bool wait(int slot, uint32_t parity) {
    return warp_wait(bars + slot, parity, abort_flag, a.status);
  }

  __device__ bool run(uint32_t tmem) {
    const int n = pl.n;
    if (!wait(kQReady, 0)) return false;
    for (int j = 0; j <= n; ++j) {
      if (j < n) {
        const int st = j % L::kStagesK, r = j & 1;
        if (!wait(kFullK + st, (j / L::kStagesK) & 1)) return false;
        if (j >= 2 && !wait(kPvDone + r, ((j - 2) >> 1) & 1)) return false;
        tc::fence_after_sync();
        const uint64_t dk = tc::smem_desc(smem_u32(sm + kOffK + st * kKVBytes), 16, 1024);
        if (elect_one()) {
          // A = Q from tensor memory (8 columns per 16 elements), B = K (K-major)
#pragma unroll
          for (int kk = 0; kk < kD / 16; ++kk)
            tc::mma_ts(tmem + kSCol + 64 * r, tmem + kQCol + 8 * kk,
                       dk + (uint64_t)(((kk >> 2) * kKVSlab + (kk & 3) * 32) >> 4), kIdescS,
                       kk > 0);
          tc::commit(bars + kSFull + r);
          tc::commit(bars + kEmptyK + st);
        }
        __syncwarp();
      }
      if (j >= 1) {
        const int jp = j - 1, st = jp % L::kStagesV, r = jp & 1;
        if (!wait(kPFull + r, (jp >> 1) & 1)) return false;
        if (!wait(kFullV + st, (jp / L::kStagesV) & 1)) return false;
        tc::fence_after_sync();
        const uint64_t dv = tc::smem_desc(smem_u32(sm + L::kOffV + st * kKVBytes), 8192, 1024);
        if (elect_one()) {
          // A = P hi (columns 0-31 of the region), then P lo (32-63); B = V (MN-major)
#pragma unroll
          for (int part = 0; part < 2; ++part)
#pragma unroll
            for (int kk = 0; kk < kKeys / 16; ++kk)
              tc::mma_ts(tmem + kOCol, tmem + kSCol + 64 * r + 32 * part + 8 * kk,
                         dv + (uint64_t)((kk * 2048) >> 4), kIdescPV,
                         jp > 0 || part > 0 || kk > 0);
          tc::commit(bars + kPvDone + r);
          tc::commit(bars + kEmptyV + st);
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

// One softmax thread per query row (thread = tensor-memory lane).
struct RowState {
  float m;  // reference max (log2 units), -inf until a key is seen
  float l;  // sum of exp2(score - m)
};

// Query row of block row i (output / partial row index without the partition).
__device__ __forceinline__ size_t query_row(const TcArgs &a, const TcPlan &pl, int i, bool *real) {
  const int col = pl.qb * kRows + i, t = col >> a.group_shift;
  *real = t < pl.T;
  const int h = (pl.g << a.group_shift) + (col & ((1 << a.group_shift) - 1));
  return ((size_t)pl.r0 + (*real ? t : 0)) * a.num_q_heads + h;
}

// Q into tensor memory: this thread's row (its CTA's 256 columns) as 128
// columns of bf16 pairs, read from the block's tensor copy (rows past the
// chunk hold other rows' queries or zeros, and see no key).
template <bool kPair>
__device__ __forceinline__ bool stage_q(const TcArgs &a, const TcPlan &pl, unsigned char *sm,
                                        uint64_t *bars, uint32_t tmem, int col0,
                                        volatile int *abort_flag) {
  const int w = (threadIdx.x >> 5) & 3, i = 32 * w + (threadIdx.x & 31);
  const uint32_t lane_base = tmem + ((uint32_t)(w * 32) << 16);
  {
    // the block's 128 rows (this CTA's columns) arrived by one tensor copy into
    // two V stages: four 64-column slabs of 128 rows, 128-byte swizzled
    if (!warp_wait(bars + kQFull, 0, abort_flag, a.status)) return false;
    const unsigned char *qs =
        sm + Lay<kPair>::kOffV + Lay<kPair>::kQStage * kKVBytes + i * 128;
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      uint32_t v[32];
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const uint4 x = *reinterpret_cast<const uint4 *>(qs + b * kQSlab + ((c ^ (i & 7)) << 4));
        v[4 * c] = x.x;
        v[4 * c + 1] = x.y;
        v[4 * c + 2] = x.z;
        v[4 * c + 3] = x.w;
      }
      tc::st32(lane_base + kQCol + 32 * b, v);
    }
    tc::wait_st();
    return true;
  }
}

// Multiply this warp's rows of O in tensor memory by alpha (1 keeps a row).
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
template <bool kPair>
__device__ __forceinline__ bool softmax_loop(const TcArgs &a, const TcPlan &pl, unsigned char *sm,
                                             uint64_t *bars, const StageInfo *info, uint32_t tmem,
                                             volatile int *abort_flag, RowState &st,
                                             uint32_t rank) {
  using L = Lay<kPair>;
  const int lane = threadIdx.x & 31, w = (threadIdx.x >> 5) & 3, i = 32 * w + lane;
  const int col = pl.qb * kRows + i, t = col >> a.group_shift;
  const bool real = t < pl.T;
  const int own = pl.len - pl.T + t;
  const int lim = real ? own + 1 : 0;  // keys below lim, from lo on, are visible
  const int lo = a.window > 0 ? max(0, own - a.window + 1) : 0;
  const uint32_t lane_base = tmem + ((uint32_t)(w * 32) << 16);
  const float sc = a.scale_log2;
  auto wait_all = [&](int slot, uint32_t parity) {
    return warp_wait(bars + slot, parity, abort_flag, a.status);
  };
  for (int j = 0; j < pl.n; ++j) {
    const int sk = j % L::kStagesK, sv = j % L::kStagesV, r = j & 1;
    const int key0 = (pl.t_begin + j) * kKeys;
    const uint32_t region = lane_base + kSCol + 64 * r;
    // (CTA pair: the exchange warps put the full scores in place)
    if (!wait_all((kPair ? kSReady : kSFull) + r, (j >> 1) & 1)) return false;
    if (!wait_all(kFullK + sk, (j / L::kStagesK) & 1)) return false;  // publishes the record
    const StageInfo inf = info[sk];
    __syncwarp();
    if (lane == 0) mbar_arrive(bars + kInfoFree + sk);  // the record may be rewritten
    tc::fence_after_sync();
    uint32_t va[32], vb[32];
    tc::ld32(region, va);
    tc::ld32(region + 32, vb);
    tc::wait_ld();
    tc::reg_fence(va);
    tc::reg_fence(vb);

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
      alpha = rescale ? ex2(st.m - mt) : 1.f;
      st.l *= alpha;
      st.m = mt;
    }

    // ---- P = exp2(x - m) as hi + lo bf16 pairs
    const float u = st.m == -CUDART_INF_F ? 0.f : st.m;
    uint32_t h[kKeys / 2], lw[kKeys / 2];
    float sum = 0.f;
#pragma unroll
    for (int e = 0; e < kKeys / 2; ++e) {
      const float p0 = ex2(x[2 * e] - u), p1 = ex2(x[2 * e + 1] - u);
      sum += p0 + p1;
      h[e] = pack_bf16x2(p0, p1);
      lw[e] = pack_bf16x2(p0 - bf16_lo(h[e]), p1 - bf16_hi(h[e]));
    }
    st.l += sum;

    // ---- V rows outside the CTA's keys or in skipped chunks: zero (they meet P = 0).
    // Every tile's V barrier is waited, in order, so that each wait's parity
    // names the phase it means.
    if (!wait_all(kFullV + sv, (j / L::kStagesV) & 1)) return false;
    if (inf.vlo > 0 || inf.vhi < kKeys || inf.bad != 0) {
      const int rr = i >> 1;
      if (rr < inf.vlo || rr >= inf.vhi || ((inf.bad >> (rr >> 4)) & 1u)) {
        unsigned char *vrow = sm + L::kOffV + sv * kKVBytes + rr * 128 + (i & 1) * 2 * kKVSlab;
#pragma unroll
        for (int sl = 0; sl < 2; ++sl)
#pragma unroll
          for (int q = 0; q < 8; ++q)
            *reinterpret_cast<uint4 *>(vrow + sl * kKVSlab + q * 16) = make_uint4(0, 0, 0, 0);
      }
      tc::fence_smem_for_async();
    }

    // ---- O of the rows whose reference moved: rescaled once PV(j - 1) is done
    if (__any_sync(0xffffffffu, rescale)) {
      // PV(j - 3) is known done (S(j - 1) waited for it), so this parity is unambiguous
      if (!wait_all(kPvDone + ((j - 1) & 1), ((j - 1) >> 1) & 1)) return false;
      tc::fence_after_sync();
      rescale_o(lane_base, alpha);
    }
    // P over the scores it came from: hi at columns 0-31 of the region, lo at 32-63
    tc::st32(region, h);
    tc::st32(region + 32, lw);
    tc::wait_st();
    tc::fence_before_sync();
    __syncwarp();
    if (lane == 0) mbar_arrive(bars + kPFull + r);
  }
  return true;
}

// The CTA pair's score exchange (warps 7-10; warp w owns tensor-memory lanes
// 32 (w % 4) .. + 31): the scores are the sum of the two CTAs' products over
// their halves of the head dim.  Per tile j each warp reads its 32 rows of
// partial scores from the tile's region, stages them (row i, 16-byte chunk q
// at q ^ (i % 16) against bank conflicts) and one bulk copy sends them into
// the peer's receive block j % 2, completing on the peer's barrier; the
// peer's rows arrive the same way, are added, and the full scores go back
// into the region for the softmax warps.  Both CTAs then hold the same bits
// and run the same softmax.  Exchanging tile j + 1 overlaps the softmax of j.
__device__ __forceinline__ bool exchange_loop(const TcArgs &a, const TcPlan &pl, unsigned char *sm,
                                              uint64_t *bars, uint32_t tmem,
                                              volatile int *abort_flag, uint32_t rank) {
  using L = Lay<true>;
  const int lane = threadIdx.x & 31, w = (threadIdx.x >> 5) & 3, i = 32 * w + lane;
  const uint32_t lane_base = tmem + ((uint32_t)(w * 32) << 16);
  const uint32_t peer = rank ^ 1u;
  const uint32_t rows_off = (uint32_t)(32 * w) * (kKeys * 4);  // this warp's rows in a block
  auto wait_all = [&](int slot, uint32_t parity) {
    return warp_wait(bars + slot, parity, abort_flag, a.status);
  };
  auto wait_cl = [&](int slot, uint32_t parity) {
    return warp_wait_cluster(bars + slot, parity, abort_flag, a.status);
  };
  unsigned char *xs = sm + L::kOffXs + i * (kKeys * 4);
  for (int j = 0; j < pl.n; ++j) {
    const int r = j & 1, xb = j & 1;
    const uint32_t region = lane_base + kSCol + 64 * r;
    if (!wait_all(kSFull + r, (j >> 1) & 1)) return false;  // this CTA's partial S(j)
    tc::fence_after_sync();
    uint32_t va[32], vb[32];
    tc::ld32(region, va);
    tc::ld32(region + 32, vb);
    tc::wait_ld();
    tc::reg_fence(va);
    tc::reg_fence(vb);
    if (lane == 0) bulk_wait_read();  // the previous send has read the staging rows
    __syncwarp();
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      *reinterpret_cast<uint4 *>(xs + 16 * (q ^ (i & 15))) =
          make_uint4(va[4 * q], va[4 * q + 1], va[4 * q + 2], va[4 * q + 3]);
      *reinterpret_cast<uint4 *>(xs + 16 * ((q + 8) ^ (i & 15))) =
          make_uint4(vb[4 * q], vb[4 * q + 1], vb[4 * q + 2], vb[4 * q + 3]);
    }
    tc::fence_smem_for_async();
    __syncwarp();
    // the peer has read what this CTA sent into its block xb for tile j - 2
    if (j >= 2 && !wait_cl(kXFree + xb, ((j - 2) >> 1) & 1)) return false;
    if (lane == 0) {
      bulk_s2peer(map_to(smem_u32(sm + L::kOffX + xb * kXBytes) + rows_off, peer),
                  smem_u32(sm + L::kOffXs) + rows_off, 32 * kKeys * 4,
                  map_to(smem_u32(bars + kXFull + xb), peer));
      mbar_arrive_expect_tx(bars + kXFull + xb, 32 * kKeys * 4);  // this warp's rows from the peer
    }
    if (!wait_cl(kXFull + xb, (j >> 1) & 1)) return false;  // the peer's partial of tile j
    const unsigned char *xo = sm + L::kOffX + xb * kXBytes + i * (kKeys * 4);
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const uint4 t = *reinterpret_cast<const uint4 *>(xo + 16 * (q ^ (i & 15)));
      const uint4 u = *reinterpret_cast<const uint4 *>(xo + 16 * ((q + 8) ^ (i & 15)));
      va[4 * q] = __float_as_uint(__uint_as_float(va[4 * q]) + __uint_as_float(t.x));
      va[4 * q + 1] = __float_as_uint(__uint_as_float(va[4 * q + 1]) + __uint_as_float(t.y));
      va[4 * q + 2] = __float_as_uint(__uint_as_float(va[4 * q + 2]) + __uint_as_float(t.z));
      va[4 * q + 3] = __float_as_uint(__uint_as_float(va[4 * q + 3]) + __uint_as_float(t.w));
      vb[4 * q] = __float_as_uint(__uint_as_float(vb[4 * q]) + __uint_as_float(u.x));
      vb[4 * q + 1] = __float_as_uint(__uint_as_float(vb[4 * q + 1]) + __uint_as_float(u.y));
      vb[4 * q + 2] = __float_as_uint(__uint_as_float(vb[4 * q + 2]) + __uint_as_float(u.z));
      vb[4 * q + 3] = __float_as_uint(__uint_as_float(vb[4 * q + 3]) + __uint_as_float(u.w));
    }
    tc::fence_smem_for_async();  // these reads before the peer's next copy into the block
    __syncwarp();
    if (lane == 0) arrive_cluster(map_to(smem_u32(bars + kXFree + xb), peer));
    tc::st32(region, va);
    tc::st32(region + 32, vb);
    tc::wait_st();
    tc::fence_before_sync();
    __syncwarp();
    if (lane == 0) mbar_arrive(bars + kSReady + r);
  }
  return true;
}

// Write row i's result (this CTA's columns): o / l to `out` (direct) or the
// partial (m, l, o); the pair's rank 0 writes m and l.
template <bool kPair>
__device__ __forceinline__ void write_rows(const TcArgs &a, const TcPlan &pl, uint32_t tmem,
                                           const RowState &st, int col0) {
  constexpr int DT = Lay<kPair>::kDT;
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
        uint4 *dst = reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(a.out) + qrow * DT +
                                               col0 + 32 * c);
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
        float4 *dst =
            reinterpret_cast<float4 *>(static_cast<float *>(a.out) + qrow * DT + col0 + 32 * c);
#pragma unroll
        for (int q = 0; q < 8; ++q)
          dst[q] = make_float4(__uint_as_float(v[4 * q]) * inv, __uint_as_float(v[4 * q + 1]) * inv,
                               __uint_as_float(v[4 * q + 2]) * inv,
                               __uint_as_float(v[4 * q + 3]) * inv);
      }
    } else {
      float4 *dst = reinterpret_cast<float4 *>(a.ws_o + prow * DT + col0 + 32 * c);
      const uint64_t keep = make_evict_last_policy();
#pragma unroll
      for (int q = 0; q < 8; ++q)
        st_keep(dst + q,
                make_float4(__uint_as_float(v[4 * q]), __uint_as_float(v[4 * q + 1]),
                            __uint_as_float(v[4 * q + 2]), __uint_as_float(v[4 * q + 3])),
                keep);
    }
  }
  if (!real || col0 != 0) return;
  if (a.direct) {
    if (empty) raise_fault(a.status, PSKV_FAULT_EMPTY_ROW);
  } else {
    a.ws_m[prow] = empty ? -CUDART_INF_F : st.m * kLn2;
    a.ws_l[prow] = st.l;
  }
}

// A block whose partition holds no tile: empty partial states, or (one
// partition) zeros flagged as empty rows.
template <bool kPair>
__device__ __forceinline__ void write_empty(const TcArgs &a, const TcPlan &pl, int col0) {
  constexpr int DT = Lay<kPair>::kDT;
  for (int i = threadIdx.x; i < kRows; i += blockDim.x) {
    bool real;
    const size_t qrow = query_row(a, pl, i, &real);
    if (!real) continue;
    if (a.direct) {
      for (int d = col0; d < col0 + kD; ++d) {
        if (a.out_dtype == PSKV_DTYPE_BF16)
          static_cast<__nv_bfloat16 *>(a.out)[qrow * DT + d] = __float2bfloat16_rn(0.f);
        else
          static_cast<float *>(a.out)[qrow * DT + d] = 0.f;
      }
      raise_fault(a.status, PSKV_FAULT_EMPTY_ROW);
    } else if (col0 == 0) {
      const size_t prow = qrow * a.num_splits + pl.p;
      a.ws_m[prow] = -CUDART_INF_F;
      a.ws_l[prow] = 0.f;
    }
  }
}

}  // namespace

template <bool kPair>
__global__ void __launch_bounds__(Lay<kPair>::kThreads, 1)
    pskv_attn_tc_kernel(const TcArgs a, const __grid_constant__ CUtensorMap kmap,
                        const __grid_constant__ CUtensorMap vmap,
                        const __grid_constant__ CUtensorMap qmap) {
  using L = Lay<kPair>;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char *sm = reinterpret_cast<unsigned char *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  uint64_t *bars = reinterpret_cast<uint64_t *>(sm + L::kOffBar);
  StageInfo *info = reinterpret_cast<StageInfo *>(sm + L::kOffInfo);
  uint32_t *slot = reinterpret_cast<uint32_t *>(sm + L::kOffSlot);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + L::kOffAbort);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // a pair's two CTAs are adjacent in x and share one plan; rank c holds columns [256 c, +256)
  const uint32_t rank = kPair ? cluster_rank() : 0u;
  const int col0 = (int)rank * kD;

  // every read of caller memory comes after the previous kernel's writes
  pdl_wait();
  pdl_launch_dependents();
  const TcPlan pl = make_plan(a, kPair ? (int)(blockIdx.x >> 1) : (int)blockIdx.x);
  if (!pl.ok && threadIdx.x == 0 && blockIdx.x == 0 && blockIdx.y == 0)
    raise_fault(a.status, PSKV_FAULT_BAD_LENGTH);
  // (both CTAs of a pair leave here together, before any exchange)
  if (pl.qb * kRows >= (pl.T << a.group_shift)) return;  // no query row in this block
  if (pl.n <= 0) {
    write_empty<kPair>(a, pl, col0);
    return;
  }

  Loader<kPair> ld(a, pl, &kmap, &vmap, sm, bars, info, abort_flag, col0);
  if (warp == 1) {
    // the copy warp sets up the barriers and requests the first tiles at once
    if (lane == 0) {
      for (int k = 0; k < kInfoFree; ++k) mbar_init(&bars[k], 1);  // full / empty K, V
      for (int k = 0; k < kStages; ++k) mbar_init(&bars[kInfoFree + k], 4);  // per softmax warp
      for (int r = 0; r < 2; ++r) {
        mbar_init(&bars[kSFull + r], 1);   // MMA commit
        mbar_init(&bars[kPFull + r], 4);   // per softmax warp
        mbar_init(&bars[kPvDone + r], 1);  // MMA commit
      }
      for (int r = 0; r < 2; ++r) {
        mbar_init(&bars[kXFull + r], 4);   // per exchange warp here (with the peer's bytes)
        mbar_init(&bars[kXFree + r], 4);   // per exchange warp of the peer
        mbar_init(&bars[kSReady + r], 4);  // per exchange warp
      }
      mbar_init(&bars[kDrain], 1);
      mbar_init(&bars[kQReady], 4);
      mbar_init(&bars[kQFull], 1);
      *abort_flag = 0;
      mbar_fence_init();
      {
        // the block's Q rows (tokens t_first .., the KV group's heads; this CTA's
        // columns) by one tensor copy of four 64-column slabs into two V stages
        const int t_first = (pl.qb * kRows) >> a.group_shift;
        mbar_arrive_expect_tx(bars + kQFull, 4 * kQSlab);
        for (int b = 0; b < 4; ++b)
          tc::tma_load_3d(sm + L::kOffV + L::kQStage * kKVBytes + b * kQSlab, &qmap,
                          col0 + 64 * b, pl.g << a.group_shift, pl.r0 + t_first,
                          bars + kQFull);
      }
    }
    __syncwarp();
    ld.prologue(false);
  } else if (warp == 0) {
    tc::alloc(slot, kTmemCols);
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (kPair) cluster_sync();  // the peer's barriers are set up before any exchange
  const uint32_t tmem = *slot;

  if (warp == 0) {
    Issuer<kPair> is{a, pl, sm, bars, abort_flag};
    is.run(tmem);
    is.drain();  // every MMA done before the memory is released
  } else if (warp == 1 || warp == 6) {
    const bool is_v = warp == 6;
    if (!is_v || ld.prologue(true)) ld.run(is_v);
    ld.drain(is_v);  // every copy landed before the CTA leaves
  } else if (warp >= 7) {
    if constexpr (kPair) {
      exchange_loop(a, pl, sm, bars, tmem, abort_flag, rank);
      if (lane == 0) bulk_wait_read();  // no send still reads this CTA's memory
    }
  } else {
    const bool q_ok = stage_q<kPair>(a, pl, sm, bars, tmem, col0, abort_flag);
    tc::fence_before_sync();
    __syncwarp();
    if (lane == 0) mbar_arrive(bars + kQReady);
    RowState st;
    st.m = -CUDART_INF_F;
    st.l = 0.f;
    if (q_ok && softmax_loop<kPair>(a, pl, sm, bars, info, tmem, abort_flag, st, rank)) {
      // PV(n - 1); PV(n - 3) is known done, as S(n - 1) waited for it
      const bool ok =
          tc_wait(bars + kPvDone + ((pl.n - 1) & 1), ((pl.n - 1) >> 1) & 1, abort_flag, a.status);
      if (__all_sync(0xffffffffu, ok)) {
        tc::fence_after_sync();
        write_rows<kPair>(a, pl, tmem, st, col0);
      }
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (kPair) cluster_sync();  // no exchange still targets this CTA's memory
  if (warp == 0) {
    tc::fence_after_sync();
    tc::dealloc(tmem, kTmemCols);
  }
}


namespace {

template <bool kPair>
cudaError_t launch_tc(const TcArgs &a, const void *k_pool, const void *v_pool, dim3 grid,
                      cudaStream_t stream) {
  using L = Lay<kPair>;
  static bool attr_set[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (!(dev >= 0 && dev < 64 && attr_set[dev])) {
    e = cudaFuncSetAttribute(pskv_attn_tc_kernel<kPair>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, L::kSmemBytes);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_set[dev] = true;
  }
  const long long rows = a.num_pages * a.num_kv_heads * a.page_size;
  const int group = 1 << a.group_shift;
  CUtensorMap km, vm, qm;
  if (!make_map(&km, k_pool, rows, L::kDT, a.box_rows) ||
      !make_map(&vm, v_pool, rows, L::kDT, a.box_rows) ||
      !tc::make_q_map(&qm, a.q, a.total_rows, a.num_q_heads, L::kDT, group, kRows / group))
    return cudaErrorInvalidValue;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = kPair ? 2 : 1;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid.x * (kPair ? 2 : 1), grid.y, grid.z);
  cfg.blockDim = dim3(L::kThreads);
  cfg.dynamicSmemBytes = L::kSmemBytes;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = kPair ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, pskv_attn_tc_kernel<kPair>, a, km, vm, qm);
}

}  // namespace

cudaError_t launch_attn_tc(const TcArgs &a, const void *k_pool, const void *v_pool,
                           int head_dim, dim3 grid, cudaStream_t stream) {
  if (head_dim == 2 * kD) return launch_tc<true>(a, k_pool, v_pool, grid, stream);
  if (head_dim == kD) return launch_tc<false>(a, k_pool, v_pool, grid, stream);
  return cudaErrorInvalidValue;
}

}  // namespace pskv
