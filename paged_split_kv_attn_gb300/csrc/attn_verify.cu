// attn_verify.cu -- verify windows (a few query tokens of a row over its long
// paged context) on the fifth-generation tensor cores, with the keys as the
// MMA's M dimension.
//
// Serves decode_attn_multirow (TensorFold #1619, description "Reads" and the
// review thread: drafted verify windows and tree-attention rows read their keys
// through the page table) when a KV head's query columns (tokens x the query
// heads of the KV head) number 17 to 64 and the rows are long.  Such a block is
// too narrow for the query-major kernel's M of 128 (and at head dim 512 that
// kernel needs a CTA pair exchanging partial scores); here the roles turn
// around: the columns, zero-padded to NC = 32 or 64, are the MMA's N.  One CTA
// takes one (row, KV head, partition of 16-key groups); per tile j of 128 keys:
//   S^T = K Q^T        M = 128 keys, N = NC, K = head dim in chunks of 128
//                      (A = the K chunk, B = Q, both K-major in shared memory)
//   softmax            one thread per key reads its NC scores, masks them
//                      (keys outside the CTA's range, causality inside the
//                      window, pages outside the pool) and checks them against
//                      each column's reference max (exp2 units, moved only past
//                      a slack of 8, as in the other kernels); when some
//                      column's max moves, the four softmax warps fold the
//                      tile's column maxima and rescale that column's sums and
//                      O.  P^T goes to shared memory as bf16 hi and lo rows of
//                      one K-major operand; each thread keeps its key row's
//                      share of every column's sum in tensor memory until the end
//   O^T += V^T P^T     per 128 head-dim columns: M = 128, K = 128 keys in 16-key
//                      steps, A = the V chunk read MN-major, B = the hi and lo
//                      rows (one product of N = 2 NC, or hi then lo where
//                      tensor memory holds only one O^T)
// Tensor memory: two S^T regions of NC columns (tile j uses region j % 2), the
// O^T blocks (head dim as lanes, query columns as columns; hi and lo halves),
// then NC columns of per-key-row shares of the column sums.  K and V tiles move
// in chunks of 128 keys x 128 head-dim columns (32 KB), each through a ring of
// its own: the score products take a K chunk as soon as it lands (S of tile
// j + 1 overlaps tile j's softmax), the value products take V chunks once P^T
// of their tile is written (P^T double-buffered where shared memory allows).
// Warp 0 issues the score MMAs, warp 7 the value MMAs, warps 1 and 6 the K and
// V copies (each finds a tile's page ids and pool rows once, at its first
// chunk); warps 2-5 stage Q and run the softmax and the epilogue (warp w owns
// tensor-memory lanes 32 (w % 4) .. + 31), which stages O through the drained
// rings and writes whole rows.  The softmax warps meet on an mbarrier of their
// own (polled: they arrive together); every wait is bounded, and on expiry the
// CTA flags PSKV_FAULT_WAIT_TIMEOUT, lets what it issued finish and frees its
// tensor memory.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <math_constants.h>

#include "attn_tc.h"
#include "pskv_internal.cuh"
#include "tc_common.cuh"
#include "tc_ops.cuh"

namespace pskv {

namespace {

// mbarrier phase test that never suspends the thread.
__device__ __forceinline__ bool mbar_test_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

using tc::elect_one;
using tc::ex2;
using tc::make_map;
using tc::PageCache;
using tc::tc_wait;
using tc::warp_wait;

constexpr int kKeys = 128;             // keys per tile (MMA M of the scores, K of the values)
constexpr int kSlab = kKeys * 128;     // one 64-column slab of a chunk: 128 rows of 128 B
constexpr int kChunkBytes = 2 * kSlab;  // 128 keys x 128 head-dim columns, bf16
constexpr int kInfo = 4;               // tile records in flight
constexpr int kTmemCols = 512;
constexpr float kSlack = 8.f;          // reference-max slack (log2 units)
constexpr int kThreads = 256;
constexpr int kDataBytes = 229376;     // Q, P^T and the rings: 224 KB of the 227

// barrier slots (then the two rings' full and empty barriers)
enum : int {
  kInfoFull = 0,               // [4] a tile's record written (K copy warp)
  kSFull = kInfoFull + kInfo,  // [2] S^T of region r done (MMA commit)
  kSFree = kSFull + 2,         // [2] the softmax warps read region r
  kPFull = kSFree + 2,         // [2] P^T buffer b written (softmax warps)
  kPvDone = kPFull + 2,        // [2] the values of P^T buffer b done (MMA commit)
  kQReady = kPvDone + 2,       // Q in shared memory (softmax warps)
  kSync = kQReady + 1,         // the softmax warps' own meeting point
  kDrainS = kSync + 1,         // every score MMA done (MMA commit)
  kDrainV = kDrainS + 1,       // every value MMA done (MMA commit)
  kFirstRing = kDrainV + 1
};

// Shared memory and tensor memory of head dim DT and NC query columns per CTA
// (offsets from a 1,024-byte aligned base).  A P^T buffer is K-major with 2 NC
// rows: row n holds column n's hi weights, row NC + n its lo weights, 64 keys
// per 128-byte slab, two slabs per tile.  Where tensor memory allows, one value
// product of N = 2 NC takes both halves (O^T keeps a hi and a lo block of NC
// columns each, summed at the end), so V is read once per tile.
template <int DT, int NC>
struct VLay {
  static constexpr int kChunks = DT / 128;    // chunks per K or V tile
  static constexpr int kQSlab = NC * 128;     // 64 head-dim columns of Q (or 64 keys of P^T)
  static constexpr int kQBytes = (DT / 64) * kQSlab;
  static constexpr int kPSlab = 2 * NC * 128;  // 64 keys of the hi and lo rows
  static constexpr int kPBuf = 2 * kPSlab;     // a tile's P^T
  static constexpr int kPBufs = DT == 512 && NC == 64 ? 1 : 2;  // P^T buffers
  static constexpr bool kMerged = !(DT == 512 && NC == 64);     // one value product of 2 NC
  static constexpr int kOBlock = kMerged ? 2 * NC : NC;         // O^T columns per block
  static constexpr int kOffQ = 0;
  static constexpr int kOffP = kOffQ + kQBytes;
  static constexpr int kOffK = kOffP + kPBufs * kPBuf;
  static constexpr int kRingK = 2;  // K stages (the score products take them at once)
  static constexpr int kRingV = (kDataBytes - kOffK) / kChunkBytes - kRingK;  // V stages
  static constexpr int kOffV = kOffK + kRingK * kChunkBytes;
  static constexpr int kFullK = kFirstRing, kEmptyK = kFullK + kRingK;
  static constexpr int kFullV = kEmptyK + kRingK, kEmptyV = kFullV + kRingV;
  static constexpr int kNumBars = kEmptyV + kRingV;
  static constexpr int kOffBar = kOffV + kRingV * kChunkBytes;
  static constexpr int kOffInfo = (kOffBar + kNumBars * 8 + 15) & ~15;  // TileInfo[kInfo]
  static constexpr int kOffVInfo = kOffInfo + kInfo * 16;  // TileInfo[kInfo], V copy warp's
  static constexpr int kOffRed = kOffVInfo + kInfo * 16;   // float[4][NC]: per-warp column values
  static constexpr int kOffM = kOffRed + 4 * NC * 4;       // float[NC]: reference max per column
  static constexpr int kOffA = kOffM + NC * 4;             // float[NC]: rescale factor, then sum
  static constexpr int kOffFlag = kOffA + NC * 4;          // int[2][4] votes, int[4] rescale
  static constexpr int kOffSlot = kOffFlag + 16 * 4;
  static constexpr int kOffCOff = kOffP;  // size_t[NC] output row offsets, once P^T is done
  static constexpr int kOffScale = kOffP + NC * 8;  // float[NC] output scales, likewise
  static constexpr int kOffAbort = kOffSlot + 4;
  static constexpr int kSmemBytes = kOffAbort + 4 + 1024;  // + alignment of the dynamic base
  static_assert(kRingV >= 2 && kOffBar <= kDataBytes, "stages");
  static_assert(kSmemBytes <= 232448, "shared memory");
  static_assert(kOffRed % 16 == 0 && kOffM % 16 == 0 && kOffA % 16 == 0, "16-byte reads");
  // tensor memory: S^T regions, O^T blocks, then the per-row shares of the sums
  static constexpr int kOCol = 2 * NC;
  static constexpr int kLCol = kOCol + kOBlock * kChunks;
  static_assert(kLCol + NC <= kTmemCols, "tensor memory");
  static constexpr uint32_t kIdescS = tc::instr_desc(kKeys, NC, false, false);
  static constexpr uint32_t kIdescPV = tc::instr_desc(128, kOBlock, true, false);
};

// What a copy warp found for a tile: rows [vlo, vhi) lie in the CTA's keys;
// bit c of `bad` marks 16-key groups whose page id lies outside the pool (not
// loaded).  Written before the tile's barrier is arrived on.
struct TileInfo {
  int vlo, vhi;
  uint32_t bad;
  int pad;
};

// The CTA's share of the work, the same in every thread.
struct VPlan {
  int b, g, p;
  int T, r0, len;
  int k_lo, k_hi;  // this partition's keys (16-key groups; the last ends with the row)
  int t_begin, n;  // the 128-key tiles they touch: [t_begin, t_begin + n)
  int ncols;       // real query columns (T x G)
  bool ok;         // the row's length is usable
};

__device__ __forceinline__ VPlan make_plan(const TcArgs &a) {
  VPlan pl;
  pl.p = blockIdx.x;
  pl.g = blockIdx.y;
  pl.b = blockIdx.z;
  pl.T = a.num_tokens;
  pl.r0 = pl.b * a.num_tokens;
  pl.ncols = a.num_tokens << a.group_shift;
  const long long cap = (long long)a.table_stride * a.page_size;
  long long len = a.seq_lens[pl.b];
  pl.ok = !(len < pl.T || len < 1 || len > cap);
  if (!pl.ok) len = len < 0 ? 0 : (len > cap ? cap : len);
  pl.len = (int)len;
  // partitions of whole 16-key groups, as many keys each as the row allows
  const int groups = (pl.len + 15) / 16;
  const int per = (groups + a.num_splits - 1) / a.num_splits;
  pl.k_lo = min(pl.p * per, groups) * 16;
  pl.k_hi = min(min(pl.p * per + per, groups) * 16, pl.len);
  pl.t_begin = pl.k_lo / kKeys;
  pl.n = pl.k_lo < pl.k_hi ? (pl.k_hi + kKeys - 1) / kKeys - pl.t_begin : 0;
  return pl;
}

// A copy warp (all lanes converged; one elected lane issues): warp 1 streams
// the K tiles, warp 6 the V tiles, each through its own ring of stages.  A
// stage is refilled once the MMAs that read its previous chunk are done.  Each
// tile's first chunk also writes the tile's record (the K side's is arrived on
// for the softmax warps; the V side's travels with its chunk's barrier to the
// value-product warp).
template <int DT, int NC>
struct VLoader {
  using L = VLay<DT, NC>;
  const TcArgs &a;
  const VPlan &pl;
  const CUtensorMap *map;
  unsigned char *stages;  // the ring's first stage
  uint64_t *bars;
  int full, empty, ring;  // barrier slots and stage count of the ring
  TileInfo *info;
  volatile int *abort_flag;
  bool is_v;
  int lane, n_slots;
  PageCache pages;
  int seq = 0;  // chunks issued so far

  __device__ VLoader(const TcArgs &a_, const VPlan &pl_, const CUtensorMap *m, bool v,
                     unsigned char *sm, uint64_t *bars_, volatile int *ab)
      : a(a_), pl(pl_), map(m), bars(bars_), abort_flag(ab), is_v(v) {
    stages = sm + (v ? L::kOffV : L::kOffK);
    full = v ? L::kFullV : L::kFullK;
    empty = v ? L::kEmptyV : L::kEmptyK;
    ring = v ? L::kRingV : L::kRingK;
    info = reinterpret_cast<TileInfo *>(sm + (v ? L::kOffVInfo : L::kOffInfo));
    lane = threadIdx.x & 31;
    n_slots = (pl.len + a.page_size - 1) / a.page_size;  // table slots in use
  }

  // The current tile's boxes: pool row of each box of box_rows keys (-1: not
  // loaded: past the partition's keys, or a page id outside the pool) and the
  // bytes one chunk of the tile brings.  Found once per tile, at its first chunk.
  int ys[kKeys / 16];
  uint32_t t_bytes = 0;

  // Tile j's page ids and box rows (every lane), and its record (one lane).
  __device__ void plan_tile(int j) {
    const int key0 = (pl.t_begin + j) * kKeys;
    const int vlo = max(0, pl.k_lo - key0), vhi = min(kKeys, pl.k_hi - key0);
    const int32_t *tbl = a.page_tables + (size_t)pl.b * a.table_stride;
    const int br = a.box_rows;
    uint32_t bad = 0, bytes = 0;
#pragma unroll
    for (int i = 0; i < kKeys / 16; ++i) {
      ys[i] = -1;
      if (i * br >= kKeys || i * br >= vhi || (i + 1) * br <= vlo) continue;
      const int key = key0 + i * br;
      const int page = pages.get(tbl, key / a.page_size, n_slots, lane);
      if (page < 0 || (long long)page >= a.num_pages) {
        bad |= (br == 16 ? 1u : 0xFu) << (i * br / 16);
        continue;
      }
      ys[i] = (page * a.num_kv_heads + pl.g) * a.page_size + key % a.page_size;
      bytes += (uint32_t)(br * 128 * 2);
    }
    t_bytes = bytes;
    if (elect_one()) {
      if (bad) raise_fault(a.status, PSKV_FAULT_BAD_PAGE);
      TileInfo &t = info[j % kInfo];
      t.vlo = vlo;
      t.vhi = vhi;
      t.bad = bad;
      if (!is_v) mbar_arrive(bars + kInfoFull + j % kInfo);
    }
    __syncwarp();
  }

  // Chunk c (head-dim columns [128 c, 128 c + 128)) of tile j: the tile's boxes,
  // each in two 64-column slabs.
  __device__ bool load(int j, int c) {
    const int st = seq % ring;
    if (seq >= ring && !warp_wait(bars + empty + st, ((seq / ring) - 1) & 1, abort_flag, a.status))
      return false;
    if (c == 0) plan_tile(j);
    unsigned char *dst = stages + st * kChunkBytes;
    uint64_t *bar = bars + full + st;
    const int br = a.box_rows;
    if (elect_one()) {
      mbar_arrive_expect_tx(bar, t_bytes);
#pragma unroll
      for (int i = 0; i < kKeys / 16; ++i) {
        if (ys[i] < 0) continue;
#pragma unroll
        for (int sl = 0; sl < 2; ++sl)
          tc::tma_load_2d(dst + sl * kSlab + i * br * 128, map, 128 * c + 64 * sl, ys[i], bar);
      }
    }
    __syncwarp();
    ++seq;
    return true;
  }

  __device__ bool run() {
    for (int j = 0; j < pl.n; ++j)
      for (int c = 0; c < L::kChunks; ++c)
        if (!load(j, c)) return false;
    return true;
  }

  // Wait (bounded) for the last copy issued into each stage.
  __device__ void drain() {
    for (int q = max(0, seq - ring); q < seq; ++q) mbar_wait(bars + full + q % ring, (q / ring) & 1);
  }
};

// The score-product warp (warp 0; all lanes converged, one elected lane
// issues): S(j) into region j % 2 once the softmax warps have read S(j - 2)
// there, chunk by chunk as K lands.
template <int DT, int NC>
struct SIssuer {
  using L = VLay<DT, NC>;
  const TcArgs &a;
  unsigned char *sm;
  uint64_t *bars;
  volatile int *abort_flag;

  __device__ bool wait(int slot, uint32_t parity) {
    return warp_wait(bars + slot, parity, abort_flag, a.status);
  }

  __device__ bool run(int n, uint32_t tmem) {
    if (!wait(kQReady, 0)) return false;
    const uint32_t q0 = smem_u32(sm + L::kOffQ);
    int seq = 0;
    for (int j = 0; j < n; ++j) {
      const int r = j & 1;
      if (j >= 2 && !wait(kSFree + r, ((j - 2) >> 1) & 1)) return false;
      for (int c = 0; c < L::kChunks; ++c) {
        const int st = seq % L::kRingK;
        if (!wait(L::kFullK + st, (seq / L::kRingK) & 1)) return false;
        tc::fence_after_sync();
        const uint32_t k0 = smem_u32(sm + L::kOffK + st * kChunkBytes);
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            // A = K (128 keys x 16 head-dim columns), B = Q (NC columns x the same 16)
            const uint64_t da = tc::smem_desc(k0 + (kk >> 2) * kSlab + (kk & 3) * 32, 16, 1024);
            const uint64_t db =
                tc::smem_desc(q0 + (2 * c + (kk >> 2)) * L::kQSlab + (kk & 3) * 32, 16, 1024);
            tc::mma(tmem + NC * r, da, db, L::kIdescS, c > 0 || kk > 0);
          }
          tc::commit(bars + L::kEmptyK + st);
        }
        __syncwarp();
        ++seq;
      }
      if (elect_one()) tc::commit(bars + kSFull + r);
      __syncwarp();
    }
    return true;
  }
};

// The value-product warp (warp 7): O^T += V^T P^T(j) once P^T(j) is written
// (buffer j % kPBufs), chunk by chunk as V lands.  16-key groups with no key
// of the row (or a page outside the pool) are skipped, and the rows past the
// row's end inside a partial group are zeroed first (they may hold anything,
// and meet P = 0).
template <int DT, int NC>
struct PVIssuer {
  using L = VLay<DT, NC>;
  const TcArgs &a;
  unsigned char *sm;
  uint64_t *bars;
  volatile int *abort_flag;

  __device__ bool wait(int slot, uint32_t parity) {
    return warp_wait(bars + slot, parity, abort_flag, a.status);
  }

  __device__ bool run(int n, uint32_t tmem) {
    const TileInfo *vinfo = reinterpret_cast<const TileInfo *>(sm + L::kOffVInfo);
    const int lane = threadIdx.x & 31;
    bool o_started = false;  // some value product has written O^T
    int seq = 0;
    for (int j = 0; j < n; ++j) {
      const int pb = j % L::kPBufs;
      if (!wait(kPFull + pb, (j / L::kPBufs) & 1)) return false;
      const uint32_t p0 = smem_u32(sm + L::kOffP + pb * L::kPBuf);
      uint32_t live = 0;  // 16-key groups that meet the values
      bool ragged_lo = false, ragged_hi = false;
      int vlo = 0, vhi = 0;
      for (int c = 0; c < L::kChunks; ++c) {
        const int st = seq % L::kRingV;
        if (!wait(L::kFullV + st, (seq / L::kRingV) & 1)) return false;
        if (c == 0) {  // the tile's record, published by this barrier
          const TileInfo inf = vinfo[j % kInfo];
          vlo = inf.vlo;
          vhi = inf.vhi;
#pragma unroll
          for (int k = 0; k < kKeys / 16; ++k)
            if (16 * k < vhi && 16 * k + 16 > vlo && !((inf.bad >> k) & 1u)) live |= 1u << k;
          ragged_lo = (vlo & 15) != 0 && ((live >> (vlo >> 4)) & 1u);
          ragged_hi = (vhi & 15) != 0 && ((live >> (vhi >> 4)) & 1u);
        }
        unsigned char *chunk = sm + L::kOffV + st * kChunkBytes;
        if (ragged_lo || ragged_hi) {
          // rows outside [vlo, vhi) inside a live group: 16 x 16-byte pieces per row
          // (two slabs)
          const int nlo = ragged_lo ? (vlo & 15) * 16 : 0;
          const int nhi = ragged_hi ? (16 - (vhi & 15)) * 16 : 0;
          for (int e = lane; e < nlo + nhi; e += 32) {
            const int f = e < nlo ? e : e - nlo;
            const int row = (e < nlo ? (vlo & ~15) : vhi) + (f >> 4), piece = f & 15;
            *reinterpret_cast<uint4 *>(chunk + (piece >> 3) * kSlab + row * 128 +
                                       (piece & 7) * 16) = make_uint4(0, 0, 0, 0);
          }
          tc::fence_smem_for_async();
          __syncwarp();
        }
        tc::fence_after_sync();
        const uint32_t v0 = smem_u32(chunk);
        if (elect_one()) {
          bool first = !o_started;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            if (!((live >> kk) & 1u)) continue;
            // A = V^T (128 head-dim columns x 16 keys, MN-major), B = P^T (the hi and lo
            // rows x 16 keys, K-major): one product of 2 NC rows, or hi then lo
            const uint64_t da = tc::smem_desc(v0 + kk * 2048, kSlab, 1024);
            const uint32_t pk = p0 + (kk >> 2) * L::kPSlab + (kk & 3) * 32;
            if (L::kMerged) {
              tc::mma(tmem + L::kOCol + L::kOBlock * c, da, tc::smem_desc(pk, 16, 1024),
                      L::kIdescPV, !first);
            } else {
#pragma unroll
              for (int part = 0; part < 2; ++part)
                tc::mma(tmem + L::kOCol + L::kOBlock * c,
                        da, tc::smem_desc(pk + part * NC * 128, 16, 1024), L::kIdescPV,
                        !first || part > 0);
            }
            first = false;
          }
          tc::commit(bars + L::kEmptyV + st);
        }
        __syncwarp();
        ++seq;
      }
      o_started = o_started || live != 0;
      if (elect_one()) tc::commit(bars + kPvDone + pb);
      __syncwarp();
    }
    return true;
  }
};

// Wait (bounded) for every MMA this warp issued.
__device__ __forceinline__ void drain_mma(uint64_t *bar, int32_t *status) {
  if (elect_one()) tc::commit(bar);
  __syncwarp();
  if (!mbar_wait(bar, 0) && (threadIdx.x & 31) == 0) raise_fault(status, PSKV_FAULT_WAIT_TIMEOUT);
}

// The softmax warps' meeting point (one arrival per warp); `ph` counts meetings.
// The four warps arrive within a few hundred cycles of each other, so the wait
// polls (mbarrier.test_wait, bounded) rather than suspending: a suspended
// thread resumed later than a polling one sees the phase complete (3 / 4 / 8
// tokens at 40,002 keys back to back 77.0 / 76.8 / 96.6 us against 78.0 / 77.2
// / 98.3 us).  The polling warp shares its scheduler only with a copy or MMA
// warp.
__device__ __forceinline__ bool meet(uint64_t *bars, int &ph, volatile int *abort_flag,
                                     int32_t *status) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(bars + kSync);
  bool done = *abort_flag == 0 && mbar_test_wait(bars + kSync, ph & 1);
  for (uint32_t i = 0; i < kWaitPolls && !done && *abort_flag == 0; ++i)
    done = mbar_test_wait(bars + kSync, ph & 1);
  if (!done && *abort_flag == 0) {
    *abort_flag = 1;
    raise_fault(status, PSKV_FAULT_WAIT_TIMEOUT);
  }
  ++ph;
  return __all_sync(0xffffffffu, done);
}

// A warp's NC values per lane (NC = 32 or 64) folded (max or sum) over its 32
// lanes by halving exchanges: lane i ends with columns (NC / 32) i ..
// (NC / 32) i + NC / 32 - 1 in out[0 ..].
template <bool kMax, int NC>
__device__ __forceinline__ void fold(const float (&v)[NC], int lane, float (&out)[NC / 32]) {
  float t[NC / 2];
  {
    const bool up = (lane & 16) != 0;
#pragma unroll
    for (int i = 0; i < NC / 2; ++i) {
      const float keep = up ? v[NC / 2 + i] : v[i], send = up ? v[i] : v[NC / 2 + i];
      const float got = __shfl_xor_sync(0xffffffffu, send, 16);
      t[i] = kMax ? fmaxf(keep, got) : keep + got;
    }
  }
#pragma unroll
  for (int half = NC / 4, x = 8; x >= 1; half >>= 1, x >>= 1) {
    const bool up = (lane & x) != 0;
#pragma unroll
    for (int i = 0; i < half; ++i) {
      const float keep = up ? t[half + i] : t[i], send = up ? t[i] : t[half + i];
      const float got = __shfl_xor_sync(0xffffffffu, send, x);
      t[i] = kMax ? fmaxf(keep, got) : keep + got;
    }
  }
#pragma unroll
  for (int i = 0; i < NC / 32; ++i) out[i] = t[i];
}

// Q into shared memory (B of the score products, K-major, 128-byte swizzled):
// column c = query column (token c / G, head c % G of the KV group), zeros
// past the window's columns.  The 128 softmax threads split each column into
// 128 / NC parts.
template <int DT, int NC>
__device__ __forceinline__ void stage_q(const TcArgs &a, const VPlan &pl, unsigned char *sm) {
  using L = VLay<DT, NC>;
  constexpr int kParts = 128 / NC, kDims = DT / kParts;
  const int i = 32 * ((threadIdx.x >> 5) & 3) + (threadIdx.x & 31);
  const int c = i / kParts, part = i % kParts;
  const bool real = c < pl.ncols;
  const int t = c >> a.group_shift;
  const int h = (pl.g << a.group_shift) + (c & ((1 << a.group_shift) - 1));
  const uint4 *src = reinterpret_cast<const uint4 *>(
      static_cast<const uint16_t *>(a.q) +
      ((size_t)(pl.r0 + (real ? t : 0)) * a.num_q_heads + h) * DT + part * kDims);
#pragma unroll 8
  for (int u = 0; u < kDims / 8; ++u) {
    const int d = part * kDims + 8 * u;
    const uint4 v = real ? __ldg(src + u) : make_uint4(0, 0, 0, 0);
    *reinterpret_cast<uint4 *>(sm + L::kOffQ + (d >> 6) * L::kQSlab + c * 128 +
                               ((((d & 63) >> 3) ^ (c & 7)) << 4)) = v;
  }
}

}  // namespace

namespace {

// The softmax warps' loop over the partition's tiles (thread = key row kr of
// the tile).  This thread's share of column c's sum gathers in its lane of
// tensor-memory column kLCol + c.  Returns false on an abort.
// In a drafted tree, `vt` holds, for the one window key this thread's row can
// meet (key row kr of some tile), bit t set iff that key is visible to token t.
template <int DT, int NC>
__device__ __forceinline__ bool softmax_loop(const TcArgs &a, const VPlan &pl, unsigned char *sm,
                                             uint64_t *bars, uint32_t tmem,
                                             volatile int *abort_flag, int &ph,
                                             unsigned long long vt) {
  using L = VLay<DT, NC>;
  const int lane = threadIdx.x & 31, w = (threadIdx.x >> 5) & 3, kr = 32 * w + lane;
  const uint32_t lane_base = tmem + ((uint32_t)(32 * w) << 16);
  const TileInfo *info = reinterpret_cast<const TileInfo *>(sm + L::kOffInfo);
  float *m_sm = reinterpret_cast<float *>(sm + L::kOffM);
  float *a_sm = reinterpret_cast<float *>(sm + L::kOffA);
  float *red = reinterpret_cast<float *>(sm + L::kOffRed);
  volatile int *flags = reinterpret_cast<volatile int *>(sm + L::kOffFlag);
  const float sc = a.scale_log2;
  const int lim0 = pl.len - pl.T + 1;  // token t sees the keys below lim0 + t
  const bool tree = a.tree_mask != nullptr;
  const int win0 = lim0 - 1;  // the window's first key
  // this thread's key in P^T's K-major rows: slab, then the 2-byte slot inside the
  // row's swizzled 16-byte chunk (the chunk index is XORed with the row's low bits)
  const int p_slab = (kr >> 6) * L::kPSlab, p_chunk = (kr & 63) >> 3, p_byte = 2 * (kr & 7);
  auto wait_all = [&](int slot, uint32_t parity) {
    return warp_wait(bars + slot, parity, abort_flag, a.status);
  };
  for (int j = 0; j < pl.n; ++j) {
    const int r = j & 1;
    // the tile's scores, and its record (published by its barrier)
    bool ok = wait_all(kSFull + r, (j >> 1) & 1);
    ok = ok && wait_all(kInfoFull + j % kInfo, (j / kInfo) & 1);
    const TileInfo inf = info[j % kInfo];
    tc::fence_after_sync();
    float x[NC];
#pragma unroll
    for (int h = 0; h < NC / 32; ++h) {
      uint32_t v[32];
      tc::ld32(lane_base + NC * r + 32 * h, v);
      tc::wait_ld();
      tc::reg_fence(v);
#pragma unroll
      for (int c = 0; c < 32; ++c) x[32 * h + c] = __uint_as_float(v[c]) * sc;
    }
    tc::fence_before_sync();
    __syncwarp();
    if (lane == 0) mbar_arrive(bars + kSFree + r);  // the region may take S(j + 2)

    // ---- mask (by selection: rows never loaded may hold anything)
    const int key = (pl.t_begin + j) * kKeys + kr;
    const bool key_ok = kr >= inf.vlo && kr < inf.vhi && !((inf.bad >> (kr >> 4)) & 1u);
    if (tree) {
      // a window key (win0 <= key < win0 + T) is this thread's one window key
      if (!(key_ok && key < win0)) {
#pragma unroll
        for (int c = 0; c < NC; ++c) {
          const int t = c >> a.group_shift;
          const bool vis = key_ok && key < lim0 + t && (key < win0 || ((vt >> t) & 1ull));
          x[c] = vis ? x[c] : -CUDART_INF_F;
        }
      }
    } else if (!(key_ok && key < lim0)) {
#pragma unroll
      for (int c = 0; c < NC; ++c) {
        const bool vis = key_ok && key < lim0 + (c >> a.group_shift);
        x[c] = vis ? x[c] : -CUDART_INF_F;
      }
    }
    // ---- does some column's reference max have to move?  (The first tile sets
    // every column's reference: no vote.)
    bool moved = true;
    if (j > 0) {
      bool rise = false;
#pragma unroll
      for (int c = 0; c < NC; c += 4) {
        const float4 m4 = *reinterpret_cast<const float4 *>(m_sm + c);
        rise |= x[c] > m4.x + kSlack || x[c + 1] > m4.y + kSlack || x[c + 2] > m4.z + kSlack ||
                x[c + 3] > m4.w + kSlack;
      }
      const int vote = __any_sync(0xffffffffu, rise);
      if (lane == 0) flags[4 * r + w] = vote;
      ok = meet(bars, ph, abort_flag, a.status) && ok;
      moved = ok && (flags[4 * r] | flags[4 * r + 1] | flags[4 * r + 2] | flags[4 * r + 3]);
    }
    if (!ok || *abort_flag) return false;
    if (moved) {
      // the tile's column maxima: per warp, then over the four warps
      float mx[NC / 32];
      fold<true, NC>(x, lane, mx);
#pragma unroll
      for (int i = 0; i < NC / 32; ++i) red[NC * w + (NC / 32) * lane + i] = mx[i];
      if (!meet(bars, ph, abort_flag, a.status)) return false;
      if (kr < NC) {  // thread kr owns column kr (whole warps)
        const float t = fmaxf(fmaxf(red[kr], red[NC + kr]), fmaxf(red[2 * NC + kr], red[3 * NC + kr]));
        const float mo = m_sm[kr];
        float al = 1.f;
        bool resc = false;
        if (t > mo + kSlack) {
          resc = mo != -CUDART_INF_F;  // with m = -inf the column's O and sums are still 0
          al = resc ? ex2(mo - t) : 0.f;
          m_sm[kr] = t;
        }
        a_sm[kr] = al;
        const int v = __any_sync(0xffffffffu, resc);
        if (lane == 0) flags[8 + w] = v;
      }
      if (!meet(bars, ph, abort_flag, a.status)) return false;
      bool resc_any = false;
#pragma unroll
      for (int i = 0; i < NC / 32; ++i) resc_any = resc_any || flags[8 + i];
      // this thread's shares of the sums (still 0 at the first tile), then (a
      // reference moved) the O^T columns once the values of tile j - 1 are in
      if (j > 0 && !resc_any) {
#pragma unroll 1
        for (int h = 0; h < NC / 32; ++h) {
          uint32_t v[32];
          const uint32_t addr = lane_base + L::kLCol + 32 * h;
          tc::ld32(addr, v);
          tc::wait_ld();
          tc::reg_fence(v);
#pragma unroll
          for (int c = 0; c < 32; ++c)
            v[c] = __float_as_uint(__uint_as_float(v[c]) * a_sm[32 * h + c]);
          tc::st32(addr, v);
        }
      } else if (j > 0) {
        if (!wait_all(kPvDone + (j - 1) % L::kPBufs, ((j - 1) / L::kPBufs) & 1)) return false;
        tc::fence_after_sync();
        // the O^T blocks (hi and lo halves), then the sums: column q of them belongs to
        // query column q % NC
#pragma unroll 1
        for (int g = 0; g < (L::kOBlock * L::kChunks + NC) / 32; ++g) {
          uint32_t v[32];
          const uint32_t addr = lane_base + L::kOCol + 32 * g;
          const float *al = a_sm + (32 * g) % NC;
          tc::ld32(addr, v);
          tc::wait_ld();
          tc::reg_fence(v);
#pragma unroll
          for (int c = 0; c < 32; ++c) v[c] = __float_as_uint(__uint_as_float(v[c]) * al[c]);
          tc::st32(addr, v);
        }
      }
      tc::wait_st();
    }

    // ---- P = exp2(x - m) as hi + lo bf16 (K-major rows of P^T), written as they
    // are made: buffer j % kPBufs is free once the values of tile j - kPBufs are done
    const int pb = j % L::kPBufs;
    if (j >= L::kPBufs &&
        !wait_all(kPvDone + pb, ((j - L::kPBufs) / L::kPBufs) & 1))
      return false;
    unsigned char *ph_hi = sm + L::kOffP + pb * L::kPBuf + p_slab + p_byte;
#pragma unroll
    for (int h = 0; h < NC / 32; ++h) {
      uint32_t lv[32];
      const uint32_t laddr = lane_base + L::kLCol + 32 * h;
      tc::ld32(laddr, lv);
      // the reference maxima in registers first (read between the P stores below,
      // each would wait for the store before it)
      float mr[32];
#pragma unroll
      for (int c = 0; c < 32; c += 4) {
        const float4 m4 = *reinterpret_cast<const float4 *>(m_sm + 32 * h + c);
        mr[c] = m4.x;
        mr[c + 1] = m4.y;
        mr[c + 2] = m4.z;
        mr[c + 3] = m4.w;
      }
      tc::wait_ld();
      tc::reg_fence(lv);
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        const int n = 32 * h + c;
        const float mc = mr[c];
        const float p = ex2(x[n] - (mc == -CUDART_INF_F ? 0.f : mc));
        lv[c] = __float_as_uint(__uint_as_float(lv[c]) + p);
        const __nv_bfloat16 hi = __float2bfloat16_rn(p);
        const __nv_bfloat16 lo = __float2bfloat16_rn(p - __bfloat162float(hi));
        unsigned char *at = ph_hi + n * 128 + ((p_chunk ^ (n & 7)) << 4);
        *reinterpret_cast<__nv_bfloat16 *>(at) = hi;
        *reinterpret_cast<__nv_bfloat16 *>(at + NC * 128) = lo;  // row NC + n
      }
      tc::st32(laddr, lv);
    }
    tc::wait_st();
    tc::fence_smem_for_async();
    tc::fence_before_sync();
    __syncwarp();
    if (lane == 0) mbar_arrive(bars + kPFull + pb);
  }
  return true;
}

// The (m, l) of the CTA's columns (partial), or the empty-row flag (direct).
template <int DT, int NC>
__device__ __forceinline__ void write_ml(const TcArgs &a, const VPlan &pl, const unsigned char *sm,
                                         bool have_o) {
  using L = VLay<DT, NC>;
  const int kr = 32 * ((threadIdx.x >> 5) & 3) + (threadIdx.x & 31);
  if (kr >= pl.ncols) return;
  const float *m_sm = reinterpret_cast<const float *>(sm + L::kOffM);
  const float *l_sm = reinterpret_cast<const float *>(sm + L::kOffA);  // column sums
  const size_t qrow = (size_t)(pl.r0 + (kr >> a.group_shift)) * a.num_q_heads +
                      (pl.g << a.group_shift) + (kr & ((1 << a.group_shift) - 1));
  const bool empty = !have_o || m_sm[kr] == -CUDART_INF_F;
  if (a.direct) {
    if (empty) raise_fault(a.status, PSKV_FAULT_EMPTY_ROW);
  } else {
    const size_t prow = qrow * a.num_splits + pl.p;
    const uint64_t keep = make_evict_last_policy();
    st_keep(a.ws_m + prow, empty ? -CUDART_INF_F : m_sm[kr] * kLn2, keep);
    st_keep(a.ws_l + prow, empty ? 0.f : l_sm[kr], keep);
  }
}

// Output row of query column c (direct: [rows][Hq][DT]) or partial row
// ([rows][Hq][P][DT]), in elements.
__device__ __forceinline__ size_t col_offset(const TcArgs &a, const VPlan &pl, int c, int dt) {
  const size_t qrow = (size_t)(pl.r0 + (c >> a.group_shift)) * a.num_q_heads +
                      (pl.g << a.group_shift) + (c & ((1 << a.group_shift) - 1));
  return (a.direct ? qrow : qrow * a.num_splits + pl.p) * dt;
}

// A partition with no tile: the empty state (partial), or zeros flagged as
// empty rows (direct).
template <int DT, int NC>
__device__ __forceinline__ void write_empty(const TcArgs &a, const VPlan &pl,
                                            const unsigned char *sm) {
  const int kr = 32 * ((threadIdx.x >> 5) & 3) + (threadIdx.x & 31);
  if (a.direct) {
    for (int e = kr; e < pl.ncols * (DT / 4); e += 128) {
      const int c = e / (DT / 4), q = e % (DT / 4);
      const size_t off = col_offset(a, pl, c, DT) + 4 * q;
      if (a.out_dtype == PSKV_DTYPE_BF16)
        *reinterpret_cast<uint2 *>(static_cast<__nv_bfloat16 *>(a.out) + off) = make_uint2(0, 0);
      else
        *reinterpret_cast<float4 *>(static_cast<float *>(a.out) + off) =
            make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
  write_ml<DT, NC>(a, pl, sm, false);
}

// Write the CTA's columns: O / sum to `out` (direct) or the partial (m, l, o).
// Thread kr holds head-dim row kr of every O^T block: it first puts its rows,
// scaled per column (1 / sum direct, 1 partial, 0 for a column that met no
// key), into a [column][head dim] f32 block of the (drained) K/V rings; after
// the softmax warps meet, every thread writes 16-byte pieces of whole rows.
template <int DT, int NC>
__device__ __forceinline__ bool write_cols(const TcArgs &a, const VPlan &pl, unsigned char *sm,
                                           uint64_t *bars, uint32_t tmem, int &ph,
                                           volatile int *abort_flag) {
  using L = VLay<DT, NC>;
  static_assert(NC * DT * 4 <= L::kRingK * kChunkBytes + L::kRingV * kChunkBytes, "staging");
  const int lane = threadIdx.x & 31, w = (threadIdx.x >> 5) & 3, kr = 32 * w + lane;
  const uint32_t lane_base = tmem + ((uint32_t)(32 * w) << 16);
  const float *scale = reinterpret_cast<const float *>(sm + L::kOffScale);
  float *stage = reinterpret_cast<float *>(sm + L::kOffK);
#pragma unroll 1
  for (int blk = 0; blk < L::kChunks; ++blk) {
#pragma unroll 1
    for (int h = 0; h < NC / 32; ++h) {
      // both loads in flight before the one wait
      uint32_t v[32], u[32];
      const uint32_t addr = lane_base + L::kOCol + L::kOBlock * blk + 32 * h;
      tc::ld32(addr, v);
      if (L::kMerged) tc::ld32(addr + NC, u);  // O = the hi products + the lo products
      tc::wait_ld();
      tc::reg_fence(v);
      if (L::kMerged) {
        tc::reg_fence(u);
#pragma unroll
        for (int c = 0; c < 32; ++c)
          v[c] = __float_as_uint(__uint_as_float(v[c]) + __uint_as_float(u[c]));
      }
      const int dim = 128 * blk + kr;
      // the scales in registers first: read between the stores below, each would
      // wait for the store before it (the compiler cannot tell them apart)
      float sc[32];
#pragma unroll
      for (int c = 0; c < 32; c += 4) {
        const float4 s4 = *reinterpret_cast<const float4 *>(scale + 32 * h + c);
        sc[c] = s4.x;
        sc[c + 1] = s4.y;
        sc[c + 2] = s4.z;
        sc[c + 3] = s4.w;
      }
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        // (a column that met no key may hold no value product at all: scale 0 by selection)
        stage[(32 * h + c) * DT + dim] = sc[c] == 0.f ? 0.f : __uint_as_float(v[c]) * sc[c];
      }
    }
  }
  if (!meet(bars, ph, abort_flag, a.status)) return false;
  const size_t *coff = reinterpret_cast<const size_t *>(sm + L::kOffCOff);
  const uint64_t keep = make_evict_last_policy();
#pragma unroll 4
  for (int e = kr; e < pl.ncols * (DT / 4); e += 128) {
    const int c = e / (DT / 4), q = e % (DT / 4);
    const float4 y = *reinterpret_cast<const float4 *>(stage + c * DT + 4 * q);
    const size_t off = coff[c] + 4 * q;
    if (!a.direct)
      st_keep(reinterpret_cast<float4 *>(a.ws_o + off), y, keep);
    else if (a.out_dtype == PSKV_DTYPE_BF16)
      *reinterpret_cast<uint2 *>(static_cast<__nv_bfloat16 *>(a.out) + off) =
          make_uint2(pack_bf16x2(y.x, y.y), pack_bf16x2(y.z, y.w));
    else
      *reinterpret_cast<float4 *>(static_cast<float *>(a.out) + off) = y;
  }
  write_ml<DT, NC>(a, pl, sm, true);
  return true;
}

}  // namespace

template <int DT, int NC>
__global__ void __launch_bounds__(kThreads, 1)
    pskv_verify_tc_kernel(const TcArgs a, const __grid_constant__ CUtensorMap kmap,
                          const __grid_constant__ CUtensorMap vmap) {
  using L = VLay<DT, NC>;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char *sm = reinterpret_cast<unsigned char *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  uint64_t *bars = reinterpret_cast<uint64_t *>(sm + L::kOffBar);
  uint32_t *slot = reinterpret_cast<uint32_t *>(sm + L::kOffSlot);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + L::kOffAbort);
  float *m_sm = reinterpret_cast<float *>(sm + L::kOffM);
  float *a_sm = reinterpret_cast<float *>(sm + L::kOffA);
  float *red = reinterpret_cast<float *>(sm + L::kOffRed);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // every read of caller memory comes after the previous kernel's writes
  pdl_wait();
  pdl_launch_dependents();
  const VPlan pl = make_plan(a);
  if (!pl.ok && threadIdx.x == 64) raise_fault(a.status, PSKV_FAULT_BAD_LENGTH);
  if (pl.n <= 0) {  // a partition past the row's keys: the empty state
    if (warp >= 2 && warp < 6) write_empty<DT, NC>(a, pl, sm);
    return;
  }

  if (warp == 1) {
    if (lane == 0) {
      for (int k = 0; k < kInfo; ++k) mbar_init(&bars[kInfoFull + k], 1);
      for (int r = 0; r < 2; ++r) {
        mbar_init(&bars[kSFull + r], 1);   // MMA commit
        mbar_init(&bars[kSFree + r], 4);   // per softmax warp
        mbar_init(&bars[kPFull + r], 4);   // per softmax warp
        mbar_init(&bars[kPvDone + r], 1);  // MMA commit
      }
      mbar_init(&bars[kQReady], 4);
      mbar_init(&bars[kSync], 4);
      mbar_init(&bars[kDrainS], 1);
      mbar_init(&bars[kDrainV], 1);
      for (int k = L::kFullK; k < L::kNumBars; ++k) mbar_init(&bars[k], 1);
      *abort_flag = 0;
      mbar_fence_init();
    }
    __syncwarp();
  } else if (warp == 0) {
    tc::alloc(slot, kTmemCols);
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *slot;

  if (warp == 0) {
    SIssuer<DT, NC> is{a, sm, bars, abort_flag};
    is.run(pl.n, tmem);
    drain_mma(bars + kDrainS, a.status);  // every MMA done before the memory is released
  } else if (warp == 7) {
    PVIssuer<DT, NC> is{a, sm, bars, abort_flag};
    is.run(pl.n, tmem);
    drain_mma(bars + kDrainV, a.status);
  } else if (warp == 1 || warp == 6) {
    VLoader<DT, NC> ld(a, pl, warp == 6 ? &vmap : &kmap, warp == 6, sm, bars, abort_flag);
    ld.run();
    ld.drain();  // every copy landed before the CTA leaves
  } else {
    const int kr = 32 * (warp & 3) + lane;
    const uint32_t lane_base = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
    stage_q<DT, NC>(a, pl, sm);
    if (kr < NC) m_sm[kr] = -CUDART_INF_F;
    // A drafted tree: the window keys are win0 .. win0 + T - 1 (T <= 64 < 128
    // keys a tile), so the only one this thread's key row kr can meet is window
    // key d = (kr - win0) mod 128 when d < T; bit t of vt: token t sees it
    // (its mask holds bit d, and d <= t).  A mask with a later bit, or
    // without its own, is flagged; the later bits are ignored.
    unsigned long long vt = 0;
    if (a.tree_mask != nullptr) {
      const int win0 = pl.len - pl.T;
      const int d = ((kr - win0) % kKeys + kKeys) % kKeys;
      const unsigned long long *tm = a.tree_mask + pl.r0;
      if (kr < pl.T) {
        const unsigned long long mk = tm[kr];
        const unsigned long long upto = kr >= 63 ? ~0ull : (2ull << kr) - 1;
        if (!((mk >> kr) & 1ull) || (mk & ~upto)) raise_fault(a.status, PSKV_FAULT_BAD_MASK);
      }
      if (d < pl.T)
        for (int t = d; t < pl.T; ++t) vt |= ((tm[t] >> d) & 1ull) << t;
    }
    tc::fence_smem_for_async();
    __syncwarp();
    if (lane == 0) mbar_arrive(bars + kQReady);
    {  // this thread's shares of the sums start at 0
      uint32_t z[32];
#pragma unroll
      for (int c = 0; c < 32; ++c) z[c] = 0u;
#pragma unroll
      for (int h = 0; h < NC / 32; ++h) tc::st32(lane_base + L::kLCol + 32 * h, z);
      tc::wait_st();
    }
    int ph = 0;
    bool ok = meet(bars, ph, abort_flag, a.status);  // the reference maxima are set
    ok = ok && softmax_loop<DT, NC>(a, pl, sm, bars, tmem, abort_flag, ph, vt);
    // the last values product (and with it every earlier one), then every column's
    // sum over the tile rows
    ok = ok && warp_wait(bars + kPvDone + (pl.n - 1) % L::kPBufs,
                         ((pl.n - 1) / L::kPBufs) & 1, abort_flag, a.status);
    if (ok) {
      tc::fence_after_sync();
      float l[NC];
#pragma unroll
      for (int h = 0; h < NC / 32; ++h) {
        uint32_t v[32];
        tc::ld32(lane_base + L::kLCol + 32 * h, v);
        tc::wait_ld();
        tc::reg_fence(v);
#pragma unroll
        for (int c = 0; c < 32; ++c) l[32 * h + c] = __uint_as_float(v[c]);
      }
      float sum[NC / 32];
      fold<false, NC>(l, lane, sum);
#pragma unroll
      for (int i = 0; i < NC / 32; ++i) red[NC * (warp & 3) + (NC / 32) * lane + i] = sum[i];
      ok = meet(bars, ph, abort_flag, a.status);
    }
    // column sums, output scales and output rows (thread kr, column kr; written
    // apart from the folds they are made from)
    if (ok && kr < NC) {
      const float t = (red[kr] + red[NC + kr]) + (red[2 * NC + kr] + red[3 * NC + kr]);
      a_sm[kr] = t;
      const bool seen = m_sm[kr] != -CUDART_INF_F;
      reinterpret_cast<float *>(sm + L::kOffScale)[kr] =
          !seen ? 0.f : (a.direct ? (t > 0.f ? 1.f / t : 0.f) : 1.f);
      reinterpret_cast<size_t *>(sm + L::kOffCOff)[kr] = col_offset(a, pl, kr, DT);
    }
    ok = ok && meet(bars, ph, abort_flag, a.status);
    if (ok) write_cols<DT, NC>(a, pl, sm, bars, tmem, ph, abort_flag);
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    tc::fence_after_sync();
    tc::dealloc(tmem, kTmemCols);
  }
}

namespace {

template <int DT, int NC>
cudaError_t launch_v(const TcArgs &a, const void *k_pool, const void *v_pool, dim3 grid,
                     cudaStream_t stream) {
  using L = VLay<DT, NC>;
  static bool attr_set[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (!(dev >= 0 && dev < 64 && attr_set[dev])) {
    e = cudaFuncSetAttribute(pskv_verify_tc_kernel<DT, NC>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, L::kSmemBytes);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_set[dev] = true;
  }
  const long long rows = a.num_pages * a.num_kv_heads * a.page_size;
  CUtensorMap km, vm;
  if (!make_map(&km, k_pool, rows, DT, a.box_rows) || !make_map(&vm, v_pool, rows, DT, a.box_rows))
    return cudaErrorInvalidValue;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = L::kSmemBytes;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, pskv_verify_tc_kernel<DT, NC>, a, km, vm);
}

}  // namespace

cudaError_t launch_attn_verify(const TcArgs &a, const void *k_pool, const void *v_pool,
                               int head_dim, dim3 grid, cudaStream_t stream) {
  const bool narrow = (a.num_tokens << a.group_shift) <= 32;
  if (head_dim == 512)
    return narrow ? launch_v<512, 32>(a, k_pool, v_pool, grid, stream)
                  : launch_v<512, 64>(a, k_pool, v_pool, grid, stream);
  if (head_dim == 256)
    return narrow ? launch_v<256, 32>(a, k_pool, v_pool, grid, stream)
                  : launch_v<256, 64>(a, k_pool, v_pool, grid, stream);
  return cudaErrorInvalidValue;
}

}  // namespace pskv
