// Prompt profiling on the tcgen05 tensor cores (bf16 Q/K, fp32 accumulate).
//
// FastGen profiles every head on A = softmax(s Q K^T) under the causal mask
// (Model Tells You What to Discard, Method, eq. (C*)); the policies need, per
// key j, colsum_j = sum_i A_ij and the band sum bandcol_j = sum_{j<=i<j+w} A_ij.
// A is never written to memory.  Two passes over 128 x 128 score tiles, each
// a persistent kernel (two CTAs per SM) whose work units are claimed in
// head-major order from a counter (the tiles of one head run together and
// share its operands through L2; within a head the longest units go first;
// with a head list, only the listed heads are profiled):
//   pass 1, query-major: unit (g, query tile) streams its causal key tiles,
//     S = Q_tile K_tile^T lands in tensor memory, the consumer warps keep the
//     running row max and sum and write the negated base-2 row log-sum-exp;
//   pass 2, key-major: unit (g, key tile) streams query tiles i >= j,
//     S^T = K_tile Q_tile^T, and each consumer thread owns one key (one TMEM
//     lane), so its column and band sums accumulate in registers.
// Warp roles: warps 0-7 consume TMEM (two per lane quarter, 64 columns each),
// warp 8 claims units and issues the TMA loads (128-byte swizzled tiles),
// warp 9 issues the MMAs (one thread) into two 128-column accumulators.  All
// pipeline state (stages, phases) carries over from unit to unit; tensor
// memory is allocated once per CTA.
// Every wait is bounded (about 1 s); a timeout sets an abort flag that ends
// every other wait of the CTA at once, records bit 1 in the error word, and
// the CTA lets its copies and MMAs land, frees tensor memory and exits.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "fg_common.cuh"
#include "fg_internal.h"
#include "fg_sm100.cuh"

namespace fg {
namespace {

using namespace sm100;

constexpr int kBlk = 128;       // tile rows and columns
constexpr int kConsumerWarps = 8;  // two per TMEM lane quarter, each taking 64 columns
constexpr int kTmaWarp = kConsumerWarps, kMmaWarp = kConsumerWarps + 1;
constexpr int kThreads = (kConsumerWarps + 2) * 32;
constexpr int kHalfCols = kBlk / 2;
constexpr int kStages = 2;      // streamed operand tiles in flight
constexpr uint32_t kTmemCols = 256;  // two 128-column fp32 accumulators
constexpr int kLseSlots = 4;    // pass 2: query-tile LSE vectors in flight

template <int D>
struct TileCfg {
  static constexpr int kHalves = D / 64;                       // 128-byte swizzle atoms per row
  static constexpr uint32_t kHalfBytes = kBlk * 64 * 2;        // 16 KB
  static constexpr uint32_t kTileBytes = kHalves * kHalfBytes;
  static constexpr int kKSteps = D / 16;                       // MMAs of K = 16 per tile
};

struct UnitMeta {
  int g, at, b_first, nb;  // head, own tile, first streamed tile, streamed tiles
  int valid;               // 0 ends the stream
};

template <int D>
struct alignas(1024) TcSmem {
  uint8_t a[TileCfg<D>::kTileBytes];             // per unit: Q (pass 1) or K (pass 2)
  uint8_t b[kStages][TileCfg<D>::kTileBytes];    // streamed: K (pass 1) or Q (pass 2)
  float nlse[kLseSlots][kBlk];                   // pass 2: negated row LSEs of a query tile
  float part[2][2][kBlk];                        // per unit parity: second-half partials
  UnitMeta unit[2];
  int abort;
  uint64_t a_full, a_empty;
  uint64_t full[kStages], empty[kStages];
  uint64_t sfull[2], sempty[2];
  uint64_t lfull[kLseSlots], lempty[kLseSlots];
  uint64_t unit_full[2], unit_empty[2];
  uint64_t part_ready[2], part_done[2];
  uint32_t tmem_base;
};

// Bounded wait that returns at once once any thread of the CTA has aborted.
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, volatile int* abort) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (!*abort) {
#pragma unroll 1
    for (int i = 0; i < 64; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (global_timer_ns() - t0 > kWaitLimitNs) {
      *abort = 1;
      return false;
    }
  }
  return false;
}

template <int D>
__device__ __forceinline__ void load_tile(uint8_t* dst, const CUtensorMap* map, uint64_t* bar,
                                          int row, int g) {
#pragma unroll
  for (int h = 0; h < TileCfg<D>::kHalves; ++h)
    tma_load_3d(dst + h * TileCfg<D>::kHalfBytes, map, bar, h * 64, row, g);
}

template <int D>
__device__ __forceinline__ void issue_tile_mma(uint32_t d_tmem, uint32_t a_base, uint32_t b_base) {
  constexpr uint32_t idesc = idesc_bf16_f32(kBlk, kBlk);
#pragma unroll
  for (int kk = 0; kk < TileCfg<D>::kKSteps; ++kk) {
    const uint32_t off = (kk >> 2) * TileCfg<D>::kHalfBytes + (kk & 3) * 32;
    umma_bf16(d_tmem, desc_kmajor_sw128(a_base + off), desc_kmajor_sw128(b_base + off), idesc,
              kk > 0 ? 1u : 0u);
  }
}

__device__ __forceinline__ float f(uint32_t u) { return __uint_as_float(u); }

// Pass 1, one thread's 64 scores of a tile row: running max m and sum l in
// base 2.  Columns c >= cut (tile-relative, 0..127) are masked (causal
// diagonal and the prompt end); cut < 0 means no masking.  c0 = first column.
__device__ __forceinline__ void lse_tile(uint32_t (&r)[2][32], float sl2, int c0, int cut,
                                         float& m, float& l) {
  if (cut >= 0) {
#pragma unroll
    for (int c = 0; c < 2; ++c)
#pragma unroll
      for (int e = 0; e < 32; ++e)
        if (c0 + c * 32 + e >= cut) r[c][e] = __float_as_uint(FG_NEG_INF);
  }
  float mx[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int c = k >> 1, e0 = (k & 1) * 16;
    mx[k] = FG_NEG_INF;
#pragma unroll
    for (int e = e0; e < e0 + 16; e += 2) mx[k] = max3(mx[k], f(r[c][e]), f(r[c][e + 1]));
  }
  const float mnew = fmaxf(m, fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * sl2);
  if (mnew == FG_NEG_INF) return;
  const uint64_t s2 = pack2(sl2, sl2), nm = pack2(-mnew, -mnew);
  uint64_t acc[4] = {0, 0, 0, 0};
#pragma unroll
  for (int c = 0; c < 2; ++c)
#pragma unroll
    for (int e = 0; e < 32; e += 2) {
      float x0, x1;
      unpack2(fma2(pack2(f(r[c][e]), f(r[c][e + 1])), s2, nm), x0, x1);
      acc[(e >> 1) & 3] = add2(acc[(e >> 1) & 3], pack2(ex2(x0), ex2(x1)));
    }
  float sum = 0.f;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    float a0, a1;
    unpack2(acc[k], a0, a1);
    sum += a0 + a1;
  }
  l = l * ex2(m - mnew) + sum;
  m = mnew;
}

// Pass 2, one thread's NC x 32 columns (starting at tile column c0) of a key row:
// adds sum A to cs and the part inside the band to bs.  Called by all lanes of
// a warp together.  Lv = the negated base-2 LSEs of those NC x 32 queries
// (-inf past the prompt end), four per vector, loaded before the scores so
// that the shared-memory reads overlap the tensor-memory load.  Tile columns
// c < lo precede the key (masked); columns c < band lie in the window.
template <int NC>
__device__ __forceinline__ void col_tile(const uint32_t (&r)[NC][32], const float4 (&Lv)[8 * NC],
                                         float sl2, int c0, int lo, int band, float& cs,
                                         float& bs) {
  constexpr int kCols = NC * 32;
  // every column precedes every lane's key (leading chunks of the diagonal tile)
  if (__all_sync(0xffffffffu, lo >= c0 + kCols)) return;
  const uint64_t s2 = pack2(sl2, sl2);
  // no lane of the warp needs a per-element test: one packed path
  if (__all_sync(0xffffffffu, lo <= c0 && (band <= c0 || band >= c0 + kCols))) {
    uint64_t acc[4] = {0, 0, 0, 0};
#pragma unroll
    for (int c = 0; c < NC; ++c)
#pragma unroll
      for (int e = 0; e < 32; e += 4) {
        const float4 L = Lv[c * 8 + e / 4];
        float x0, x1, x2, x3;
        unpack2(fma2(pack2(f(r[c][e]), f(r[c][e + 1])), s2, pack2(L.x, L.y)), x0, x1);
        unpack2(fma2(pack2(f(r[c][e + 2]), f(r[c][e + 3])), s2, pack2(L.z, L.w)), x2, x3);
        acc[(e >> 2) & 3] = add2(acc[(e >> 2) & 3],
                                 add2(pack2(ex2(x0), ex2(x1)), pack2(ex2(x2), ex2(x3))));
      }
    float t = 0.f;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      float a0, a1;
      unpack2(acc[k], a0, a1);
      t += a0 + a1;
    }
    cs += t;
    if (band >= c0 + kCols) bs += t;
    return;
  }
  // Some lane of the warp needs per-element tests (its causal diagonal or
  // band edge falls in these columns).  The decision is made for the whole
  // warp, so its lanes never split between two paths: every lane runs the
  // packed arithmetic, the causal test only when some lane needs it, and the
  // band split by 0/1 weights, each the saturated difference of two exact
  // small integers (the lane's band end and the column offset).
  const bool diag = __any_sync(0xffffffffu, lo > c0);
  const float dband = (float)(band - c0);
  uint64_t at = 0, ab = 0;
#pragma unroll
  for (int c = 0; c < NC; ++c)
#pragma unroll
    for (int e = 0; e < 32; e += 4) {
      const float k = (float)(c * 32 + e);
      const float4 L = Lv[c * 8 + e / 4];
      float x0, x1, x2, x3;
      unpack2(fma2(pack2(f(r[c][e]), f(r[c][e + 1])), s2, pack2(L.x, L.y)), x0, x1);
      unpack2(fma2(pack2(f(r[c][e + 2]), f(r[c][e + 3])), s2, pack2(L.z, L.w)), x2, x3);
      uint64_t p01 = pack2(ex2(x0), ex2(x1)), p23 = pack2(ex2(x2), ex2(x3));
      if (diag) {  // a select, not a product: a score past the key may overflow
        const int col = c0 + c * 32 + e;
        float p0, p1, p2, p3;
        unpack2(p01, p0, p1);
        unpack2(p23, p2, p3);
        p01 = pack2(col < lo ? 0.f : p0, col + 1 < lo ? 0.f : p1);
        p23 = pack2(col + 2 < lo ? 0.f : p2, col + 3 < lo ? 0.f : p3);
      }
      at = add2(at, add2(p01, p23));
      ab = fma2(p01, pack2(__saturatef(dband - k), __saturatef(dband - k - 1.f)), ab);
      ab = fma2(p23, pack2(__saturatef(dband - k - 2.f), __saturatef(dband - k - 3.f)), ab);
    }
  float t0, t1, b0, b1;
  unpack2(at, t0, t1);
  unpack2(ab, b0, b1);
  cs += t0 + t1;
  bs += b0 + b1;
}

// PASS 1: nlse2[g, i] = -log2 sum_j 2^(s' q_i.k_j) (row stride ld); rows past
//         the prompt get -inf.
// PASS 2: colsum / bandcol.
// sched: this pass's unit counter (zero at launch).
template <int PASS, int D>
__global__ void __launch_bounds__(kThreads, 2)
    profile_tc_kernel(const __grid_constant__ CUtensorMap tmQ,
                      const __grid_constant__ CUtensorMap tmK, float* __restrict__ nlse2,
                      float* __restrict__ colsum, float* __restrict__ bandcol, int G, int n,
                      int ld, int nt, int w, float sl2, int H, int R,
                      const int32_t* __restrict__ heads, const int32_t* __restrict__ n_heads,
                      int32_t* __restrict__ sched, int32_t* __restrict__ err, int stall) {
  extern __shared__ uint8_t smem_raw[];
  TcSmem<D>& s = *reinterpret_cast<TcSmem<D>*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int* abort = &s.abort;
  const CUtensorMap* mapA = PASS == 1 ? &tmQ : &tmK;
  const CUtensorMap* mapB = PASS == 1 ? &tmK : &tmQ;

  if (warp == 0) {
    tmem_alloc(&s.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  if (threadIdx.x == kTmaWarp * 32) {
    s.abort = 0;
    mbar_init(&s.a_full, 1);
    mbar_init(&s.a_empty, 1);
#pragma unroll
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&s.full[i], 1);
      mbar_init(&s.empty[i], 1);
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s.sfull[i], 1);
      mbar_init(&s.sempty[i], kConsumerWarps);
      mbar_init(&s.unit_full[i], 1);
      mbar_init(&s.unit_empty[i], kConsumerWarps + 1);
      mbar_init(&s.part_ready[i], kConsumerWarps / 2);
      mbar_init(&s.part_done[i], kConsumerWarps / 2);
    }
#pragma unroll
    for (int i = 0; i < kLseSlots; ++i) {
      mbar_init(&s.lfull[i], 1);
      mbar_init(&s.lempty[i], kConsumerWarps);
    }
    fence_barrier_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s.tmem_base;
  // the set-up above overlaps the previous kernel; its outputs are read below
  griddep_wait();
  griddep_launch_dependents();

  if (warp == kTmaWarp) {
    // ------------------------------------------------------- producer (TMA)
    // stall != 0 (a test of the error path only): the producer never starts,
    // so the other warps' first waits run out and the CTA unwinds with
    // nothing in flight
    if (lane == 0 && !stall) {
      // every head, or the listed ones (a saved policy map)
      const int total_units = (heads ? *n_heads : G) * nt;
      int bseq = 0, lseq = 0, ucount = 0;
      int u = atomicAdd(sched, 1);
      while (true) {
        const int us = ucount & 1;
        if (ucount >= 2 && !wait_or_abort(&s.unit_empty[us], ((ucount >> 1) - 1) & 1, abort))
          break;
        if (u >= total_units) {
          s.unit[us].valid = 0;
          mbar_arrive(&s.unit_full[us]);
          break;
        }
        const int g = heads ? heads[u / nt] : u / nt, tile = u % nt;
        UnitMeta um;
        um.g = g;
        um.valid = 1;
        if (PASS == 1) {
          um.at = nt - 1 - tile;
          um.b_first = 0;
          um.nb = um.at + 1;
        } else {
          um.at = tile;
          um.b_first = tile;
          um.nb = nt - tile;
        }
        s.unit[us] = um;
        mbar_arrive(&s.unit_full[us]);
        const int nxt = atomicAdd(sched, 1);  // claimed now, used after this unit
        // the operand loaded per unit may be replaced once the previous
        // unit's MMAs are done with it
        if (ucount >= 1 && !wait_or_abort(&s.a_empty, (ucount - 1) & 1, abort)) break;
        // Q rows come from query head g, K rows from its key/value head
        const int gk = kv_head(g, H, R);
        mbar_expect_tx(&s.a_full, TileCfg<D>::kTileBytes);
        load_tile<D>(s.a, mapA, &s.a_full, um.at * kBlk, PASS == 1 ? g : gk);
        bool stop = false;
        for (int t = 0; t < um.nb; ++t) {
          const int st = bseq % kStages;
          if (bseq >= kStages && !wait_or_abort(&s.empty[st], ((bseq / kStages) - 1) & 1, abort)) {
            stop = true;
            break;
          }
          mbar_expect_tx(&s.full[st], TileCfg<D>::kTileBytes);
          load_tile<D>(s.b[st], mapB, &s.full[st], (um.b_first + t) * kBlk, PASS == 1 ? gk : g);
          ++bseq;
          if (PASS == 2) {
            const int ls = lseq % kLseSlots;
            if (lseq >= kLseSlots &&
                !wait_or_abort(&s.lempty[ls], ((lseq / kLseSlots) - 1) & 1, abort)) {
              stop = true;
              break;
            }
            mbar_expect_tx(&s.lfull[ls], kBlk * sizeof(float));
            bulk_load(s.nlse[ls], nlse2 + (size_t)g * ld + (size_t)(um.b_first + t) * kBlk,
                      kBlk * sizeof(float), &s.lfull[ls]);
            ++lseq;
          }
        }
        if (stop) break;
        ++ucount;
        u = nxt;
      }
      if (*abort) {  // let the copies still in flight land before exiting
        for (int q = bseq > kStages ? bseq - kStages : 0; q < bseq; ++q)
          mbar_wait(&s.full[q % kStages], (q / kStages) & 1);
        for (int q = lseq > kLseSlots ? lseq - kLseSlots : 0; q < lseq; ++q)
          mbar_wait(&s.lfull[q % kLseSlots], (q / kLseSlots) & 1);
        mbar_wait(&s.a_full, ucount & 1);
      }
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------------ MMA
    if (lane == 0) {
      int bseq = 0, sseq = 0, ucount = 0, acommits = 0;
      while (true) {
        const int us = ucount & 1;
        if (!wait_or_abort(&s.unit_full[us], (ucount >> 1) & 1, abort)) break;
        const UnitMeta um = s.unit[us];
        mbar_arrive(&s.unit_empty[us]);
        if (!um.valid) break;
        if (!wait_or_abort(&s.a_full, ucount & 1, abort)) break;
        bool stop = false;
        for (int t = 0; t < um.nb; ++t) {
          const int st = bseq % kStages, buf = sseq & 1;
          if (!wait_or_abort(&s.full[st], (bseq / kStages) & 1, abort) ||
              (sseq >= 2 && !wait_or_abort(&s.sempty[buf], ((sseq >> 1) - 1) & 1, abort))) {
            stop = true;
            break;
          }
          tc_fence_after();
          issue_tile_mma<D>(tmem + buf * kBlk, smem_addr(s.a), smem_addr(s.b[st]));
          umma_commit(&s.sfull[buf]);
          umma_commit(&s.empty[st]);
          ++bseq;
          ++sseq;
        }
        umma_commit(&s.a_empty);  // the unit's operand is free once these complete
        ++acommits;
        if (stop) break;
        ++ucount;
      }
      // every MMA (and the arrivals it triggers) must complete before exit;
      // the operand-release commit is the last one issued
      for (int q = bseq > kStages ? bseq - kStages : 0; q < bseq; ++q)
        mbar_wait(&s.empty[q % kStages], (q / kStages) & 1);
      if (acommits > 0) mbar_wait(&s.a_empty, (acommits - 1) & 1);
    }
  } else {
    // ------------------------------------------------------------ consumers
    // warp w reads TMEM lanes 32*(w%4).. (its rows) and columns 64*(w/4)..
    const int row = (warp & 3) * 32 + lane;  // TMEM lane = tile row
    const int c0 = (warp >> 2) * kHalfCols;
    const uint32_t lane_base = tmem + ((uint32_t)((warp & 3) * 32) << 16) + c0;
    int sseq = 0, lseq = 0, ucount = 0;
    while (true) {
      const int us = ucount & 1;
      if (!wait_or_abort(&s.unit_full[us], (ucount >> 1) & 1, abort)) break;
      const UnitMeta um = s.unit[us];
      __syncwarp();
      if (lane == 0) mbar_arrive(&s.unit_empty[us]);
      if (!um.valid) break;
      const int self = um.at * kBlk + row;  // query (pass 1) or key (pass 2) position
      float m = FG_NEG_INF, l = 0.f;         // pass 1: running max and sum (base 2)
      float cs = 0.f, bs = 0.f;              // pass 2: column and band sums
      bool stop = false;
      for (int t = 0; t < um.nb; ++t) {
        const int buf = sseq & 1;
        const int other0 = (um.b_first + t) * kBlk;  // first key / query of the tile
        if (!wait_or_abort(&s.sfull[buf], (sseq >> 1) & 1, abort)) {
          stop = true;
          break;
        }
        tc_fence_after();
        if (PASS == 1) {
          uint32_t r[2][32];
          tmem_ld32(lane_base + buf * kBlk, r[0]);
          tmem_ld32(lane_base + buf * kBlk + 32, r[1]);
          tmem_wait_ld(r[0]);
          reg_barrier(r[1]);
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&s.sempty[buf]);
          ++sseq;
          // key columns j = other0 + c are valid for j <= self and j < n
          const int lim = min(self + 1, n) - other0;
          lse_tile(r, sl2, c0, lim < kBlk ? max(lim, 0) : -1, m, l);
        } else {
          const int ls = lseq % kLseSlots;
          if (!wait_or_abort(&s.lfull[ls], (lseq / kLseSlots) & 1, abort)) {
            stop = true;
            break;
          }
          // query columns i = other0 + c count for i >= self and lie in the
          // window for i < self + w; the row is read in two halves of 32
          // columns to keep the register pressure low
          uint32_t r[1][32];
          float4 Lv[8];
#pragma unroll
          for (int e = 0; e < 8; ++e)
            Lv[e] = *reinterpret_cast<const float4*>(s.nlse[ls] + c0 + 4 * e);
          tmem_ld32(lane_base + buf * kBlk, r[0]);
          tmem_wait_ld(r[0]);
          col_tile<1>(r, Lv, sl2, c0, self - other0, self + w - other0, cs, bs);
#pragma unroll
          for (int e = 0; e < 8; ++e)
            Lv[e] = *reinterpret_cast<const float4*>(s.nlse[ls] + c0 + 32 + 4 * e);
          tmem_ld32(lane_base + buf * kBlk + 32, r[0]);
          tmem_wait_ld(r[0]);
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&s.sempty[buf]);
          ++sseq;
          col_tile<1>(r, Lv, sl2, c0 + 32, self - other0, self + w - other0, cs, bs);
          __syncwarp();
          if (lane == 0) mbar_arrive(&s.lempty[ls]);
          ++lseq;
        }
      }
      if (stop) break;
      // merge the two column halves of every row: the second half hands over
      const int ps = ucount & 1;
      if (c0 != 0) {
        if (ucount >= 2 && !wait_or_abort(&s.part_done[ps], ((ucount >> 1) - 1) & 1, abort))
          break;
        s.part[ps][0][row] = PASS == 1 ? m : cs;
        s.part[ps][1][row] = PASS == 1 ? l : bs;
        __syncwarp();
        if (lane == 0) mbar_arrive(&s.part_ready[ps]);
      } else {
        if (!wait_or_abort(&s.part_ready[ps], (ucount >> 1) & 1, abort)) break;
        const float p0 = s.part[ps][0][row], p1 = s.part[ps][1][row];
        __syncwarp();
        if (lane == 0) mbar_arrive(&s.part_done[ps]);
        if (PASS == 1) {
          const float M = fmaxf(m, p0);
          const float L = l * ex2(m - M) + p1 * ex2(p0 - M);
          nlse2[(size_t)um.g * ld + self] = self < n ? -(M + __log2f(L)) : FG_NEG_INF;
        } else if (self < n) {
          colsum[(size_t)um.g * n + self] = cs + p0;
          bandcol[(size_t)um.g * n + self] = bs + p1;
        }
      }
      ++ucount;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0 && s.abort) atomicOr(err, 2);
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ---------------------------------------------------------------------------
// Pass 3: the prompt attention output O = A V (query-major), with the row
// log-sum-exps of pass 1, so every weight is final when it is formed and the
// accumulator is never rescaled.  Unit (g, query tile) streams key tiles
// j <= i: S = Q K^T lands in tensor memory (two buffers), 16 consumer warps
// (four per TMEM lane quarter, 32 columns each) form P = 2^(s' S + nlse) in
// bf16 and store it back to tensor memory (two P buffers; row = lane, key
// pairs packed per column), where the MMA warp takes it as the A operand of
// O += P V, V read straight from its TMA tile as an MN-major B operand.  At
// the end of a unit the consumers read O (d fp32 columns) and store it.  The
// query tile is double-buffered so the next unit's loads during this one.
// One CTA per SM (the Q, K and V buffers fill shared memory).
constexpr int kAttnConsumerWarps = 16;
constexpr int kAttnTmaWarp = kAttnConsumerWarps, kAttnMmaWarp = kAttnConsumerWarps + 1;
constexpr int kAttnThreads = (kAttnConsumerWarps + 2) * 32;
// tensor memory: S buffers at columns 0 and 128, O at 256, P buffers at 384, 448
constexpr uint32_t kAttnTmemCols = 512;
constexpr uint32_t kAttnOCol = 2 * kBlk;
constexpr uint32_t kAttnPCol = 3 * kBlk;

template <int D>
struct alignas(1024) AttnSmem {
  uint8_t q[2][TileCfg<D>::kTileBytes];  // this unit's and the next unit's queries
  uint8_t k[kStages][TileCfg<D>::kTileBytes];
  uint8_t v[kStages][TileCfg<D>::kTileBytes];
  UnitMeta unit[2];
  int abort;
  uint64_t a_full[2], a_empty[2];
  uint64_t kfull[kStages], kempty[kStages], vfull[kStages], vempty[kStages];
  uint64_t s_full[2], s_empty[2], pfull[2], pempty[2], o_full, o_empty;
  uint64_t unit_full[2], unit_empty[2];
  uint32_t tmem_base;
};

// Shared-memory descriptor of an MN-major bf16 operand in the 128-byte
// swizzled layout TMA writes for a [K rows x 64 elements] box: 8-row groups
// (along K) 1024 bytes apart, 64-element column blocks (along MN) one box
// (kHalfBytes) apart.
__device__ __forceinline__ uint64_t desc_mnmajor_sw128(uint32_t saddr, uint32_t mn_stride) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)((mn_stride >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)(1024u >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

// (lo, hi) -> bf16x2, lo in the low half, round to nearest even.
__device__ __forceinline__ uint32_t pack_bf16x2_rn(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// D[tmem] (+)= A[tmem] * B[smem]: the A operand read from tensor memory (its
// rows on the lanes, two bf16 per 32-bit column along K).
__device__ __forceinline__ void umma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                             uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// 16 consecutive 32-bit columns of this thread's TMEM lane (32x32b shape).
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15])
      : "memory");
}

// Non-blocking test of an mbarrier phase.
__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// O += P V over one key tile: P [128 x 128 keys] in tensor memory (64
// columns), V [128 keys x D] MN-major in shared memory (D of N).
template <int D>
__device__ __forceinline__ void issue_pv_mma(uint32_t o_tmem, uint32_t p_tmem, uint32_t v_base,
                                             bool accumulate) {
  constexpr uint32_t idesc = idesc_bf16_f32(kBlk, D) | (1u << 16);  // B MN-major
#pragma unroll
  for (int kk = 0; kk < kBlk / 16; ++kk)
    umma_bf16_ts(o_tmem, p_tmem + kk * 8,
                 desc_mnmajor_sw128(v_base + kk * 16 * 128, TileCfg<D>::kHalfBytes), idesc,
                 (accumulate || kk > 0) ? 1u : 0u);
}

// nlse2: pass 1's negated base-2 row LSEs (row stride ld); out [G, n, D].
template <int D>
__global__ void __launch_bounds__(kAttnThreads, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, const float* __restrict__ nlse2,
                   __nv_bfloat16* __restrict__ out, int G, int n, int ld, int nt, float sl2,
                   int H, int R, int32_t* __restrict__ sched, int32_t* __restrict__ err) {
  extern __shared__ uint8_t smem_raw[];
  AttnSmem<D>& s = *reinterpret_cast<AttnSmem<D>*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int* abort = &s.abort;

  if (warp == 0) {
    tmem_alloc(&s.tmem_base, kAttnTmemCols);
    tmem_relinquish();
  }
  if (threadIdx.x == kAttnTmaWarp * 32) {
    s.abort = 0;
#pragma unroll
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&s.kfull[i], 1);
      mbar_init(&s.kempty[i], 1);
      mbar_init(&s.vfull[i], 1);
      mbar_init(&s.vempty[i], 1);
    }
    mbar_init(&s.o_full, 1);
    mbar_init(&s.o_empty, kAttnConsumerWarps);
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s.a_full[i], 1);
      mbar_init(&s.a_empty[i], 1);
      mbar_init(&s.s_full[i], 1);
      mbar_init(&s.s_empty[i], kAttnConsumerWarps);
      mbar_init(&s.pfull[i], kAttnConsumerWarps);
      mbar_init(&s.pempty[i], 1);
      mbar_init(&s.unit_full[i], 1);
      mbar_init(&s.unit_empty[i], kAttnConsumerWarps + 1);
    }
    fence_barrier_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s.tmem_base;
  griddep_wait();
  griddep_launch_dependents();

  if (warp == kAttnTmaWarp) {
    // ------------------------------------------------------- producer (TMA)
    if (lane == 0) {
      const int total_units = G * nt;
      int kseq = 0, vseq = 0, ucount = 0;
      int u = atomicAdd(sched, 1);
      while (true) {
        const int us = ucount & 1;
        if (ucount >= 2 && !wait_or_abort(&s.unit_empty[us], ((ucount >> 1) - 1) & 1, abort))
          break;
        if (u >= total_units) {
          s.unit[us].valid = 0;
          mbar_arrive(&s.unit_full[us]);
          break;
        }
        const int g = u / nt, tile = u % nt;
        UnitMeta um;
        um.g = g;
        um.valid = 1;
        um.at = nt - 1 - tile;  // longest units first
        um.b_first = 0;
        um.nb = um.at + 1;
        s.unit[us] = um;
        mbar_arrive(&s.unit_full[us]);
        const int nxt = atomicAdd(sched, 1);
        // the query tile of the unit two back must be released
        if (ucount >= 2 && !wait_or_abort(&s.a_empty[us], ((ucount >> 1) - 1) & 1, abort)) break;
        const int gk = kv_head(g, H, R);
        mbar_expect_tx(&s.a_full[us], TileCfg<D>::kTileBytes);
        load_tile<D>(s.q[us], &tmQ, &s.a_full[us], um.at * kBlk, g);
        bool stop = false;
        for (int t = 0; t < um.nb && !stop; ++t) {
          const int ks = kseq % kStages;
          if (kseq >= kStages && !wait_or_abort(&s.kempty[ks], ((kseq / kStages) - 1) & 1, abort)) {
            stop = true;
            break;
          }
          mbar_expect_tx(&s.kfull[ks], TileCfg<D>::kTileBytes);
          load_tile<D>(s.k[ks], &tmK, &s.kfull[ks], t * kBlk, gk);
          ++kseq;
          const int vs = vseq % kStages;
          if (vseq >= kStages && !wait_or_abort(&s.vempty[vs], ((vseq / kStages) - 1) & 1, abort)) {
            stop = true;
            break;
          }
          mbar_expect_tx(&s.vfull[vs], TileCfg<D>::kTileBytes);
          load_tile<D>(s.v[vs], &tmV, &s.vfull[vs], t * kBlk, gk);
          ++vseq;
        }
        if (stop) break;
        ++ucount;
        u = nxt;
      }
      if (*abort) {  // let the copies still in flight land before exiting
        for (int q = kseq > kStages ? kseq - kStages : 0; q < kseq; ++q)
          mbar_wait(&s.kfull[q % kStages], (q / kStages) & 1);
        for (int q = vseq > kStages ? vseq - kStages : 0; q < vseq; ++q)
          mbar_wait(&s.vfull[q % kStages], (q / kStages) & 1);
        mbar_wait(&s.a_full[ucount & 1], (ucount >> 1) & 1);
      }
    }
  } else if (warp == kAttnMmaWarp) {
    // ------------------------------------------------------------------ MMA
    if (lane == 0) {
      int kseq = 0, vseq = 0, sseq = 0, pseq = 0, ucount = 0, ocount = 0, acommits = 0;
      while (true) {
        const int us = ucount & 1;
        if (!wait_or_abort(&s.unit_full[us], (ucount >> 1) & 1, abort)) break;
        const UnitMeta um = s.unit[us];
        mbar_arrive(&s.unit_empty[us]);
        if (!um.valid) break;
        if (!wait_or_abort(&s.a_full[us], (ucount >> 1) & 1, abort)) break;
        // Issue order follows readiness: a tile's scores go out as soon as
        // its K tile has landed and the score buffer it reuses has been read
        // (up to two tiles ahead of the consumers), a tile's P V as soon as
        // its weights are in tensor memory.  One thread polls both.
        bool stop = false;
        int si = 0, pi = 0, idle = 0;
        uint64_t t0 = global_timer_ns();
        while (pi < um.nb) {
          bool did = false;
          if (si < um.nb) {  // scores of key tile si
            const int ks = kseq % kStages, sb = sseq & 1;
            if (mbar_test(&s.kfull[ks], (kseq / kStages) & 1) &&
                (sseq < 2 || mbar_test(&s.s_empty[sb], ((sseq >> 1) - 1) & 1))) {
              tc_fence_after();
              issue_tile_mma<D>(tmem + sb * kBlk, smem_addr(s.q[us]), smem_addr(s.k[ks]));
              umma_commit(&s.s_full[sb]);
              umma_commit(&s.kempty[ks]);
              ++kseq;
              ++sseq;
              ++si;
              did = true;
            }
          }
          if (pi < si) {  // weighted values of key tile pi
            const int vs = vseq % kStages, pb = pseq & 1;
            if (mbar_test(&s.pfull[pb], (pseq >> 1) & 1) &&
                mbar_test(&s.vfull[vs], (vseq / kStages) & 1) &&
                (pi > 0 || ocount == 0 || mbar_test(&s.o_empty, (ocount - 1) & 1))) {
              tc_fence_after();
              issue_pv_mma<D>(tmem + kAttnOCol, tmem + kAttnPCol + pb * 64, smem_addr(s.v[vs]),
                              pi > 0);
              umma_commit(&s.pempty[pb]);
              umma_commit(&s.vempty[vs]);
              ++pseq;
              ++vseq;
              ++pi;
              did = true;
            }
          }
          if (did) {
            idle = 0;
            t0 = global_timer_ns();
            continue;
          }
          if (*abort) {
            stop = true;
            break;
          }
          if (++idle >= 64) {  // bounded like every other wait
            idle = 0;
            if (global_timer_ns() - t0 > kWaitLimitNs) {
              *abort = 1;
              stop = true;
              break;
            }
          }
        }
        if (stop) break;
        umma_commit(&s.o_full);
        ++ocount;
        umma_commit(&s.a_empty[us]);
        ++acommits;
        ++ucount;
      }
      // every MMA issued must complete before exit; the last commits cover them
      if (acommits > 0) mbar_wait(&s.a_empty[(acommits - 1) & 1], ((acommits - 1) >> 1) & 1);
      for (int q = kseq > kStages ? kseq - kStages : 0; q < kseq; ++q)
        mbar_wait(&s.kempty[q % kStages], (q / kStages) & 1);
      for (int q = vseq > kStages ? vseq - kStages : 0; q < vseq; ++q)
        mbar_wait(&s.vempty[q % kStages], (q / kStages) & 1);
    }
  } else {
    // ------------------------------------------------------------ consumers
    // warp w reads TMEM lanes 32*(w%4).. (its rows), S columns 32*(w/4)..
    // and O columns 32*(w/4).. (those below D)
    const int qd = warp & 3, cg = warp >> 2;
    const int row = qd * 32 + lane;
    const uint32_t lane_base = tmem + ((uint32_t)(qd * 32) << 16);
    int sseq = 0, pseq = 0, ucount = 0;
    while (true) {
      const int us = ucount & 1;
      if (!wait_or_abort(&s.unit_full[us], (ucount >> 1) & 1, abort)) break;
      const UnitMeta um = s.unit[us];
      __syncwarp();
      if (lane == 0) mbar_arrive(&s.unit_empty[us]);
      if (!um.valid) break;
      const int qpos = um.at * kBlk + row;                   // query position
      const float nl = nlse2[(size_t)um.g * ld + qpos];      // -inf past the prompt
      bool stop = false;
      for (int t = 0; t < um.nb; ++t) {
        const int sb = sseq & 1;
        if (!wait_or_abort(&s.s_full[sb], (sseq >> 1) & 1, abort)) {
          stop = true;
          break;
        }
        tc_fence_after();
        uint32_t r[32];
        tmem_ld32(lane_base + sb * kBlk + cg * 32, r);
        tmem_wait_ld(r);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&s.s_empty[sb]);
        ++sseq;
        // keys t*128 + cg*32 + e count for key <= query and key < n
        const int lim = min(qpos + 1, n) - (t * kBlk + cg * 32);
        uint32_t pk[16];
        if (lim >= 32) {  // every key of the chunk counts: packed arithmetic, no tests
          const uint64_t s2 = pack2(sl2, sl2), nl2 = pack2(nl, nl);
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            float x0, x1;
            unpack2(fma2(pack2(f(r[e]), f(r[e + 1])), s2, nl2), x0, x1);
            pk[e >> 1] = pack_bf16x2_rn(ex2(x0), ex2(x1));
          }
        } else {
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            const float p0 = e < lim ? ex2(fmaf(f(r[e]), sl2, nl)) : 0.f;
            const float p1 = e + 1 < lim ? ex2(fmaf(f(r[e + 1]), sl2, nl)) : 0.f;
            pk[e >> 1] = pack_bf16x2_rn(p0, p1);
          }
        }
        const int pb = pseq & 1;
        if (pseq >= 2 && !wait_or_abort(&s.pempty[pb], ((pseq >> 1) - 1) & 1, abort)) {
          stop = true;
          break;
        }
        tc_fence_after();
        tmem_st16(lane_base + kAttnPCol + pb * 64 + cg * 16, pk);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&s.pfull[pb]);
        ++pseq;
      }
      if (stop) break;
      // the unit's output rows
      if (!wait_or_abort(&s.o_full, ucount & 1, abort)) break;
      tc_fence_after();
      uint32_t o[32];
      if (cg * 32 < D) {  // D = 64: the warps of column groups 0 and 1 read 32 columns each
        const int c0 = cg * 32;
        tmem_ld32(lane_base + kAttnOCol + c0, o);
        tmem_wait_ld(o);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&s.o_empty);
        if (qpos < n) {
          __nv_bfloat16* dst = out + ((size_t)um.g * n + qpos) * D + c0;
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            uint32_t w4[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              __nv_bfloat162 h = __floats2bfloat162_rn(f(o[8 * c + 2 * e]), f(o[8 * c + 2 * e + 1]));
              w4[e] = *reinterpret_cast<uint32_t*>(&h);
            }
            *reinterpret_cast<uint4*>(dst + 8 * c) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
          }
        }
      } else {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&s.o_empty);
      }
      ++ucount;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0 && s.abort) atomicOr(err, 2);
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kAttnTmemCols);
  }
}

using EncodeFn = PFN_cuTensorMapEncodeTiled_v12000;

EncodeFn encoder() {
  static EncodeFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeFn>(p);
  }
  return fn;
}

// [G, n, D] bf16 viewed as a 3-D tensor (D innermost); box 64 x 128 x 1 with
// the 128-byte swizzle, out-of-range rows read as zero.
bool make_map(CUtensorMap* map, const void* base, int G, int n, int D) {
  EncodeFn enc = encoder();
  if (!enc) return false;
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)n, (cuuint64_t)G};
  cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)n * D * 2};
  cuuint32_t box[3] = {64, (cuuint32_t)kBlk, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
             box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

int sm_count() {
  static int cached[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (!cached[dev]) {
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    cached[dev] = v;
  }
  return cached[dev];
}

template <int D>
cudaError_t run(const ProfileDims& pd, const void* Q, const void* K, float* nlse2, int ld,
                float* colsum, float* bandcol, const int32_t* heads, const int32_t* n_heads,
                int32_t* sched, int32_t* err, int stall_pass, cudaStream_t s) {
  CUtensorMap tq, tk;
  if (!make_map(&tq, Q, pd.G, pd.n, D) || !make_map(&tk, K, pd.Gkv, pd.n, D))
    return cudaErrorInvalidValue;
  const int nt = cdiv(pd.n, kBlk);
  const size_t smem = sizeof(TcSmem<D>) + 1024;
  cudaError_t e = cudaFuncSetAttribute(profile_tc_kernel<1, D>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(profile_tc_kernel<2, D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem);
  if (e != cudaSuccess) return e;
  const long long units = (long long)pd.G * nt;
  const int sms = sm_count();
  if (sms <= 0) return cudaErrorInvalidDevice;
  const unsigned grid = (unsigned)(units < 2LL * sms ? units : 2LL * sms);
  // the work counters were zeroed by the token-class kernel launched before
  e = launch_pdl(profile_tc_kernel<1, D>, grid, kThreads, smem, s, tq, tk, nlse2, colsum, bandcol,
                 pd.G, pd.n, ld, nt, pd.w, pd.sl2, pd.H, pd.R, heads, n_heads, sched, err,
                 (int)(stall_pass == 1));
  if (e == cudaSuccess)
    e = launch_pdl(profile_tc_kernel<2, D>, grid, kThreads, smem, s, tq, tk, nlse2, colsum,
                   bandcol, pd.G, pd.n, ld, nt, pd.w, pd.sl2, pd.H, pd.R, heads, n_heads,
                   sched + 1, err, (int)(stall_pass == 2));
  return e;
}

template <int D>
cudaError_t run_attn(const ProfileDims& pd, const void* Q, const void* K, const void* V,
                     const float* nlse2, int ld, void* out, int32_t* sched, int32_t* err,
                     cudaStream_t s) {
  CUtensorMap tq, tk, tv;
  if (!make_map(&tq, Q, pd.G, pd.n, D) || !make_map(&tk, K, pd.Gkv, pd.n, D) ||
      !make_map(&tv, V, pd.Gkv, pd.n, D))
    return cudaErrorInvalidValue;
  const int nt = cdiv(pd.n, kBlk);
  const size_t smem = sizeof(AttnSmem<D>) + 1024;
  cudaError_t e = cudaFuncSetAttribute(attn_tc_kernel<D>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const long long units = (long long)pd.G * nt;
  const int sms = sm_count();
  if (sms <= 0) return cudaErrorInvalidDevice;
  const unsigned grid = (unsigned)(units < sms ? units : sms);
  return launch_pdl(attn_tc_kernel<D>, grid, kAttnThreads, smem, s, tq, tk, tv, nlse2,
                    (__nv_bfloat16*)out, pd.G, pd.n, ld, nt, pd.sl2, pd.H, pd.R, sched, err);
}

}  // namespace

bool profile_tc_supported(const ProfileDims& pd) {
  return pd.dtype == FG_BF16 && (pd.d == 64 || pd.d == 128) &&
         (long long)pd.G * cdiv(pd.n, kBlk) < (1LL << 31);
}

cudaError_t launch_profile_tc(const ProfileDims& pd, const void* Q, const void* K, float* lse2,
                              int ld, float* colsum, float* bandcol, const int32_t* heads,
                              const int32_t* n_heads, int32_t* sched, int32_t* err,
                              int stall_pass, cudaStream_t s) {
  return pd.d == 64 ? run<64>(pd, Q, K, lse2, ld, colsum, bandcol, heads, n_heads, sched, err,
                              stall_pass, s)
                    : run<128>(pd, Q, K, lse2, ld, colsum, bandcol, heads, n_heads, sched, err,
                               stall_pass, s);
}

cudaError_t launch_attn_tc(const ProfileDims& pd, const void* Q, const void* K, const void* V,
                           const float* lse2, int ld, void* out, int32_t* sched, int32_t* err,
                           cudaStream_t s) {
  return pd.d == 64 ? run_attn<64>(pd, Q, K, V, lse2, ld, out, sched, err, s)
                    : run_attn<128>(pd, Q, K, V, lse2, ld, out, sched, err, s);
}

}  // namespace fg
