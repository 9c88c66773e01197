// Prompt profiling on the tcgen05 tensor cores (bf16 Q/K, fp32 accumulate).
//
// FastGen profiles every head on A = softmax(s Q K^T) under the causal mask
// (Model Tells You What to Discard, Method, eq. (C*)); the policies need, per
// key j, colsum_j = sum_i A_ij and the band sum bandcol_j = sum_{j<=i<j+w} A_ij.
// A is never written to memory.  Two passes over 128 x 128 score tiles:
//   pass 1, query-major: CTA (g, query tile) streams its causal key tiles,
//     S = Q_tile K_tile^T lands in tensor memory, the consumer warps keep the
//     running row max and sum and write the base-2 row log-sum-exp;
//   pass 2, key-major: CTA (g, key tile) streams query tiles i >= j,
//     S^T = K_tile Q_tile^T, and each consumer thread owns one key (one TMEM
//     lane), so its column and band sums accumulate in registers.
// Warp roles per CTA: warps 0-3 consume TMEM (thread = tile row), warp 4
// issues TMA loads (128-byte swizzled tiles, double-buffered), warp 5 issues
// the MMAs (one thread) into two TMEM accumulators of 128 columns.
// Every wait is bounded (about 1 s); on timeout the CTA records bit 1 in the
// error word, lets its copies and MMAs land, frees tensor memory and exits.
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

template <int D>
struct alignas(1024) TcSmem {
  uint8_t a[TileCfg<D>::kTileBytes];             // loaded once: Q (pass 1) or K (pass 2)
  uint8_t b[kStages][TileCfg<D>::kTileBytes];    // streamed: K (pass 1) or Q (pass 2)
  float nlse[kLseSlots][kBlk];                   // pass 2: negated row LSEs of a query tile
  float part[2][kBlk];                           // second-half partial results per row
  int bad;                                       // some thread timed out
  uint64_t bar_a;
  uint64_t bar_full[kStages], bar_empty[kStages];
  uint64_t bar_sfull[2], bar_sempty[2];
  uint64_t bar_lfull[kLseSlots], bar_lempty[kLseSlots];
  uint32_t tmem_base;
};

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

// Pass 2, one thread's 64 columns (starting at tile column c0) of a key row:
// adds sum A to cs and the part inside the band to bs.  nl = negated base-2
// LSEs of the tile's 128 queries (-inf past the prompt end).  Tile columns
// c < lo precede the key (masked); columns c < band lie in the window.
__device__ __forceinline__ void col_tile(const uint32_t (&r)[2][32], const float* nl, float sl2,
                                         int c0, int lo, int band, float& cs, float& bs) {
  const uint64_t s2 = pack2(sl2, sl2);
  if (lo <= c0 && (band <= c0 || band >= c0 + kHalfCols)) {  // no per-element test
    uint64_t acc[4] = {0, 0, 0, 0};
#pragma unroll
    for (int c = 0; c < 2; ++c)
#pragma unroll
      for (int e = 0; e < 32; e += 4) {
        const float4 L = *reinterpret_cast<const float4*>(nl + c0 + c * 32 + e);
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
    if (band >= c0 + kHalfCols) bs += t;
    return;
  }
  float ta[4] = {0.f, 0.f, 0.f, 0.f}, ba[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int c = 0; c < 2; ++c)
#pragma unroll
    for (int e = 0; e < 32; ++e) {
      const int col = c0 + c * 32 + e;
      float p = ex2(fmaf(f(r[c][e]), sl2, nl[col]));
      p = col < lo ? 0.f : p;
      ta[e & 3] += p;
      ba[e & 3] += col < band ? p : 0.f;
    }
  cs += (ta[0] + ta[1]) + (ta[2] + ta[3]);
  bs += (ba[0] + ba[1]) + (ba[2] + ba[3]);
}

// PASS 1: nlse2[g, i] = -log2 sum_j 2^(s' q_i.k_j) (row stride ld) of the
//         CTA's query tile; rows past the prompt get -inf.
// PASS 2: colsum / bandcol of the CTA's key tile.
template <int PASS, int D>
__global__ void __launch_bounds__(kThreads, 2)
    profile_tc_kernel(const __grid_constant__ CUtensorMap tmQ,
                      const __grid_constant__ CUtensorMap tmK, float* __restrict__ nlse2,
                      float* __restrict__ colsum, float* __restrict__ bandcol, int G, int n,
                      int ld, int nt, int w, float sl2, int32_t* __restrict__ err) {
  extern __shared__ uint8_t smem_raw[];
  TcSmem<D>& s = *reinterpret_cast<TcSmem<D>*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // Head-major order, so the tiles of one head run together and share its
  // K (pass 1) or Q (pass 2) tiles through L2; longest tiles first in a head.
  const int g = blockIdx.x / nt, tile = blockIdx.x % nt;
  int at, b_first, nb;
  if (PASS == 1) {
    at = nt - 1 - tile;
    b_first = 0;
    nb = at + 1;
  } else {
    at = tile;
    b_first = tile;
    nb = nt - tile;
  }
  const CUtensorMap* mapA = PASS == 1 ? &tmQ : &tmK;
  const CUtensorMap* mapB = PASS == 1 ? &tmK : &tmQ;

  if (warp == 0) {
    tmem_alloc(&s.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  if (threadIdx.x == kTmaWarp * 32) {
    s.bad = 0;
    mbar_init(&s.bar_a, 1);
#pragma unroll
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&s.bar_full[i], 1);
      mbar_init(&s.bar_empty[i], 1);
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s.bar_sfull[i], 1);
      mbar_init(&s.bar_sempty[i], kConsumerWarps);
    }
#pragma unroll
    for (int i = 0; i < kLseSlots; ++i) {
      mbar_init(&s.bar_lfull[i], 1);
      mbar_init(&s.bar_lempty[i], kConsumerWarps);
    }
    fence_barrier_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s.tmem_base;
  bool ok = true;
  float m = FG_NEG_INF, l = 0.f;  // pass 1 consumer state: running max and sum (base 2)
  float cs = 0.f, bs = 0.f;       // pass 2 consumer state: column and band sums

  if (warp == kTmaWarp) {
    // ---------------------------------------------------------------- TMA
    if (lane == 0) {
      mbar_expect_tx(&s.bar_a, TileCfg<D>::kTileBytes);
      load_tile<D>(s.a, mapA, &s.bar_a, at * kBlk, g);
      int issued = 0, lissued = 0;
      for (int t = 0; t < nb; ++t) {
        const int st = t % kStages;
        if (t >= kStages && !mbar_wait(&s.bar_empty[st], ((t / kStages) - 1) & 1)) {
          ok = false;
          break;
        }
        mbar_expect_tx(&s.bar_full[st], TileCfg<D>::kTileBytes);
        load_tile<D>(s.b[st], mapB, &s.bar_full[st], (b_first + t) * kBlk, g);
        issued = t + 1;
        if (PASS == 2) {
          const int ls = t % kLseSlots;
          if (t >= kLseSlots && !mbar_wait(&s.bar_lempty[ls], ((t / kLseSlots) - 1) & 1)) {
            ok = false;
            break;
          }
          mbar_expect_tx(&s.bar_lfull[ls], kBlk * sizeof(float));
          bulk_load(s.nlse[ls], nlse2 + (size_t)g * ld + (size_t)(b_first + t) * kBlk,
                    kBlk * sizeof(float), &s.bar_lfull[ls]);
          lissued = t + 1;
        }
      }
      if (!ok) {  // let every issued copy land before the CTA can exit
        mbar_wait(&s.bar_a, 0);
        for (int t = issued > kStages ? issued - kStages : 0; t < issued; ++t)
          mbar_wait(&s.bar_full[t % kStages], (t / kStages) & 1);
        for (int t = lissued > kLseSlots ? lissued - kLseSlots : 0; t < lissued; ++t)
          mbar_wait(&s.bar_lfull[t % kLseSlots], (t / kLseSlots) & 1);
      }
    }
  } else if (warp == kMmaWarp) {
    // ---------------------------------------------------------------- MMA
    if (lane == 0) {
      int issued = 0;
      if (!mbar_wait(&s.bar_a, 0)) ok = false;
      for (int t = 0; ok && t < nb; ++t) {
        const int st = t % kStages, buf = t & 1;
        if (!mbar_wait(&s.bar_full[st], (t / kStages) & 1)) {
          ok = false;
          break;
        }
        if (t >= 2 && !mbar_wait(&s.bar_sempty[buf], ((t >> 1) - 1) & 1)) {
          ok = false;
          break;
        }
        tc_fence_after();
        issue_tile_mma<D>(tmem + buf * kBlk, smem_addr(s.a), smem_addr(s.b[st]));
        umma_commit(&s.bar_sfull[buf]);
        umma_commit(&s.bar_empty[st]);
        issued = t + 1;
      }
      // the MMAs (and the arrivals they trigger) must complete before exit
      for (int t = issued > kStages ? issued - kStages : 0; t < issued; ++t)
        mbar_wait(&s.bar_empty[t % kStages], (t / kStages) & 1);
    }
  } else {
    // ------------------------------------------------------------ consumers
    // warp w reads TMEM lanes 32*(w%4).. (its rows) and columns 64*(w/4)..
    const int row = (warp & 3) * 32 + lane;  // TMEM lane = tile row
    const int c0 = (warp >> 2) * kHalfCols;
    const uint32_t lane_base = tmem + ((uint32_t)((warp & 3) * 32) << 16) + c0;
    const int self = at * kBlk + row;  // query (pass 1) or key (pass 2) position
    for (int t = 0; t < nb; ++t) {
      const int buf = t & 1;
      const int other0 = (b_first + t) * kBlk;  // first key (pass 1) / query (pass 2) of the tile
      if (!mbar_wait(&s.bar_sfull[buf], (t >> 1) & 1)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t r[2][32];
      tmem_ld32(lane_base + buf * kBlk, r[0]);
      tmem_ld32(lane_base + buf * kBlk + 32, r[1]);
      tmem_wait_ld(r[0]);
      reg_barrier(r[1]);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&s.bar_sempty[buf]);

      if (PASS == 1) {
        // key columns j = other0 + c are valid for j <= self and j < n
        const int lim = min(self + 1, n) - other0;
        lse_tile(r, sl2, c0, lim < kBlk ? max(lim, 0) : -1, m, l);
      } else {
        const int ls = t % kLseSlots;
        if (!mbar_wait(&s.bar_lfull[ls], (t / kLseSlots) & 1)) {
          ok = false;
          break;
        }
        // query columns i = other0 + c count for i >= self and lie in the
        // window for i < self + w
        col_tile(r, s.nlse[ls], sl2, c0, self - other0, self + w - other0, cs, bs);
        __syncwarp();
        if (lane == 0) mbar_arrive(&s.bar_lempty[ls]);
      }
    }
    if (c0 != 0) {  // hand the second half's partial state to the first half
      s.part[0][row] = PASS == 1 ? m : cs;
      s.part[1][row] = PASS == 1 ? l : bs;
    }
  }
  if (!ok) {
    atomicOr(err, 2);
    s.bad = 1;
  }
  tc_fence_before();
  __syncthreads();
  if (warp < 4 && !s.bad) {  // first-half threads merge the halves and write
    const int row = warp * 32 + lane;
    const int self = at * kBlk + row;
    const float p0 = s.part[0][row], p1 = s.part[1][row];
    if (PASS == 1) {
      const float M = fmaxf(m, p0);
      const float L = l * ex2(m - M) + p1 * ex2(p0 - M);
      nlse2[(size_t)g * ld + self] = self < n ? -(M + __log2f(L)) : FG_NEG_INF;
    } else if (self < n) {
      colsum[(size_t)g * n + self] = cs + p0;
      bandcol[(size_t)g * n + self] = bs + p1;
    }
  }
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
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

template <int D>
cudaError_t run(const ProfileDims& pd, const void* Q, const void* K, float* nlse2, int ld,
                float* colsum, float* bandcol, int32_t* err, cudaStream_t s) {
  CUtensorMap tq, tk;
  if (!make_map(&tq, Q, pd.G, pd.n, D) || !make_map(&tk, K, pd.G, pd.n, D))
    return cudaErrorInvalidValue;
  const int nt = cdiv(pd.n, kBlk);
  const size_t smem = sizeof(TcSmem<D>) + 1024;
  cudaError_t e = cudaFuncSetAttribute(profile_tc_kernel<1, D>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(profile_tc_kernel<2, D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem);
  if (e != cudaSuccess) return e;
  const unsigned grid = (unsigned)pd.G * (unsigned)nt;
  profile_tc_kernel<1, D><<<grid, kThreads, smem, s>>>(tq, tk, nlse2, colsum, bandcol, pd.G, pd.n,
                                                      ld, nt, pd.w, pd.sl2, err);
  profile_tc_kernel<2, D><<<grid, kThreads, smem, s>>>(tq, tk, nlse2, colsum, bandcol, pd.G, pd.n,
                                                      ld, nt, pd.w, pd.sl2, err);
  return cudaGetLastError();
}

}  // namespace

bool profile_tc_supported(const ProfileDims& pd) {
  return pd.dtype == FG_BF16 && (pd.d == 64 || pd.d == 128) &&
         (long long)pd.G * cdiv(pd.n, kBlk) < (1LL << 31);
}

cudaError_t launch_profile_tc(const ProfileDims& pd, const void* Q, const void* K, float* lse2,
                              int ld, float* colsum, float* bandcol, int32_t* err,
                              cudaStream_t s) {
  return pd.d == 64 ? run<64>(pd, Q, K, lse2, ld, colsum, bandcol, err, s)
                    : run<128>(pd, Q, K, lse2, ld, colsum, bandcol, err, s);
}

}  // namespace fg
