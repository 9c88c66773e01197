// One generation step over the per-head compressed caches (Model Tells You
// What to Discard, Method: head-specific KV caches, keys/values appended at
// each step, the prompt-time policy reused during generation).
//
// Split-K over a static work list: item (c, i) covers rpw rows (256, or 512
// in plans with many items) of
// cache c's never-evicted segment or of its window ring (one cache per
// key/value head; its R query heads all attend over it).  The segment's last
// item also covers every row appended after the prompt, so no item is spent
// on the reserve that is still empty.  Each CTA
//   * places the new token if its slot falls in the item (the only writer of
//     that row; it attends with the new key/value from registers, so no CTA
//     reads a row written in this launch),
//   * streams its K/V rows once with 16-byte loads (one row per LPR lanes)
//     and scores every row against the R queries of the group: fp32 dots
//     (fp64 for fp32 inputs) and an online base-2 softmax per lane group and
//     query,
//   * writes (max, sum, acc[d]) per query for the item.
// A second launch merges each query head's items (log-sum-exp merge), writes
// out[g] and bumps the cache's never-evicted row count.  Both are launched as
// programmatic dependents of the kernel before them.  With one query per
// cache the pass is HBM-bound on the SIMT lanes; grouped bf16 caches score
// and accumulate with warp-level MMAs (split_mma_kernel).
#include <type_traits>

#include "fg_common.cuh"
#include "fg_internal.h"

namespace fg {
namespace {

constexpr int kDecThreads = 256;
constexpr int kDecWarps = kDecThreads / 32;

struct Placement {
  bool st;        // joins the never-evicted segment
  bool overflow;  // wanted to, but the segment is full
};

// The parts of a work item fixed before the step: the item, its cache's
// descriptor and the step token's class.  Kernels read them before waiting
// on the previous kernel (programmatic launch), which never writes them: the
// plan wrote the work list and descriptors, the caller the token ids.  Only
// the segment's row count (n_static) changes from step to step (the combine
// advances it); it is read after the wait, from L2, since the descriptor's
// line may sit in L1 from the earlier read.
struct ItemStatic {
  int2 it;          // (cache, item of the cache)
  fg_head_desc hd;  // its n_static is not current until live_rows replaces it
  bool is_s, is_p;  // the step's token is special / punctuation
};

// c: cache (key/value head) index; HLkv = L * Hkv caches per sequence.
__device__ __forceinline__ ItemStatic item_static(const DecodeArgs& a, int HLkv, int2 it) {
  ItemStatic s;
  s.it = it;
  s.hd = a.desc[it.x];
  const int tau = a.new_ids[it.x / HLkv];
  s.is_s = id_in(tau, a.special, a.ns);
  s.is_p = id_in(tau, a.punct, a.np);
  return s;
}

__device__ __forceinline__ int live_rows(const DecodeArgs& a, int c) {
  return __ldcg(&a.desc[c].n_static);
}

__device__ __forceinline__ Placement place(const fg_head_desc& hd, bool is_s, bool is_p) {
  Placement pl;
  pl.st = joins_static(hd.policy, is_s, is_p);
  pl.overflow = pl.st && hd.n_static >= hd.static_cap;
  if (pl.overflow) pl.st = false;
  return pl;
}

// The rows of one work item and the step's bookkeeping on them.
struct Item {
  int c;         // cache
  int r0, r1;    // rows [r0, r1) of the segment
  int new_slot;  // row of the new token in the segment, or -1
  int evict;     // ring row that left the window, or -1
  bool ring;     // the item covers the window ring (else the never-evicted segment)
  long long base;  // first pool row of the segment
};

// Sets up work item s.it (after the wait), writes the new token's row if its
// slot falls in the item (the only writer of that row) and marks an evicted
// ring row empty.  Only the segment's last item depends on the live row
// count: every earlier item was full at the prompt's end (the plan gives a
// segment ceil(kept / rpw) items) and never holds the new slot, and whether
// the token enters the ring does not depend on the count either (it does
// unless it is one the never-evicted segment takes, whether or not that
// segment has room).
template <typename T, int D>
__device__ __forceinline__ Item item_setup(const DecodeArgs& a, const ItemStatic& s) {
  constexpr int LPR = D / Vec16<T>::kElems;
  Item m;
  m.c = s.it.x;
  int chunk = s.it.y;
  fg_head_desc hd = s.hd;
  const int rpw = a.rpw;
  const int nsc = hd.n_work - cdiv(hd.w, rpw);  // items of the never-evicted segment
  m.ring = chunk >= nsc;
  m.evict = -1;
  m.new_slot = -1;
  if (!m.ring) {
    m.r0 = chunk * rpw;
    m.base = hd.off;
    if (chunk == nsc - 1) {
      hd.n_static = live_rows(a, m.c);
      const Placement pl = place(hd, s.is_s, s.is_p);
      m.r1 = hd.n_static + (pl.st ? 1 : 0);
      m.new_slot = pl.st ? hd.n_static : -1;
      if (pl.overflow && threadIdx.x == 0) atomicOr(a.dev_err, 1);
    } else {
      m.r1 = m.r0 + rpw;
    }
  } else {
    chunk -= nsc;
    m.r0 = chunk * rpw;
    m.r1 = min(m.r0 + rpw, hd.w);
    m.base = hd.win_off;
    const int slot = a.pos % hd.w;
    const bool ring_put = hd.policy == FG_POLICY_SPFL && hd.w > 0 &&
                          !joins_static(hd.policy, s.is_s, s.is_p);
    m.new_slot = ring_put ? slot : -1;
    m.evict = ring_put ? -1 : slot;  // the row that left the window
  }
  if (m.new_slot >= m.r0 && m.new_slot < m.r1) {
    T* Kp = (T*)a.Kp;
    T* Vp = (T*)a.Vp;
    const T* kn = (const T*)a.k_new + (size_t)m.c * D;
    const T* vn = (const T*)a.v_new + (size_t)m.c * D;
    constexpr int E = Vec16<T>::kElems;
    for (int v = threadIdx.x; v < LPR; v += blockDim.x) {
      const size_t d = (size_t)(m.base + m.new_slot) * D + v * E;
      *reinterpret_cast<uint4*>(Kp + d) = *reinterpret_cast<const uint4*>(kn + v * E);
      *reinterpret_cast<uint4*>(Vp + d) = *reinterpret_cast<const uint4*>(vn + v * E);
    }
    if (threadIdx.x == 0) {
      a.posp[m.base + m.new_slot] = a.pos;
      if (a.row_acc) a.row_acc[m.base + m.new_slot] = 0.f;  // a generated token starts at 0
    }
  }
  if (m.evict >= m.r0 && m.evict < m.r1 && threadIdx.x == 0) a.posp[m.base + m.evict] = -1;
  return m;
}

// R = queries per cache (group size).  Rows are unrolled by U per warp so
// that 2 * U 16-byte loads per thread are in flight.
// kAcc (one query per cache): also write every row's score to a.row_sc.
// Single-query bf16 caches keep four CTAs per SM (64 registers): the row
// stream needs that many rows in flight.
template <typename T, int D, int R, bool kAcc = false>
__global__ void __launch_bounds__(kDecThreads, R == 1 && sizeof(T) == 2 ? 4 : 1)
    split_kernel(const DecodeArgs a, int H, int HLkv, float sl2) {
  static_assert(!kAcc || R == 1, "row scores are kept for single-query caches only");
  constexpr int E = Vec16<T>::kElems;
  constexpr int LPR = D / E;     // lanes per row
  constexpr int RPW = 32 / LPR;  // rows per warp per load
  constexpr int STEP = kDecWarps * RPW;
  constexpr int U = R <= 2 ? 4 : 2;
  constexpr bool kWide = sizeof(T) == 4;  // fp32 inputs: fp64 dot, scaled once
  using Score = typename std::conditional<kWide, double, float>::type;
  __shared__ float sm_m[R][kDecWarps], sm_l[R][kDecWarps];
  __shared__ float sm_acc[R][kDecWarps][D];

  const ItemStatic st = item_static(a, HLkv, a.work[blockIdx.x]);
  griddep_wait();
  griddep_launch_dependents();
  const Item it = item_setup<T, D>(a, st);
  const int wi = blockIdx.x;
  const int c = it.c, r0 = it.r0, r1 = it.r1, new_slot = it.new_slot, evict = it.evict;
  const bool ring = it.ring;
  const long long base = it.base;
  const T* Kp = (const T*)a.Kp;
  const T* Vp = (const T*)a.Vp;
  const T* kn = (const T*)a.k_new + (size_t)c * D;
  const T* vn = (const T*)a.v_new + (size_t)c * D;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int grp = lane / LPR, gl = lane % LPR;
  const int Hkv = H / R;
  const size_t g0 = (size_t)(c / Hkv) * H + (size_t)(c % Hkv) * R;  // first query head
  float qf[R][E];
#pragma unroll
  for (int q = 0; q < R; ++q) {
    load16((const T*)a.q + (g0 + q) * D + gl * E, qf[q]);
    if (!kWide) {
#pragma unroll
      for (int e = 0; e < E; ++e) qf[q][e] *= sl2;
    }
  }
  float m[R], l[R], acc[R][E];
#pragma unroll
  for (int q = 0; q < R; ++q) {
    m[q] = FG_NEG_INF;
    l[q] = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) acc[q][e] = 0.f;
  }

  for (int rb = r0; rb < r1; rb += STEP * U) {
    uint4 kv[U], vv[U];
    bool ok[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int r = rb + (u * kDecWarps + warp) * RPW + grp;
      const bool in = r < r1;
      const bool fresh = r == new_slot;
      ok[u] = in && (fresh || !ring || (r != evict && a.posp[base + r] >= 0));
      if (in) {
        const T* kr = fresh ? kn : Kp + (size_t)(base + r) * D;
        const T* vr = fresh ? vn : Vp + (size_t)(base + r) * D;
        kv[u] = ldg_stream(kr + gl * E);
        vv[u] = ldg_stream(vr + gl * E);
      } else {
        kv[u] = make_uint4(0, 0, 0, 0);
        vv[u] = make_uint4(0, 0, 0, 0);
      }
    }
    // fp32 inputs keep the score in fp64 and round the running max up to an
    // integer, so that score - max and the merges of partial maxima are exact
    // (an fp32 score of ~185 in base-2 units carries ~1e-5 of rounding)
    Score sc[U][R];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      float f[E];
      unpack16(kv[u], f, (const T*)nullptr);
#pragma unroll
      for (int q = 0; q < R; ++q) {
        Score dot;
        if (kWide) {
          double dd = 0.0;
#pragma unroll
          for (int e = 0; e < E; ++e) dd = fma((double)qf[q][e], (double)f[e], dd);
#pragma unroll
          for (int o = LPR / 2; o >= 1; o >>= 1) dd += __shfl_xor_sync(0xffffffffu, dd, o);
          dot = (Score)(dd * (double)sl2);
        } else {
          float df = 0.f;
#pragma unroll
          for (int e = 0; e < E; ++e) df = fmaf(qf[q][e], f[e], df);
#pragma unroll
          for (int o = LPR / 2; o >= 1; o >>= 1) df += __shfl_xor_sync(0xffffffffu, df, o);
          dot = (Score)df;
        }
        sc[u][q] = ok[u] ? dot : (Score)FG_NEG_INF;
      }
      if constexpr (kAcc) {
        const int r = rb + (u * kDecWarps + warp) * RPW + grp;
        if (gl == 0 && r < r1) a.row_sc[base + r] = (float)sc[u][0];
      }
    }
#pragma unroll
    for (int q = 0; q < R; ++q) {
      Score mloc = (Score)FG_NEG_INF;
#pragma unroll
      for (int u = 0; u < U; ++u) mloc = sc[u][q] > mloc ? sc[u][q] : mloc;
      float mnew = kWide ? (float)ceil((double)mloc) : (float)mloc;
      mnew = fmaxf(m[q], mnew);
      if (mnew == FG_NEG_INF) continue;
      const float corr = exp2f(m[q] - mnew);
      l[q] *= corr;
#pragma unroll
      for (int e = 0; e < E; ++e) acc[q][e] *= corr;
#pragma unroll
      for (int u = 0; u < U; ++u) {
        if (ok[u]) {
          const float p = exp2f((float)(sc[u][q] - (Score)mnew));
          float f[E];
          unpack16(vv[u], f, (const T*)nullptr);
          l[q] += p;
#pragma unroll
          for (int e = 0; e < E; ++e) acc[q][e] = fmaf(p, f[e], acc[q][e]);
        }
      }
      m[q] = mnew;
    }
  }
#pragma unroll
  for (int q = 0; q < R; ++q) {
    // merge the lane groups of the warp
#pragma unroll
    for (int o = LPR; o < 32; o <<= 1) {
      const float m2 = __shfl_xor_sync(0xffffffffu, m[q], o);
      const float l2 = __shfl_xor_sync(0xffffffffu, l[q], o);
      float a2[E];
#pragma unroll
      for (int e = 0; e < E; ++e) a2[e] = __shfl_xor_sync(0xffffffffu, acc[q][e], o);
      const float M = fmaxf(m[q], m2);
      if (M != FG_NEG_INF) {
        const float fa = exp2f(m[q] - M), fb = exp2f(m2 - M);
        l[q] = l[q] * fa + l2 * fb;
#pragma unroll
        for (int e = 0; e < E; ++e) acc[q][e] = acc[q][e] * fa + a2[e] * fb;
        m[q] = M;
      }
    }
    if (grp == 0) {
#pragma unroll
      for (int e = 0; e < E; ++e) sm_acc[q][warp][gl * E + e] = acc[q][e];
      if (gl == 0) {
        sm_m[q][warp] = m[q];
        sm_l[q][warp] = l[q];
      }
    }
  }
  __syncthreads();
  if (threadIdx.x < D) {
    const int t = threadIdx.x;
#pragma unroll
    for (int q = 0; q < R; ++q) {
      float M = FG_NEG_INF;
#pragma unroll
      for (int w = 0; w < kDecWarps; ++w) M = fmaxf(M, sm_m[q][w]);
      float L = 0.f, A = 0.f;
      if (M != FG_NEG_INF) {
#pragma unroll
        for (int w = 0; w < kDecWarps; ++w) {
          const float f = exp2f(sm_m[q][w] - M);
          L += sm_l[q][w] * f;
          A += sm_acc[q][w][t] * f;
        }
      }
      const size_t slot = (size_t)wi * R + q;
      a.part_acc[slot * D + t] = A;
      if (t == 0) {
        a.part_ml[2 * slot] = M;
        a.part_ml[2 * slot + 1] = L;
      }
    }
  }
}

// ---------------------------------------------------------------------------
// bf16 caches on warp MMAs.
//
// Scoring every row against R queries on the SIMT lanes costs R dot products,
// R lane reductions and R rescaled accumulators per row: at R >= 4 that is
// instruction-bound well below the bandwidth of the row stream.  Here each
// warp takes 16-row blocks and does both products as register-level bf16
// MMAs (m16n8k16, fp32 accumulate), with the queries on the N = 8 side:
//   S^T[16 keys x 8 q]  = K[16 keys x d] . Q^T[d x 8 q]
//   O^T[d x 8 q]       += V^T[d x 16 keys] . P^T[16 keys x 8 q]
// Rows reach shared memory through cp.async (16-byte pieces, zero-filled for
// rows that must not be read, the new token's row taken from the step's
// input), in a per-warp ring of kMmaStages blocks, so loads stay in flight
// without holding registers; fragments come from ldmatrix (K) and
// ldmatrix.trans (V) on rows padded by 16 bytes (conflict-free).  P is split
// into a bf16 high part and a bf16 remainder (two MMAs), so the weights keep
// ~16 significant bits, as the fp32 SIMT path does.  S^T's accumulator
// fragment becomes P^T's operand fragment with one 8x8 transpose per half
// (movmatrix).  tcgen05's smallest tile (M >= 64) is far above the <= 8
// queries of a group, so these are warp MMAs.
constexpr int kMmaWarps = 4;
constexpr int kMmaThreads = kMmaWarps * 32;
constexpr int kMmaBlk = 16;                                   // rows per MMA tile
constexpr int kMmaStages = 2;                                 // V blocks in flight per warp
static_assert(kRowsPerWork % (kMmaWarps * kMmaBlk) == 0, "items are whole blocks");

template <int D>
struct MmaSmem {
  static constexpr int kStride = D + 8;                        // padded V row, elements
  static constexpr int kStageElems = kMmaBlk * kStride;
  static constexpr size_t kRingBytes = (size_t)kMmaWarps * kMmaStages * kStageElems * 2;
  template <int R>
  static constexpr size_t bytes() {
    // the merge buffers reuse the rings once every warp is done with them
    constexpr size_t merge = (size_t)kMmaWarps * R * D * 4;
    return kRingBytes > merge ? kRingBytes : merge;
  }
};

__device__ __forceinline__ void mma_bf16_16816(float (&c)[4], uint32_t a0, uint32_t a1,
                                               uint32_t a2, uint32_t a3, uint32_t b0,
                                               uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Transpose of an 8x8 b16 matrix held one row pair per lane (lane l: row l/4,
// columns 2(l%4), 2(l%4)+1).
__device__ __forceinline__ uint32_t transpose8x8(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

// (lo, hi) -> bf16x2 with lo in the low half, round to nearest even.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

// 16-byte global -> shared copy; bytes past src_bytes (0 or 16) are zeroed.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
               "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                          uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ uint32_t word(const uint4& v, int i) {
  return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

template <int D, int R>
__global__ void __launch_bounds__(kMmaThreads, 4) split_mma_kernel(const DecodeArgs a, int H,
                                                                   int HLkv, float sl2) {
  using T = __nv_bfloat16;
  using SM = MmaSmem<D>;
  constexpr int KI = D / 32;       // 16-byte pieces of a K row per lane (2 k-steps each)
  constexpr int MT = D / 16;       // 16-row tiles of O^T
  constexpr int PPR = D / 8;       // 16-byte pieces per V row
  constexpr int NP = kMmaBlk * PPR / 32;  // V pieces per lane per block
  constexpr int STR = SM::kStride;
  extern __shared__ __align__(16) uint8_t mma_smem[];
  __shared__ float sm_m[kMmaWarps][R], sm_l[kMmaWarps][R], sm_f[kMmaWarps][R];

  const ItemStatic st = item_static(a, HLkv, a.work[blockIdx.x]);
  griddep_wait();
  griddep_launch_dependents();
  const Item it = item_setup<T, D>(a, st);
  const int wi = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t4 = lane & 3;
  const T* Kp = (const T*)a.Kp;
  const T* Vp = (const T*)a.Vp;
  const T* kn = (const T*)a.k_new + (size_t)it.c * D;
  const T* vn = (const T*)a.v_new + (size_t)it.c * D;
  const int Hkv = H / R;
  const size_t g0 = (size_t)(it.c / Hkv) * H + (size_t)(it.c % Hkv) * R;  // first query head

  auto row_ok = [&](int r) -> bool {
    if (r >= it.r1) return false;
    if (r == it.new_slot || !it.ring) return true;
    return r != it.evict && a.posp[it.base + r] >= 0;
  };
  // This warp's blocks: rows first + W*16*b, b = 0 .. nblk-1, one after the
  // other with an online softmax across them.  K rows go to registers: the
  // next block's are requested as soon as the scores are formed.  V rows go
  // through a two-stage shared-memory ring by cp.async, the next block's
  // requested before this block's scores.
  const int first = it.r0 + warp * kMmaBlk;
  const int nblk =
      first < it.r1 ? cdiv(it.r1 - first, kMmaWarps * kMmaBlk) : 0;
  const uint32_t vring =
      smem_u32(mma_smem) + (uint32_t)(warp * kMmaStages * SM::kStageElems * 2);
  // K: rows g and g + 8 of a block, pieces {32 i + 8 t4}; k-step 2i + h takes
  // words 2h (d positions 2t4, 2t4+1) and 2h + 1 (positions 2t4+8, 2t4+9) of
  // piece i.  Q^T is loaded with the same permutation of d.
  auto load_k = [&](int rb, uint4 (&kr)[2][KI], bool (&kok)[2]) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int r = rb + g + 8 * h;
      kok[h] = row_ok(r);
      const T* p = r == it.new_slot ? kn : Kp + (size_t)(it.base + r) * D;
#pragma unroll
      for (int i = 0; i < KI; ++i)
        kr[h][i] = kok[h] ? ldg_stream(p + 32 * i + 8 * t4) : make_uint4(0, 0, 0, 0);
    }
  };
  auto issue_v = [&](int rb, int st) {
    const uint32_t vs = vring + (uint32_t)(st * SM::kStageElems * 2);
#pragma unroll
    for (int i = 0; i < NP; ++i) {
      const int pc = (lane + 32 * i) % PPR, row = (lane + 32 * i) / PPR;
      const int r = rb + row;
      const bool ok = row_ok(r);  // empty ring slots may hold anything: never read them
      const T* src = !ok ? vn : r == it.new_slot ? vn + pc * 8
                                                  : Vp + (size_t)(it.base + r) * D + pc * 8;
      cp_async16(vs + (uint32_t)((row * STR + pc * 8) * 2), src, ok ? 16 : 0);
    }
  };

  uint4 qv[KI];
  {
    const T* qr = (const T*)a.q + (g0 + (g < R ? g : 0)) * D;
#pragma unroll
    for (int i = 0; i < KI; ++i)
      qv[i] = g < R ? *reinterpret_cast<const uint4*>(qr + 32 * i + 8 * t4) : make_uint4(0, 0, 0, 0);
  }
  float m[2] = {FG_NEG_INF, FG_NEG_INF}, l[2] = {0.f, 0.f};
  float o[MT][4];
#pragma unroll
  for (int j = 0; j < MT; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
  uint4 kr[2][KI];
  bool kok[2];
  if (nblk > 0) {
    load_k(first, kr, kok);
    issue_v(first, 0);
  }
  cp_async_commit();
  // ldmatrix row addresses: lane l serves matrix l/8, row l%8; V^T tile j:
  // matrices (keys 8(lm>>1).., d 16j + 8(lm&1)..), transposed
  const int lm = lane >> 3, lr = lane & 7;
  const uint32_t vlane = (uint32_t)(((lr + 8 * (lm >> 1)) * STR + 8 * (lm & 1)) * 2);
#pragma unroll 1
  for (int b = 0; b < nblk; ++b) {
    const int rb = first + b * kMmaWarps * kMmaBlk, rn = rb + kMmaWarps * kMmaBlk;
    const bool more = b + 1 < nblk;
    if (more) issue_v(rn, (b + 1) % kMmaStages);
    cp_async_commit();
    // scores, base-2 units: (key g, q 2t4), (key g, q 2t4+1), (key g+8, q 2t4),
    // (key g+8, q 2t4+1)
    float sc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int i = 0; i < KI; ++i)
#pragma unroll
      for (int h = 0; h < 2; ++h)
        mma_bf16_16816(sc, word(kr[0][i], 2 * h), word(kr[1][i], 2 * h),
                       word(kr[0][i], 2 * h + 1), word(kr[1][i], 2 * h + 1), word(qv[i], 2 * h),
                       word(qv[i], 2 * h + 1));
#pragma unroll
    for (int e = 0; e < 4; ++e) sc[e] = kok[e >> 1] ? sc[e] * sl2 : FG_NEG_INF;
    if (more) load_k(rn, kr, kok);  // the K registers are free now
    // per query column: max over the block's rows (lanes of equal t4), then
    // the running max and the rescale of what is accumulated
    float me[2];
#pragma unroll
    for (int qc = 0; qc < 2; ++qc) {
      float v = fmaxf(sc[qc], sc[qc + 2]);
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
      const float mn = fmaxf(m[qc], v);
      const float corr = mn == FG_NEG_INF ? 1.f : exp2f(m[qc] - mn);
      l[qc] *= corr;
#pragma unroll
      for (int j = 0; j < MT; ++j) {
        o[j][qc] *= corr;
        o[j][qc + 2] *= corr;
      }
      m[qc] = mn;
      me[qc] = mn == FG_NEG_INF ? 0.f : mn;
    }
    float p[4];
    p[0] = exp2f(sc[0] - me[0]);
    p[1] = exp2f(sc[1] - me[1]);
    p[2] = exp2f(sc[2] - me[0]);
    p[3] = exp2f(sc[3] - me[1]);
    l[0] += p[0] + p[2];
    l[1] += p[1] + p[3];
    const uint32_t hi0 = pack_bf16x2(p[0], p[1]), hi1 = pack_bf16x2(p[2], p[3]);
    const uint32_t lo0 = pack_bf16x2(p[0] - bf16_lo(hi0), p[1] - bf16_hi(hi0));
    const uint32_t lo1 = pack_bf16x2(p[2] - bf16_lo(hi1), p[3] - bf16_hi(hi1));
    const uint32_t bh0 = transpose8x8(hi0), bh1 = transpose8x8(hi1);
    const uint32_t bl0 = transpose8x8(lo0), bl1 = transpose8x8(lo1);
    cp_async_wait<1>();  // this block's V rows have landed
    __syncwarp();
    {
      const uint32_t vaddr = vring + (uint32_t)((b % kMmaStages) * SM::kStageElems * 2) + vlane;
#pragma unroll
      for (int j = 0; j < MT; ++j) {
        uint32_t a0, a1, a2, a3;
        ldsm_x4_t(vaddr + j * 32, a0, a1, a2, a3);
        mma_bf16_16816(o[j], a0, a1, a2, a3, bh0, bh1);
        mma_bf16_16816(o[j], a0, a1, a2, a3, bl0, bl1);
      }
    }
    __syncwarp();  // the stage is refilled two blocks later
  }
  cp_async_wait<0>();
#pragma unroll
  for (int qc = 0; qc < 2; ++qc)
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) l[qc] += __shfl_xor_sync(0xffffffffu, l[qc], off);

  // O^T fragment of tile j: rows d = 16 j + g and d + 8, columns q = 2t4, 2t4 + 1.
  __syncthreads();  // every warp is done with its ring: the merge buffers reuse it
  float* sm_acc = reinterpret_cast<float*>(mma_smem);  // [W][R][D]
#pragma unroll
  for (int qc = 0; qc < 2; ++qc) {
    const int q = 2 * t4 + qc;
    if (q < R) {
      if (g == 0) {
        sm_m[warp][q] = m[qc];
        sm_l[warp][q] = l[qc];
      }
#pragma unroll
      for (int j = 0; j < MT; ++j) {
        sm_acc[(warp * R + q) * D + 16 * j + g] = o[j][qc];
        sm_acc[(warp * R + q) * D + 16 * j + g + 8] = o[j][qc + 2];
      }
    }
  }
  __syncthreads();
  if (threadIdx.x < R) {
    const int q = threadIdx.x;
    float M = FG_NEG_INF;
#pragma unroll
    for (int w = 0; w < kMmaWarps; ++w) M = fmaxf(M, sm_m[w][q]);
    float L = 0.f;
#pragma unroll
    for (int w = 0; w < kMmaWarps; ++w) {
      const float f = M == FG_NEG_INF || sm_m[w][q] == FG_NEG_INF ? 0.f : exp2f(sm_m[w][q] - M);
      sm_f[w][q] = f;
      L += sm_l[w][q] * f;
    }
    const size_t slot = (size_t)wi * R + q;
    a.part_ml[2 * slot] = M;
    a.part_ml[2 * slot + 1] = L;
  }
  __syncthreads();
  for (int x = threadIdx.x; x < R * D; x += kMmaThreads) {
    const int q = x / D, d = x % D;
    float A = 0.f;
#pragma unroll
    for (int w = 0; w < kMmaWarps; ++w) A = fmaf(sm_f[w][q], sm_acc[(w * R + q) * D + d], A);
    a.part_acc[((size_t)wi * R + q) * D + d] = A;
  }
}

// One CTA of D threads per query head, thread t = dimension t: every thread
// forms the item weights itself (a few exp2 per item, from broadcast loads)
// and sums its dimension over the items, so each item costs one coalesced
// row load for the whole CTA.
// kAcc (one query per cache): also record the head's final (M, L), from
// which acc_kernel adds each cached row's weight 2^(sc - M) / L.
template <typename T, int D, bool kAcc = false>
__global__ void __launch_bounds__(D) combine_kernel(const DecodeArgs a, int H, int R, int HLkv) {
  const int g = blockIdx.x;  // query head
  const int t = threadIdx.x;
  const int c = kv_head(g, H, R), q = (g % H) % R;  // its cache and place in the group
  ItemStatic st = item_static(a, HLkv, make_int2(c, 0));
  griddep_wait();
  griddep_launch_dependents();
  const fg_head_desc& hd = st.hd;
  // one member advances the shared cache; its row count is requested now so
  // that the load overlaps the partials'
  const bool bump = t == 0 && q == 0;
  const int live = bump ? live_rows(a, c) : 0;
  const size_t w0 = (size_t)hd.work_off;
  const int nw = hd.n_work;
  // items in chunks of 8: every load of a chunk is issued before any is used
  // (one memory round trip per chunk), then merged into the running
  // (M, L, acc) with a log-sum-exp rescale
  float M = FG_NEG_INF, L = 0.f, acc = 0.f;
  for (int i0 = 0; i0 < nw; i0 += 8) {
    float m[8], l[8], x[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const bool ok = i0 + j < nw;
      const size_t slot = (w0 + i0 + j) * R + q;
      m[j] = ok ? a.part_ml[2 * slot] : FG_NEG_INF;
      l[j] = ok ? a.part_ml[2 * slot + 1] : 0.f;
      x[j] = ok ? a.part_acc[slot * D + t] : 0.f;
    }
    float mc = m[0];
#pragma unroll
    for (int j = 1; j < 8; ++j) mc = fmaxf(mc, m[j]);
    const float Mn = fmaxf(M, mc);
    if (Mn == FG_NEG_INF) continue;
    const float f = M == FG_NEG_INF ? 0.f : exp2f(M - Mn);
    L *= f;
    acc *= f;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float wgt = m[j] == FG_NEG_INF ? 0.f : exp2f(m[j] - Mn);
      L = fmaf(wgt, l[j], L);
      acc = fmaf(wgt, x[j], acc);
    }
    M = Mn;
  }
  store_out((T*)a.out + (size_t)g * D + t, L > 0.f ? acc / L : 0.f);
  if (bump) {
    st.hd.n_static = live;
    const Placement pl = place(st.hd, st.is_s, st.is_p);
    if (pl.st) a.desc[c].n_static = live + 1;
  }
  if constexpr (kAcc) {
    if (t == 0) {
      a.head_ml[2 * g] = M;
      a.head_ml[2 * g + 1] = L;
    }
  }
}

// Adds every cached row's weight of the step, 2^(sc - M) / L with its head's
// final (M, L), to the row's accumulated score: one CTA per work item, one
// thread per row (the item's rows as the split kernel saw them).
__global__ void __launch_bounds__(kDecThreads) acc_kernel(const DecodeArgs a) {
  const int2 it = a.work[blockIdx.x];
  fg_head_desc hd = a.desc[it.x];
  griddep_wait();
  griddep_launch_dependents();
  hd.n_static = live_rows(a, it.x);
  const int rpw = a.rpw;
  const int nsc = hd.n_work - cdiv(hd.w, rpw);
  long long base;
  int r0, r1;
  if (it.y < nsc) {  // never-evicted segment (its row count already includes the new token)
    base = hd.off;
    r0 = it.y * rpw;
    r1 = it.y == nsc - 1 ? hd.n_static : min(r0 + rpw, hd.n_static);
  } else {
    base = hd.win_off;
    r0 = (it.y - nsc) * rpw;
    r1 = min(r0 + rpw, hd.w);
  }
  const float M = a.head_ml[2 * it.x], L = a.head_ml[2 * it.x + 1];
  if (M == FG_NEG_INF || !(L > 0.f)) return;
  const float inv = 1.f / L;
  for (int r = r0 + threadIdx.x; r < r1; r += blockDim.x) {
    const float sv = a.row_sc[base + r];
    if (sv != FG_NEG_INF) a.row_acc[base + r] += exp2f(sv - M) * inv;
  }
}

// Single-query caches with accumulated row scores (refresh of C_frequent).
template <typename T, int D>
cudaError_t run_acc(const ProfileDims& pd, const DecodeArgs& a, cudaStream_t s) {
  cudaError_t e = launch_pdl(split_kernel<T, D, 1, true>, a.n_work, kDecThreads, 0, s, a, pd.H,
                             pd.HLkv, pd.sl2);
  if (e == cudaSuccess)
    e = launch_pdl(combine_kernel<T, D, true>, pd.G, D, 0, s, a, pd.H, pd.R, pd.HLkv);
  if (e == cudaSuccess) e = launch_pdl(acc_kernel, a.n_work, kDecThreads, 0, s, a);
  return e;
}

template <typename T, int D, int R>
cudaError_t run(const ProfileDims& pd, const DecodeArgs& a, cudaStream_t s) {
  cudaError_t e;
  if constexpr (std::is_same<T, __nv_bfloat16>::value && R >= 2) {
    constexpr size_t smem = MmaSmem<D>::template bytes<R>();
    e = cudaFuncSetAttribute(split_mma_kernel<D, R>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem);
    if (e == cudaSuccess)
      e = launch_pdl(split_mma_kernel<D, R>, a.n_work, kMmaThreads, smem, s, a, pd.H, pd.HLkv,
                     pd.sl2);
  } else {
    e = launch_pdl(split_kernel<T, D, R>, a.n_work, kDecThreads, 0, s, a, pd.H, pd.HLkv, pd.sl2);
  }
  if (e == cudaSuccess)
    e = launch_pdl(combine_kernel<T, D>, pd.G, D, 0, s, a, pd.H, pd.R, pd.HLkv);
  return e;
}

template <typename T, int D>
cudaError_t run_r(const ProfileDims& pd, const DecodeArgs& a, cudaStream_t s) {
  switch (pd.R) {
    case 1: return run<T, D, 1>(pd, a, s);
    case 2: return run<T, D, 2>(pd, a, s);
    case 4: return run<T, D, 4>(pd, a, s);
    case 8: return run<T, D, 8>(pd, a, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_decode(const ProfileDims& pd, const DecodeArgs& a, cudaStream_t s) {
  if (a.row_acc) {
    if (pd.R != 1 || !a.row_sc || !a.head_ml) return cudaErrorInvalidValue;
    if (pd.dtype == FG_FP32)
      return pd.d == 64 ? run_acc<float, 64>(pd, a, s) : run_acc<float, 128>(pd, a, s);
    return pd.d == 64 ? run_acc<__nv_bfloat16, 64>(pd, a, s)
                      : run_acc<__nv_bfloat16, 128>(pd, a, s);
  }
  if (pd.dtype == FG_FP32)
    return pd.d == 64 ? run_r<float, 64>(pd, a, s) : run_r<float, 128>(pd, a, s);
  return pd.d == 64 ? run_r<__nv_bfloat16, 64>(pd, a, s) : run_r<__nv_bfloat16, 128>(pd, a, s);
}

}  // namespace fg
