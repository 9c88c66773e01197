// One generation step over the per-head compressed caches (Model Tells You
// What to Discard, Method: head-specific KV caches, keys/values appended at
// each step, the prompt-time policy reused during generation).
//
// Split-K over a static work list: item (c, i) covers up to kRowsPerWork
// rows of cache c's never-evicted segment or of its window ring (one cache
// per key/value head; its R query heads all attend over it).  Each CTA
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
// programmatic dependents of the kernel before them.  HBM-bound: no tensor
// cores (at most 8 queries share a K/V row).
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
  bool ring_put;  // goes into the window ring
};

// c: cache (key/value head) index; HLkv = L * Hkv caches per sequence.
__device__ __forceinline__ Placement place(const fg_head_desc& hd, const DecodeArgs& a, int HLkv,
                                           int c) {
  const int tau = a.new_ids[c / HLkv];
  const bool is_s = id_in(tau, a.special, a.ns), is_p = id_in(tau, a.punct, a.np);
  Placement pl;
  pl.st = joins_static(hd.policy, is_s, is_p);
  pl.overflow = pl.st && hd.n_static >= hd.static_cap;
  if (pl.overflow) pl.st = false;
  pl.ring_put = hd.policy == FG_POLICY_SPFL && !pl.st && !pl.overflow && hd.w > 0;
  return pl;
}

// R = queries per cache (group size).  Rows are unrolled by U per warp so
// that 2 * U 16-byte loads per thread are in flight.
template <typename T, int D, int R>
__global__ void __launch_bounds__(kDecThreads) split_kernel(const DecodeArgs a, int H, int HLkv,
                                                           float sl2) {
  constexpr int E = Vec16<T>::kElems;
  constexpr int LPR = D / E;     // lanes per row
  constexpr int RPW = 32 / LPR;  // rows per warp per load
  constexpr int STEP = kDecWarps * RPW;
  constexpr int U = R <= 2 ? 4 : 2;
  constexpr bool kWide = sizeof(T) == 4;  // fp32 inputs: fp64 dot, scaled once
  using Score = typename std::conditional<kWide, double, float>::type;
  __shared__ float sm_m[R][kDecWarps], sm_l[R][kDecWarps];
  __shared__ float sm_acc[R][kDecWarps][D];

  griddep_wait();
  griddep_launch_dependents();
  const int wi = blockIdx.x;
  const int2 it = a.work[wi];
  const int c = it.x;  // cache
  int chunk = it.y;
  const fg_head_desc hd = a.desc[c];
  const Placement pl = place(hd, a, HLkv, c);
  const int nsc = cdiv(hd.static_cap, kRowsPerWork);
  const bool ring = chunk >= nsc;
  int r0, r1, new_slot, evict = -1;
  long long base;
  if (!ring) {
    r0 = chunk * kRowsPerWork;
    r1 = min(r0 + kRowsPerWork, hd.n_static + (pl.st ? 1 : 0));
    base = hd.off;
    new_slot = pl.st ? hd.n_static : -1;
    if (pl.overflow && chunk == 0 && threadIdx.x == 0) atomicOr(a.dev_err, 1);
  } else {
    chunk -= nsc;
    r0 = chunk * kRowsPerWork;
    r1 = min(r0 + kRowsPerWork, hd.w);
    base = hd.win_off;
    const int slot = a.pos % hd.w;
    new_slot = pl.ring_put ? slot : -1;
    evict = pl.ring_put ? -1 : slot;  // the row that left the window
  }
  T* Kp = (T*)a.Kp;
  T* Vp = (T*)a.Vp;
  const T* kn = (const T*)a.k_new + (size_t)c * D;
  const T* vn = (const T*)a.v_new + (size_t)c * D;
  if (new_slot >= r0 && new_slot < r1) {
    for (int v = threadIdx.x; v < LPR; v += blockDim.x) {
      const size_t d = (size_t)(base + new_slot) * D + v * E;
      *reinterpret_cast<uint4*>(Kp + d) = *reinterpret_cast<const uint4*>(kn + v * E);
      *reinterpret_cast<uint4*>(Vp + d) = *reinterpret_cast<const uint4*>(vn + v * E);
    }
    if (threadIdx.x == 0) a.posp[base + new_slot] = a.pos;
  }
  if (evict >= r0 && evict < r1 && threadIdx.x == 0) a.posp[base + evict] = -1;

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

template <typename T, int D>
__global__ void __launch_bounds__(256) combine_kernel(const DecodeArgs a, int G, int H, int R,
                                                      int HLkv) {
  constexpr int PL = D / 32;
  griddep_wait();
  griddep_launch_dependents();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = blockIdx.x * 8 + warp;  // query head
  if (g >= G) return;
  const int c = kv_head(g, H, R), q = (g % H) % R;  // its cache and place in the group
  const fg_head_desc hd = a.desc[c];
  const size_t w0 = (size_t)hd.work_off;
  // items in groups of 32: lane i holds item i's (max, sum); the weights are
  // then broadcast while every lane sums its PL dimensions over the items
  float M = FG_NEG_INF;
  for (int i = lane; i < hd.n_work; i += 32) M = fmaxf(M, a.part_ml[2 * ((w0 + i) * R + q)]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  float L = 0.f, acc[PL];
#pragma unroll
  for (int e = 0; e < PL; ++e) acc[e] = 0.f;
  if (M != FG_NEG_INF) {
    for (int base = 0; base < hd.n_work; base += 32) {
      const int i = base + lane;
      float wgt = 0.f;
      if (i < hd.n_work) {
        const size_t slot = (w0 + i) * R + q;
        const float mi = a.part_ml[2 * slot];
        wgt = mi == FG_NEG_INF ? 0.f : exp2f(mi - M);
        L += wgt * a.part_ml[2 * slot + 1];
      }
      const int cnt = min(32, hd.n_work - base);
#pragma unroll 4
      for (int j = 0; j < cnt; ++j) {
        const float wj = __shfl_sync(0xffffffffu, wgt, j);
        const float* pa = a.part_acc + ((w0 + base + j) * R + q) * D + lane * PL;
#pragma unroll
        for (int e = 0; e < PL; ++e) acc[e] = fmaf(wj, pa[e], acc[e]);
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
  }
  T* out = (T*)a.out + (size_t)g * D;
  const float inv = L > 0.f ? 1.f / L : 0.f;
#pragma unroll
  for (int e = 0; e < PL; ++e) store_out(out + lane * PL + e, acc[e] * inv);
  if (lane == 0 && q == 0) {  // one member advances the shared cache
    const Placement pl = place(hd, a, HLkv, c);
    if (pl.st) a.desc[c].n_static = hd.n_static + 1;
  }
}

template <typename T, int D, int R>
cudaError_t run(const ProfileDims& pd, const DecodeArgs& a, cudaStream_t s) {
  cudaError_t e = launch_pdl(split_kernel<T, D, R>, a.n_work, kDecThreads, 0, s, a, pd.H, pd.HLkv,
                             pd.sl2);
  if (e == cudaSuccess)
    e = launch_pdl(combine_kernel<T, D>, cdiv(pd.G, 8), 256, 0, s, a, pd.G, pd.H, pd.R, pd.HLkv);
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
  if (pd.dtype == FG_FP32)
    return pd.d == 64 ? run_r<float, 64>(pd, a, s) : run_r<float, 128>(pd, a, s);
  return pd.d == 64 ? run_r<__nv_bfloat16, 64>(pd, a, s) : run_r<__nv_bfloat16, 128>(pd, a, s);
}

}  // namespace fg
