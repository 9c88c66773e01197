// One generation step over the per-head compressed caches (Model Tells You
// What to Discard, Method: head-specific KV caches, keys/values appended at
// each step, the prompt-time policy reused during generation).
//
// Split-K over a static work list: item (g, c) covers up to kRowsPerWork
// rows of head g's never-evicted segment or of its window ring.  Each CTA
//   * places the new token if its slot falls in the item (the only writer of
//     that row; it attends with the new key/value from registers, so no CTA
//     reads a row written in this launch),
//   * streams its K/V rows with 16-byte loads (one row per LPR lanes), does
//     the q.k dot in fp32 and an online base-2 softmax per lane group,
//   * writes (max, sum, acc[d]) for the item.
// A second launch merges the items of each head (log-sum-exp merge), writes
// out[g] and bumps the head's never-evicted row count.  HBM-bound: no tensor
// cores (a single query per head gives no reuse of the K/V rows).
#include "fg_common.cuh"
#include "fg_internal.h"

namespace fg {
namespace {

constexpr int kDecThreads = 256;
constexpr int kDecWarps = kDecThreads / 32;
constexpr int kUnroll = 4;

struct Placement {
  bool st;        // joins the never-evicted segment
  bool overflow;  // wanted to, but the segment is full
  bool ring_put;  // goes into the window ring
};

__device__ __forceinline__ Placement place(const fg_head_desc& hd, const DecodeArgs& a, int HL,
                                           int g) {
  const int tau = a.new_ids[g / HL];
  const bool is_s = id_in(tau, a.special, a.ns), is_p = id_in(tau, a.punct, a.np);
  Placement pl;
  pl.st = joins_static(hd.policy, is_s, is_p);
  pl.overflow = pl.st && hd.n_static >= hd.static_cap;
  if (pl.overflow) pl.st = false;
  pl.ring_put = hd.policy == FG_POLICY_SPFL && !pl.st && !pl.overflow && hd.w > 0;
  return pl;
}

template <typename T, int D>
__global__ void __launch_bounds__(kDecThreads) split_kernel(const DecodeArgs a, int HL, float sl2) {
  constexpr int E = Vec16<T>::kElems;
  constexpr int LPR = D / E;     // lanes per row
  constexpr int RPW = 32 / LPR;  // rows per warp per load
  constexpr int STEP = kDecWarps * RPW;
  __shared__ float sm_m[kDecWarps], sm_l[kDecWarps];
  __shared__ float sm_acc[kDecWarps][D];

  // Programmatic dependent launch: this grid may be scheduled while the
  // previous kernel of the stream finishes; wait for it before any access,
  // then let the next kernel be scheduled early in turn.
  griddep_wait();
  griddep_launch_dependents();
  const int wi = blockIdx.x;
  const int2 it = a.work[wi];
  const int g = it.x;
  int chunk = it.y;
  const fg_head_desc hd = a.desc[g];
  const Placement pl = place(hd, a, HL, g);
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
  const T* kn = (const T*)a.k_new + (size_t)g * D;
  const T* vn = (const T*)a.v_new + (size_t)g * D;
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
  // fp32 inputs: the dot is accumulated in fp64 and scaled once, so that
  // rounding does not perturb the scores key by key (the fp32 path is held
  // to 1e-5 on the outputs); bf16 inputs use an fp32 dot on a pre-scaled q.
  constexpr bool kWide = sizeof(T) == 4;
  float qf[E];
  load16((const T*)a.q + (size_t)g * D + gl * E, qf);
  if (!kWide) {
#pragma unroll
    for (int e = 0; e < E; ++e) qf[e] *= sl2;
  }
  float m = FG_NEG_INF, l = 0.f, acc[E];
#pragma unroll
  for (int e = 0; e < E; ++e) acc[e] = 0.f;

  for (int rb = r0; rb < r1; rb += STEP * kUnroll) {
    uint4 kv[kUnroll], vv[kUnroll];
    bool ok[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
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
    float s[kUnroll];
    float mloc = FG_NEG_INF;
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      float f[E];
      unpack16(kv[u], f, (const T*)nullptr);
      float dot;
      if (kWide) {
        double dd = 0.0;
#pragma unroll
        for (int e = 0; e < E; ++e) dd = fma((double)qf[e], (double)f[e], dd);
#pragma unroll
        for (int o = LPR / 2; o >= 1; o >>= 1) dd += __shfl_xor_sync(0xffffffffu, dd, o);
        dot = (float)(dd * (double)sl2);
      } else {
        dot = 0.f;
#pragma unroll
        for (int e = 0; e < E; ++e) dot = fmaf(qf[e], f[e], dot);
#pragma unroll
        for (int o = LPR / 2; o >= 1; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
      }
      s[u] = ok[u] ? dot : FG_NEG_INF;
      mloc = fmaxf(mloc, s[u]);
    }
    const float mnew = fmaxf(m, mloc);
    if (mnew != FG_NEG_INF) {
      const float corr = exp2f(m - mnew);
      l *= corr;
#pragma unroll
      for (int e = 0; e < E; ++e) acc[e] *= corr;
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        if (ok[u]) {
          const float p = exp2f(s[u] - mnew);
          float f[E];
          unpack16(vv[u], f, (const T*)nullptr);
          l += p;
#pragma unroll
          for (int e = 0; e < E; ++e) acc[e] = fmaf(p, f[e], acc[e]);
        }
      }
      m = mnew;
    }
  }
  // merge the lane groups of the warp
#pragma unroll
  for (int o = LPR; o < 32; o <<= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
    const float l2 = __shfl_xor_sync(0xffffffffu, l, o);
    float a2[E];
#pragma unroll
    for (int e = 0; e < E; ++e) a2[e] = __shfl_xor_sync(0xffffffffu, acc[e], o);
    const float M = fmaxf(m, m2);
    if (M != FG_NEG_INF) {
      const float fa = exp2f(m - M), fb = exp2f(m2 - M);
      l = l * fa + l2 * fb;
#pragma unroll
      for (int e = 0; e < E; ++e) acc[e] = acc[e] * fa + a2[e] * fb;
      m = M;
    }
  }
  if (grp == 0) {
#pragma unroll
    for (int e = 0; e < E; ++e) sm_acc[warp][gl * E + e] = acc[e];
    if (gl == 0) {
      sm_m[warp] = m;
      sm_l[warp] = l;
    }
  }
  __syncthreads();
  if (threadIdx.x < D) {
    const int t = threadIdx.x;
    float M = FG_NEG_INF;
#pragma unroll
    for (int w = 0; w < kDecWarps; ++w) M = fmaxf(M, sm_m[w]);
    float L = 0.f, A = 0.f;
    if (M != FG_NEG_INF) {
#pragma unroll
      for (int w = 0; w < kDecWarps; ++w) {
        const float f = exp2f(sm_m[w] - M);
        L += sm_l[w] * f;
        A += sm_acc[w][t] * f;
      }
    }
    a.part_acc[(size_t)wi * D + t] = A;
    if (t == 0) {
      a.part_ml[2 * (size_t)wi] = M;
      a.part_ml[2 * (size_t)wi + 1] = L;
    }
  }
}

template <typename T, int D>
__global__ void __launch_bounds__(256) combine_kernel(const DecodeArgs a, int G, int HL) {
  constexpr int PL = D / 32;
  griddep_wait();
  griddep_launch_dependents();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = blockIdx.x * 8 + warp;
  if (g >= G) return;
  const fg_head_desc hd = a.desc[g];
  const size_t w0 = (size_t)hd.work_off;
  // items in groups of 32: lane i holds item i's (max, sum); the weights are
  // then broadcast while every lane sums its PL dimensions over the items
  float M = FG_NEG_INF;
  for (int i = lane; i < hd.n_work; i += 32) M = fmaxf(M, a.part_ml[2 * (w0 + i)]);
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
        const float mi = a.part_ml[2 * (w0 + i)];
        wgt = mi == FG_NEG_INF ? 0.f : exp2f(mi - M);
        L += wgt * a.part_ml[2 * (w0 + i) + 1];
      }
      const int cnt = min(32, hd.n_work - base);
#pragma unroll 4
      for (int j = 0; j < cnt; ++j) {
        const float wj = __shfl_sync(0xffffffffu, wgt, j);
        const float* pa = a.part_acc + (w0 + base + j) * D + lane * PL;
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
  if (lane == 0) {
    const Placement pl = place(hd, a, HL, g);
    if (pl.st) a.desc[g].n_static = hd.n_static + 1;
  }
}

// Both kernels are launched as programmatic dependents of the kernel before
// them in the stream, hiding the launch gaps between decode steps.
template <typename T, int D>
cudaError_t run(const ProfileDims& pd, const DecodeArgs& a, cudaStream_t s) {
  cudaError_t e = launch_pdl(split_kernel<T, D>, a.n_work, kDecThreads, 0, s, a, pd.HL, pd.sl2);
  if (e == cudaSuccess)
    e = launch_pdl(combine_kernel<T, D>, cdiv(pd.G, 8), 256, 0, s, a, pd.G, pd.HL);
  return e;
}

}  // namespace

cudaError_t launch_decode(const ProfileDims& pd, const DecodeArgs& a, cudaStream_t s) {
  if (pd.dtype == FG_FP32)
    return pd.d == 64 ? run<float, 64>(pd, a, s) : run<float, 128>(pd, a, s);
  return pd.d == 64 ? run<__nv_bfloat16, 64>(pd, a, s) : run<__nv_bfloat16, 128>(pd, a, s);
}

}  // namespace fg
