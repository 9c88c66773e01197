// Prompt profiling in plain fp32 SIMT arithmetic: the path for fp32 inputs
// (the tensor cores' TF32 mode is too coarse for 1e-4 mass parity there).
//
// FastGen profiles each head on A = softmax(s Q K^T) under the causal mask
// (Model Tells You What to Discard, Method, eq. (C*)).  The map is never
// stored: pass 1 walks query tiles and keeps the running row maximum and
// sum (base-2 log-sum-exp per row); pass 2 walks key tiles, recomputes the
// scores and accumulates, per key j, colsum_j = sum_i A_ij and the band sum
// bandcol_j = sum_{j <= i < j+w} A_ij that the local-window mass needs.
#include "fg_common.cuh"
#include "fg_internal.h"

namespace fg {
namespace {

constexpr int kTile = 64;      // queries x keys per tile
constexpr int kThreads = 256;  // 16 x 16 threads, 4 x 4 scores each

// Loads rows [row0, row0 + 64) of one head's [n, D] matrix into smem as fp32
// (row stride D + 1), multiplied by `mul`; rows past n are zero.
template <typename T, int D>
__device__ __forceinline__ void load_tile(float* dst, const T* __restrict__ src, int row0, int n,
                                          float mul) {
  constexpr int E = Vec16<T>::kElems;
  constexpr int VPR = D / E;  // vectors per row
  for (int v = threadIdx.x; v < kTile * VPR; v += kThreads) {
    const int r = v / VPR, c = (v % VPR) * E;
    float f[E];
    if (row0 + r < n) {
      load16(src + (size_t)(row0 + r) * D + c, f);
    } else {
#pragma unroll
      for (int e = 0; e < E; ++e) f[e] = 0.f;
    }
#pragma unroll
    for (int e = 0; e < E; ++e) dst[r * (D + 1) + c + e] = f[e] * mul;
  }
}

// 4 x 4 block of dot products: rows a0..a0+3 of A against rows b0..b0+3 of B.
template <int D>
__device__ __forceinline__ void dot4x4(const float* A, int a0, const float* B, int b0,
                                       float (&s)[4][4]) {
#pragma unroll
  for (int r = 0; r < 4; ++r)
#pragma unroll
    for (int c = 0; c < 4; ++c) s[r][c] = 0.f;
#pragma unroll 8
  for (int k = 0; k < D; ++k) {
    float a[4], b[4];
#pragma unroll
    for (int r = 0; r < 4; ++r) a[r] = A[(a0 + r) * (D + 1) + k];
#pragma unroll
    for (int c = 0; c < 4; ++c) b[c] = B[(b0 + c) * (D + 1) + k];
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int c = 0; c < 4; ++c) s[r][c] = fmaf(a[r], b[c], s[r][c]);
  }
}

__device__ __forceinline__ float group16_max(float v) {
#pragma unroll
  for (int o = 1; o < 16; o <<= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float group16_sum(float v) {
#pragma unroll
  for (int o = 1; o < 16; o <<= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Pass 1: lse2[g, i] = -log2 sum_{j <= i} 2^(s log2e q_i.k_j) (negated row LSE).
template <typename T, int D>
__global__ void __launch_bounds__(kThreads) lse_kernel(const T* __restrict__ Q,
                                                       const T* __restrict__ K,
                                                       float* __restrict__ lse2, int n,
                                                       int ld, float sl2, int H, int R) {
  extern __shared__ float smem[];
  float* Qs = smem;
  float* Ks = smem + kTile * (D + 1);
  const int g = blockIdx.x, i0 = blockIdx.y * kTile;
  const T* Qg = Q + (size_t)g * n * D;
  const T* Kg = K + (size_t)kv_head(g, H, R) * n * D;  // the query head's key/value head
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  load_tile<T, D>(Qs, Qg, i0, n, sl2);
  float m[4], l[4];
#pragma unroll
  for (int r = 0; r < 4; ++r) { m[r] = FG_NEG_INF; l[r] = 0.f; }
  const int last = min(i0 + kTile, n) - 1;
  for (int j0 = 0; j0 <= last; j0 += kTile) {
    __syncthreads();
    load_tile<T, D>(Ks, Kg, j0, n, 1.f);
    __syncthreads();
    float s[4][4];
    dot4x4<D>(Qs, ty * 4, Ks, tx * 4, s);
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int i = i0 + ty * 4 + r;
      float mx = FG_NEG_INF;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int j = j0 + tx * 4 + c;
        if (j > i || j >= n) s[r][c] = FG_NEG_INF;
        mx = fmaxf(mx, s[r][c]);
      }
      mx = group16_max(mx);
      const float mnew = fmaxf(m[r], mx);
      float part = 0.f;
      if (mnew != FG_NEG_INF) {
#pragma unroll
        for (int c = 0; c < 4; ++c) part += exp2f(s[r][c] - mnew);
      }
      part = group16_sum(part);
      if (mnew != FG_NEG_INF) {
        l[r] = l[r] * exp2f(m[r] - mnew) + part;
        m[r] = mnew;
      }
    }
  }
  if (tx == 0) {
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int i = i0 + ty * 4 + r;
      if (i < n) lse2[(size_t)g * ld + i] = -(m[r] + log2f(l[r]));
    }
  }
}

// Pass 2: colsum[g, j] = sum_{i >= j} 2^(s'_ij + lse2_i), bandcol over i < j + w.
template <typename T, int D>
__global__ void __launch_bounds__(kThreads) colsum_kernel(const T* __restrict__ Q,
                                                          const T* __restrict__ K,
                                                          const float* __restrict__ lse2,
                                                          float* __restrict__ colsum,
                                                          float* __restrict__ bandcol, int n,
                                                          int ld, int w, float sl2, int H, int R) {
  extern __shared__ float smem[];
  float* Ks = smem;
  float* Qs = smem + kTile * (D + 1);
  float* Ls = Qs + kTile * (D + 1);
  const int g = blockIdx.x, j0 = blockIdx.y * kTile;
  const T* Qg = Q + (size_t)g * n * D;
  const T* Kg = K + (size_t)kv_head(g, H, R) * n * D;  // the query head's key/value head
  const float* Lg = lse2 + (size_t)g * ld;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  load_tile<T, D>(Ks, Kg, j0, n, 1.f);
  float cs[4] = {0.f, 0.f, 0.f, 0.f}, bs[4] = {0.f, 0.f, 0.f, 0.f};
  for (int i0 = j0; i0 < n; i0 += kTile) {
    __syncthreads();
    load_tile<T, D>(Qs, Qg, i0, n, sl2);
    if (threadIdx.x < kTile) Ls[threadIdx.x] = i0 + threadIdx.x < n ? Lg[i0 + threadIdx.x] : 0.f;
    __syncthreads();
    float s[4][4];
    dot4x4<D>(Ks, ty * 4, Qs, tx * 4, s);
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int j = j0 + ty * 4 + r;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int i = i0 + tx * 4 + c;
        if (i >= j && i < n) {
          const float p = exp2f(s[r][c] + Ls[tx * 4 + c]);
          cs[r] += p;
          if (i < j + w) bs[r] += p;
        }
      }
    }
  }
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const float c = group16_sum(cs[r]), b = group16_sum(bs[r]);
    const int j = j0 + ty * 4 + r;
    if (tx == 0 && j < n) {
      colsum[(size_t)g * n + j] = c;
      bandcol[(size_t)g * n + j] = b;
    }
  }
}

template <typename T, int D>
cudaError_t run(const ProfileDims& pd, const void* Q, const void* K, float* lse2, int ld,
                float* colsum, float* bandcol, cudaStream_t s) {
  const size_t sm1 = 2 * kTile * (D + 1) * sizeof(float);
  const size_t sm2 = sm1 + kTile * sizeof(float);
  cudaError_t e = cudaFuncSetAttribute(lse_kernel<T, D>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm1);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(colsum_kernel<T, D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)sm2);
  if (e != cudaSuccess) return e;
  dim3 grid(pd.G, cdiv(pd.n, kTile));
  lse_kernel<T, D><<<grid, kThreads, sm1, s>>>((const T*)Q, (const T*)K, lse2, pd.n, ld,
                                               pd.sl2, pd.H, pd.R);
  colsum_kernel<T, D><<<grid, kThreads, sm2, s>>>((const T*)Q, (const T*)K, lse2, colsum,
                                                  bandcol, pd.n, ld, pd.w, pd.sl2, pd.H, pd.R);
  return cudaGetLastError();
}

// Pass 3: out[g, i] = sum_{j <= i} 2^(s'_ij + lse2_i) v_j, one warp per query
// row (lanes split d), keys in order.
template <typename T, int D>
__global__ void __launch_bounds__(256) attn_kernel(const T* __restrict__ Q, const T* __restrict__ K,
                                                   const T* __restrict__ V,
                                                   const float* __restrict__ lse2, T* __restrict__ out,
                                                   int n, int ld, float sl2, int H, int R) {
  constexpr int E = D / 32;
  const int g = blockIdx.x, i = blockIdx.y * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (i >= n) return;
  const size_t kv = (size_t)kv_head(g, H, R) * n * D;
  float q[E], acc[E];
#pragma unroll
  for (int e = 0; e < E; ++e) {
    q[e] = to_f32(Q[((size_t)g * n + i) * D + lane * E + e]) * sl2;
    acc[e] = 0.f;
  }
  const float nl = lse2[(size_t)g * ld + i];
  for (int j = 0; j <= i; ++j) {
    float d = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) d = fmaf(q[e], to_f32(K[kv + (size_t)j * D + lane * E + e]), d);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) d += __shfl_xor_sync(0xffffffffu, d, o);
    const float p = exp2f(d + nl);
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] = fmaf(p, to_f32(V[kv + (size_t)j * D + lane * E + e]), acc[e]);
  }
#pragma unroll
  for (int e = 0; e < E; ++e) store_out(out + ((size_t)g * n + i) * D + lane * E + e, acc[e]);
}

template <typename T, int D>
cudaError_t run_attn(const ProfileDims& pd, const void* Q, const void* K, const void* V,
                     const float* lse2, int ld, void* out, cudaStream_t s) {
  dim3 grid(pd.G, cdiv(pd.n, 8));
  attn_kernel<T, D><<<grid, 256, 0, s>>>((const T*)Q, (const T*)K, (const T*)V, lse2, (T*)out,
                                         pd.n, ld, pd.sl2, pd.H, pd.R);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn_simt(const ProfileDims& pd, const void* Q, const void* K, const void* V,
                             const float* lse2, int ld, void* out, cudaStream_t s) {
  if (pd.dtype == FG_FP32)
    return pd.d == 64 ? run_attn<float, 64>(pd, Q, K, V, lse2, ld, out, s)
                      : run_attn<float, 128>(pd, Q, K, V, lse2, ld, out, s);
  return pd.d == 64 ? run_attn<__nv_bfloat16, 64>(pd, Q, K, V, lse2, ld, out, s)
                    : run_attn<__nv_bfloat16, 128>(pd, Q, K, V, lse2, ld, out, s);
}

cudaError_t launch_profile_simt(const ProfileDims& pd, const void* Q, const void* K, float* lse2,
                                int ld, float* colsum, float* bandcol, cudaStream_t s) {
  if (pd.dtype == FG_FP32)
    return pd.d == 64 ? run<float, 64>(pd, Q, K, lse2, ld, colsum, bandcol, s)
                      : run<float, 128>(pd, Q, K, lse2, ld, colsum, bandcol, s);
  return pd.d == 64 ? run<__nv_bfloat16, 64>(pd, Q, K, lse2, ld, colsum, bandcol, s)
                    : run<__nv_bfloat16, 128>(pd, Q, K, lse2, ld, colsum, bandcol, s);
}

}  // namespace fg
