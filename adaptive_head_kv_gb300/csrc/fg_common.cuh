// Device helpers shared by the FastGen kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "fastgen.h"

namespace fg {

constexpr float kLog2e = 1.4426950408889634f;
#define FG_NEG_INF (-__int_as_float(0x7f800000))

__host__ __device__ inline int cdiv(int a, int b) { return (a + b - 1) / b; }

// Elements of T held by one 16-byte vector.
template <typename T>
struct Vec16 {
  static constexpr int kElems = 16 / sizeof(T);
};

// bf16 -> fp32 is exact: the bf16 bits are the high half of the fp32 word.
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ void unpack16(const uint4& v, float* f, const float*) {
  f[0] = __uint_as_float(v.x);
  f[1] = __uint_as_float(v.y);
  f[2] = __uint_as_float(v.z);
  f[3] = __uint_as_float(v.w);
}

__device__ __forceinline__ void unpack16(const uint4& v, float* f, const __nv_bfloat16*) {
  f[0] = bf16_lo(v.x); f[1] = bf16_hi(v.x);
  f[2] = bf16_lo(v.y); f[3] = bf16_hi(v.y);
  f[4] = bf16_lo(v.z); f[5] = bf16_hi(v.z);
  f[6] = bf16_lo(v.w); f[7] = bf16_hi(v.w);
}

// Loads 16 bytes of T and widens them to fp32.
template <typename T>
__device__ __forceinline__ void load16(const T* p, float* f) {
  uint4 v = *reinterpret_cast<const uint4*>(p);
  unpack16(v, f, p);
}

// Streaming 16-byte load that does not allocate in L1.
__device__ __forceinline__ uint4 ldg_stream(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

__device__ __forceinline__ void store_out(float* p, float v) { *p = v; }
__device__ __forceinline__ void store_out(__nv_bfloat16* p, float v) { *p = __float2bfloat16_rn(v); }

// Is `id` one of the `cnt` ids of `set`?  The sets are small (special and
// punctuation ids), so a linear scan through the read-only cache is enough.
__device__ __forceinline__ bool id_in(int id, const int32_t* __restrict__ set, int cnt) {
  for (int i = 0; i < cnt; ++i)
    if (__ldg(set + i) == id) return true;
  return false;
}

// Placement rule of a generated token for a head with policy `p`: does it
// join the never-evicted segment?
__device__ __forceinline__ bool joins_static(int p, bool is_special, bool is_punct) {
  if (p == FG_POLICY_FULL) return true;
  if (p == FG_POLICY_S) return is_special;
  return is_special || is_punct;
}

// Block-wide exclusive scan (blockDim.x a multiple of 32, <= 1024).
// `scratch` must hold 33 values.  Returns the exclusive prefix; *total gets
// the block sum.  Contains __syncthreads(): call from every thread.
template <typename I>
__device__ __forceinline__ I block_exclusive_scan(I x, I* scratch, I* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nwarps = blockDim.x >> 5;
  I v = x;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    I y = __shfl_up_sync(0xffffffffu, v, off);
    if (lane >= off) v += y;
  }
  if (lane == 31) scratch[warp] = v;
  __syncthreads();
  if (warp == 0) {
    I s = lane < nwarps ? scratch[lane] : I(0);
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      I y = __shfl_up_sync(0xffffffffu, s, off);
      if (lane >= off) s += y;
    }
    if (lane < nwarps) scratch[lane] = s;  // inclusive warp totals
    if (lane == 31) scratch[32] = s;
  }
  __syncthreads();
  I before = warp > 0 ? scratch[warp - 1] : I(0);
  *total = scratch[32];
  I r = before + v - x;
  __syncthreads();
  return r;
}

// Launches `kernel` as a programmatic dependent of the kernel before it in
// the stream: its CTAs may be scheduled while that kernel finishes, so they
// must execute griddep_wait() before touching memory the previous kernels
// write (the wait returns once those kernels have completed and their
// writes are visible).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), unsigned grid, unsigned block,
                              size_t smem, cudaStream_t s, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;");
}

}  // namespace fg
