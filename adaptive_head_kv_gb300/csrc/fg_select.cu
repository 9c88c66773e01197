// Policy selection per head (Model Tells You What to Discard, Method:
// base policies, shortlist and eq. (C*)).
//
// One CTA per head.  From the column sums of the attention map it
//   1. picks C_frequent = the k keys of largest colsum (ties to the lower
//      index) by an MSB-first radix select on the fp32 bit patterns (colsum
//      >= 0, so unsigned order is value order);
//   2. forms the four candidate masses from column sums alone:
//        mass_p = sum_{j in K^p} colsum_j / n                    (p <= 2)
//        mass_3 = [sum_j bandcol_j + sum_{j in K^2} (colsum_j - bandcol_j)] / n
//      which equals the per-row mean of the kept attention (the local set of
//      row i, {i-w < j <= i}, contributes band sums column by column);
//   3. takes the first shortlist entry with mass >= T (the cheapest, as the
//      entries are nested) and writes the keep codes of its final cache.
// With a saved head-policy map (`fixed`), step 3 takes the head's saved
// entry instead: no masses are formed, and the top-k select runs only for
// entries containing C_frequent (the only heads the profiler scored).
#include "fg_common.cuh"
#include "fg_internal.h"

namespace fg {
namespace {

constexpr int kSelThreads = 256;
constexpr int kSmemN = 8192;  // longest prompt whose column sums are staged in shared memory

__global__ void token_class_kernel(const int32_t* __restrict__ ids, int count,
                                   const int32_t* __restrict__ special, int ns,
                                   const int32_t* __restrict__ punct, int np,
                                   uint8_t* __restrict__ cls, int32_t* __restrict__ counters) {
  griddep_wait();
  griddep_launch_dependents();
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i == 0 && counters) counters[0] = counters[1] = counters[3] = 0;  // passes' work counters
  if (i >= count) return;
  const int id = ids[i];
  cls[i] = (uint8_t)((id_in(id, special, ns) ? 1 : 0) | (id_in(id, punct, np) ? 2 : 0));
}

// Membership bits kept in `keep` between the two sweeps: 1 = K^0,
// 2 = K^1, 4 = K^2, 8 = inside the last-w window.
__global__ void __launch_bounds__(kSelThreads) select_kernel(
    const float* __restrict__ colsum, const float* __restrict__ bandcol,
    const uint8_t* __restrict__ cls, int n, int HL, int k, int w, float T,
    const int8_t* __restrict__ fixed, int8_t* __restrict__ policy, float* __restrict__ mass,
    int32_t* __restrict__ cost, uint8_t* __restrict__ keep, int32_t* __restrict__ kept,
    int32_t* __restrict__ err) {
  extern __shared__ float cs_smem[];  // the head's colsum when it fits (n <= kSmemN)
  __shared__ unsigned hist[256];
  __shared__ int s_bin, s_krem, s_eq;
  __shared__ int scan_scratch[33];
  __shared__ double sred_a[kSelThreads / 32][4];
  __shared__ int sred_c[kSelThreads / 32][4];
  __shared__ int s_policy;

  griddep_wait();
  griddep_launch_dependents();
  const int g = blockIdx.x;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  // saved entry of this head (an out-of-range value is recorded and read as full)
  int saved = -1;
  if (fixed) {
    saved = fixed[g];
    if (saved < FG_POLICY_S || saved > FG_POLICY_FULL) {
      if (threadIdx.x == 0) atomicOr(err, 4);
      saved = FG_POLICY_FULL;
    }
  }
  const bool need_f = !fixed || saved == FG_POLICY_SPF || saved == FG_POLICY_SPFL;
  const float* c = colsum + (size_t)g * n;
  if (need_f && n <= kSmemN) {  // read the head's column sums once
    for (int j = threadIdx.x; j < n; j += blockDim.x) cs_smem[j] = c[j];
    __syncthreads();
    c = cs_smem;
  }
  const float* bc = bandcol + (size_t)g * n;
  const uint8_t* cl = cls + (size_t)(g / HL) * n;
  uint8_t* kp = keep + (size_t)g * n;
  const bool partial = need_f && k > 0 && k < n;

  // --- 1. radix select of the k-th largest colsum (8-bit digits, MSB first)
  unsigned prefix = 0, mask = 0;
  int krem = k, eq_count = 0;
  if (partial) {
    for (int shift = 24; shift >= 0; shift -= 8) {
      for (int b = threadIdx.x; b < 256; b += blockDim.x) hist[b] = 0;
      __syncthreads();
      for (int j = threadIdx.x; j < n; j += blockDim.x) {
        const unsigned u = __float_as_uint(c[j]);
        if ((u & mask) == prefix) atomicAdd(&hist[(u >> shift) & 255u], 1u);
      }
      __syncthreads();
      if (warp == 0) {
        // lane l owns bins 255-8l .. 248-8l, scanned from the top down
        unsigned h[8], tot = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          h[i] = hist[255 - 8 * lane - i];
          tot += h[i];
        }
        unsigned incl = tot;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const unsigned y = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += y;
        }
        const unsigned hit = __ballot_sync(0xffffffffu, incl >= (unsigned)krem);
        const int L = hit ? __ffs(hit) - 1 : 31;
        if (lane == L) {
          unsigned acc = incl - tot;
          int i = 0;
          for (; i < 7; ++i) {
            if (acc + h[i] >= (unsigned)krem) break;
            acc += h[i];
          }
          s_bin = 255 - 8 * lane - i;
          s_krem = krem - (int)acc;
          s_eq = (int)h[i];
        }
      }
      __syncthreads();
      prefix |= (unsigned)s_bin << shift;
      mask |= 255u << shift;
      krem = s_krem;
      eq_count = s_eq;  // after the last digit: values equal to the threshold
    }
  }
  // Selected: value above the threshold, or equal to it and among the first
  // `krem` equal values in index order (all of them when krem covers them).
  const unsigned thr = prefix;
  const bool rank_ties = partial && krem < eq_count;

  // --- 2. masses and costs --------------------------------------------------
  double a0 = 0, a1 = 0, a2 = 0, a3 = 0;
  int c0 = 0, c1 = 0, c2 = 0, c3 = 0;
  int eq_seen = 0;
  for (int base = 0; base < n; base += blockDim.x) {
    const int j = base + threadIdx.x;
    const bool valid = j < n;
    const float cj = valid && need_f ? c[j] : 0.f;
    const unsigned u = __float_as_uint(cj);
    const int is_eq = (valid && partial && u == thr) ? 1 : 0;
    int eq_rank = 0;
    if (rank_ties) {  // block-uniform branch
      int eq_total;
      eq_rank = eq_seen + block_exclusive_scan(is_eq, scan_scratch, &eq_total);
      eq_seen += eq_total;
    }
    if (!valid) continue;
    bool in_f;
    if (!need_f || k == 0) in_f = false;
    else if (k >= n) in_f = true;
    else in_f = (u > thr) || (is_eq && (!rank_ties || eq_rank < krem));
    const uint8_t t = cl[j];
    const bool s0 = t & 1, s1 = t != 0, s2 = s1 || in_f, win = j >= n - w;
    const float bj = fixed ? 0.f : bc[j];
    if (s0) { a0 += cj; ++c0; }
    if (s1) { a1 += cj; ++c1; }
    if (s2) { a2 += cj; a3 += (double)cj - (double)bj; ++c2; }
    a3 += bj;
    if (s2 || win) ++c3;
    kp[j] = (uint8_t)((s0 ? 1 : 0) | (s1 ? 2 : 0) | (s2 ? 4 : 0) | (win ? 8 : 0));
  }
  // the eight sums at once: warp shuffles, then one pass over the warps
  {
    double av[4] = {a0, a1, a2, a3};
    int cv[4] = {c0, c1, c2, c3};
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        av[q] += __shfl_xor_sync(0xffffffffu, av[q], o);
        cv[q] += __shfl_xor_sync(0xffffffffu, cv[q], o);
      }
    if (lane == 0)
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        sred_a[warp][q] = av[q];
        sred_c[warp][q] = cv[q];
      }
    __syncthreads();
    if (threadIdx.x == 0) {
      a0 = a1 = a2 = a3 = 0.0;
      c0 = c1 = c2 = c3 = 0;
      for (int w = 0; w < kSelThreads / 32; ++w) {
        a0 += sred_a[w][0]; a1 += sred_a[w][1]; a2 += sred_a[w][2]; a3 += sred_a[w][3];
        c0 += sred_c[w][0]; c1 += sred_c[w][1]; c2 += sred_c[w][2]; c3 += sred_c[w][3];
      }
    }
  }
  if (threadIdx.x == 0) {
    const double inv = 1.0 / (double)n;
    const double m[5] = {a0 * inv, a1 * inv, a2 * inv, a3 * inv, 1.0};
    const int cs[5] = {c0, c1, c2, c3, n};
    int p = 4;
    if (fixed) {
      p = saved;
    } else {
      for (int q = 0; q < 4; ++q)
        if (m[q] >= (double)T) { p = q; break; }
      for (int q = 0; q < 5; ++q) {
        mass[(size_t)g * 5 + q] = (float)m[q];
        cost[(size_t)g * 5 + q] = cs[q];
      }
      policy[g] = (int8_t)p;
    }
    kept[g] = cs[p];
    s_policy = p;
  }
  __syncthreads();

  // --- 3. keep codes of the chosen policy ----------------------------------
  const int p = s_policy;
  for (int j = threadIdx.x; j < n; j += blockDim.x) {
    const uint8_t bits = kp[j];
    uint8_t code;
    switch (p) {
      case FG_POLICY_S: code = (bits & 1) ? FG_KEEP_STATIC : FG_KEEP_DROP; break;
      case FG_POLICY_SP: code = (bits & 2) ? FG_KEEP_STATIC : FG_KEEP_DROP; break;
      case FG_POLICY_SPF: code = (bits & 4) ? FG_KEEP_STATIC : FG_KEEP_DROP; break;
      case FG_POLICY_SPFL:
        code = (bits & 4) ? FG_KEEP_STATIC : ((bits & 8) ? FG_KEEP_WINDOW : FG_KEEP_DROP);
        break;
      default: code = FG_KEEP_STATIC;
    }
    kp[j] = code;
  }
}

// Heads whose saved entry contains C_frequent (the only ones the profiler
// scores under a saved map), in increasing order, and their count.  One CTA.
__global__ void __launch_bounds__(1024) head_list_kernel(const int8_t* __restrict__ fixed, int G,
                                                         int32_t* __restrict__ heads,
                                                         int32_t* __restrict__ count) {
  __shared__ int scratch[33];
  griddep_wait();
  griddep_launch_dependents();
  int base = 0;
  for (int g0 = 0; g0 < G; g0 += blockDim.x) {
    const int g = g0 + threadIdx.x;
    const int p = g < G ? fixed[g] : -1;
    const int f = (p == FG_POLICY_SPF || p == FG_POLICY_SPFL) ? 1 : 0;
    int total;
    const int at = base + block_exclusive_scan(f, scratch, &total);
    if (f) heads[at] = g;
    base += total;
  }
  if (threadIdx.x == 0) *count = base;
}

}  // namespace

cudaError_t launch_head_list(const int8_t* fixed, int G, int32_t* heads, int32_t* count,
                             cudaStream_t s) {
  return launch_pdl(head_list_kernel, 1, 1024, 0, s, fixed, G, heads, count);
}

cudaError_t launch_token_class(const int32_t* ids, int count, const int32_t* special, int ns,
                               const int32_t* punct, int np, uint8_t* cls, int32_t* counters,
                               cudaStream_t s) {
  return launch_pdl(token_class_kernel, cdiv(count, 256), 256, 0, s, ids, count, special, ns,
                    punct, np, cls, counters);
}

cudaError_t launch_select(const ProfileDims& pd, const float* colsum, const float* bandcol,
                          const uint8_t* cls, const int8_t* fixed, int8_t* policy, float* mass,
                          int32_t* cost, uint8_t* keep, int32_t* kept, int32_t* err,
                          cudaStream_t s) {
  const size_t smem = pd.n <= kSmemN ? (size_t)pd.n * sizeof(float) : 0;
  if (smem > 48 * 1024) {
    const cudaError_t e = cudaFuncSetAttribute(
        select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  return launch_pdl(select_kernel, pd.G, kSelThreads, smem, s, colsum, bandcol, cls, pd.n, pd.HL,
                    pd.k, pd.w, pd.T, fixed, policy, mass, cost, keep, kept, err);
}

}  // namespace fg
