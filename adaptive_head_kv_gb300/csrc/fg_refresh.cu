// Decode-time refresh of C_frequent from accumulated attention (an opt-in
// variant; Model Tells You What to Discard, Method: C_frequent keeps the
// tokens with the largest cumulative attention scores, and the stability
// paragraph examines accumulated attention at the prompt and at later
// decoding steps; the pages state no update rule, so the rule here is this
// library's own).
//
// State per pool row (caller-owned, fastgen_refresh_state_bytes):
//   acc  [pool_rows] f32: accumulated score of the row: its prompt column sum
//        at the end of the prompt (0 for a generated token), plus the
//        attention weight every later step's query gives it;
//   sc   [pool_rows] f32: the current step's score of the row (base-2
//        logit, -inf for rows not attended), written by the split kernel and
//        turned into acc += 2^(sc - M) / L after the combine (acc_kernel);
//   role [pool_rows] u8: 1 for the never-evicted slots that hold frequent
//        members, 0 otherwise.  Set once here; a refresh swaps rows between
//        a frequent slot and the window ring, so the slots keep their role;
//   ml   [G, 2] f32: each head's softmax maximum and sum of the step (written
//        by the combine kernel, read by the kernel that updates acc).
//
// Refresh of one local-hybrid cache (one CTA, after the step's combine):
//   candidates = the rows in frequent slots and the rows of the window ring;
//   the |F| candidates of largest (acc, -position) become the frequent
//   members; a member that lost its place moves to its window slot
//   (position mod w) if it is still inside the window, else it leaves; a
//   window row that won a place moves into a freed frequent slot and its
//   ring slot becomes empty.  Keys (acc bits, ~position) are unique, so the
//   outcome is the top-|F| set regardless of thread timing, and the slot
//   pairing follows a block scan in row order (deterministic layout).
#include "fg_common.cuh"
#include "fg_internal.h"

namespace fg {
namespace {

constexpr int kInitThreads = 256;
constexpr int kRefreshThreads = 1024;

__global__ void __launch_bounds__(kInitThreads) refresh_init_kernel(
    const fg_head_desc* __restrict__ desc, const int32_t* __restrict__ posp,
    const float* __restrict__ colsum, const int32_t* __restrict__ ids,
    const int32_t* __restrict__ special, int ns, const int32_t* __restrict__ punct, int np, int n,
    int HL, float* __restrict__ acc, uint8_t* __restrict__ role) {
  const int c = blockIdx.x;  // cache = head (no groups in refresh mode)
  const fg_head_desc hd = desc[c];
  const int b = c / HL;
  const bool uses_f = hd.policy == FG_POLICY_SPF || hd.policy == FG_POLICY_SPFL;
  const float* cs = colsum + (size_t)c * n;
  for (int r = threadIdx.x; r < hd.static_cap; r += blockDim.x) {
    const long long row = hd.off + r;
    const int p = posp[row];
    float a = 0.f;
    uint8_t f = 0;
    if (p >= 0 && p < n) {
      a = cs[p];
      const int tau = ids[(size_t)b * n + p];
      f = uses_f && !id_in(tau, special, ns) && !id_in(tau, punct, np);
    }
    acc[row] = a;
    role[row] = f;
  }
  for (int r = threadIdx.x; r < hd.w; r += blockDim.x) {
    const long long row = hd.win_off + r;
    const int p = posp[row];
    acc[row] = (p >= 0 && p < n) ? cs[p] : 0.f;
    role[row] = 0;
  }
}

// Sort key of a candidate: larger acc first, then the lower position.  acc is
// never negative, so its bit pattern orders like its value.
__device__ __forceinline__ unsigned long long cand_key(float a, int pos) {
  return ((unsigned long long)__float_as_uint(a) << 32) | (unsigned)(0xffffffffu - (unsigned)pos);
}

// Copies one pool row (K and V) from src to dst with the lanes of one warp.
template <typename T, int D>
__device__ __forceinline__ void copy_row(T* Kp, T* Vp, long long dst, long long src, int lane) {
  constexpr int E = Vec16<T>::kElems;
  constexpr int LPR = D / E;
  for (int v = lane; v < LPR; v += 32) {
    const size_t s = (size_t)src * D + v * E, d = (size_t)dst * D + v * E;
    const uint4 kv = *reinterpret_cast<const uint4*>(Kp + s);
    const uint4 vv = *reinterpret_cast<const uint4*>(Vp + s);
    *reinterpret_cast<uint4*>(Kp + d) = kv;
    *reinterpret_cast<uint4*>(Vp + d) = vv;
  }
}

// One CTA per cache.  `cap` is the size of the shared key array (a power of
// two >= k + w, which bounds the candidate count); t is the step's position.
template <typename T, int D>
__global__ void __launch_bounds__(kRefreshThreads) refresh_kernel(
    const fg_head_desc* __restrict__ desc, T* Kp, T* Vp, int32_t* posp, float* acc,
    const uint8_t* __restrict__ role, int t, int cap) {
  extern __shared__ unsigned long long keys[];
  __shared__ int scr[33];
  __shared__ int s_cnt, s_kf;
  griddep_wait();
  griddep_launch_dependents();
  fg_head_desc hd = desc[blockIdx.x];
  if (hd.policy != FG_POLICY_SPFL || hd.w <= 0) return;  // no window: nothing to promote
  // the row count that the step's combine advanced, read from L2: decode
  // kernels read descriptors before their wait, so a line in L1 may be older
  hd.n_static = __ldcg(&desc[blockIdx.x].n_static);
  if (threadIdx.x == 0) {
    s_cnt = 0;
    s_kf = 0;
  }
  __syncthreads();
  for (int r = threadIdx.x; r < hd.n_static; r += blockDim.x) {
    const long long row = hd.off + r;
    if (role[row]) {
      const int i = atomicAdd(&s_cnt, 1);
      atomicAdd(&s_kf, 1);
      if (i < cap) keys[i] = cand_key(acc[row], posp[row]);
    }
  }
  for (int r = threadIdx.x; r < hd.w; r += blockDim.x) {
    const long long row = hd.win_off + r;
    const int p = posp[row];
    if (p >= 0) {
      const int i = atomicAdd(&s_cnt, 1);
      if (i < cap) keys[i] = cand_key(acc[row], p);
    }
  }
  __syncthreads();
  const int cnt = s_cnt, kf = s_kf;
  if (kf == 0 || kf >= cnt || cnt > cap) return;  // no window candidate (or no room: unreachable)
  int P = 2;
  while (P < cnt) P <<= 1;
  for (int i = cnt + threadIdx.x; i < P; i += blockDim.x) keys[i] = 0ull;  // below every key
  __syncthreads();
  // bitonic sort, descending
  for (int size = 2; size <= P; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = threadIdx.x; i < P; i += blockDim.x) {
        const int j = i ^ stride;
        if (j > i) {
          const unsigned long long a = keys[i], b = keys[j];
          const bool down = (i & size) == 0;
          if (down ? (a < b) : (a > b)) {
            keys[i] = b;
            keys[j] = a;
          }
        }
      }
      __syncthreads();
    }
  }
  const unsigned long long thr = keys[kf - 1];  // the |F|-th largest key
  __syncthreads();
  // freed frequent slots (members that lost their place) and promoted ring
  // slots, each listed in row order; the key array's memory holds the lists
  int* freed = reinterpret_cast<int*>(keys);
  int* promoted = freed + cap;
  int n_freed = 0, n_prom = 0;
  for (int base = 0; base < hd.n_static; base += blockDim.x) {
    const int r = base + threadIdx.x;
    int lose = 0;
    if (r < hd.n_static) {
      const long long row = hd.off + r;
      lose = role[row] && cand_key(acc[row], posp[row]) < thr;
    }
    int tot;
    const int at = n_freed + block_exclusive_scan(lose, scr, &tot);
    if (lose) freed[at] = r;
    n_freed += tot;
  }
  for (int base = 0; base < hd.w; base += blockDim.x) {
    const int r = base + threadIdx.x;
    int win = 0;
    if (r < hd.w) {
      const long long row = hd.win_off + r;
      const int p = posp[row];
      win = p >= 0 && cand_key(acc[row], p) >= thr;
    }
    int tot;
    const int at = n_prom + block_exclusive_scan(win, scr, &tot);
    if (win) promoted[at] = r;
    n_prom += tot;
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nwarps = blockDim.x >> 5;
  // phase A: a member that lost its place but is still inside the window
  // (t - w, t] moves to its ring slot, which is empty while it is static
  for (int i = warp; i < n_freed; i += nwarps) {
    const long long row = hd.off + freed[i];
    const int p = posp[row];
    if (p > t - hd.w) {
      const long long dst = hd.win_off + p % hd.w;
      copy_row<T, D>(Kp, Vp, dst, row, lane);
      if (lane == 0) {
        posp[dst] = p;
        acc[dst] = acc[row];
      }
    }
  }
  __syncthreads();
  // phase B: promoted window rows take the freed slots; their ring slots empty
  const int pairs = min(n_freed, n_prom);  // equal: the top-|F| set has |F| rows
  for (int i = warp; i < pairs; i += nwarps) {
    const long long dst = hd.off + freed[i];
    const long long src = hd.win_off + promoted[i];
    copy_row<T, D>(Kp, Vp, dst, src, lane);
    if (lane == 0) {
      posp[dst] = posp[src];
      acc[dst] = acc[src];
      posp[src] = -1;
    }
  }
}

template <typename T, int D>
cudaError_t run_refresh(int caches, fg_head_desc* desc, void* Kp, void* Vp, int32_t* posp,
                        float* acc, const uint8_t* role, int t, int cap, cudaStream_t s) {
  const size_t smem = (size_t)cap * sizeof(unsigned long long);
  cudaError_t e = cudaFuncSetAttribute(refresh_kernel<T, D>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(refresh_kernel<T, D>, caches, kRefreshThreads, smem, s, desc, (T*)Kp,
                    (T*)Vp, posp, acc, role, t, cap);
}

}  // namespace

cudaError_t launch_refresh_init(const ProfileDims& pd, const fg_head_desc* desc,
                                const int32_t* posp, const float* colsum, const int32_t* ids,
                                const int32_t* special, int ns, const int32_t* punct, int np,
                                float* acc, uint8_t* role, cudaStream_t s) {
  refresh_init_kernel<<<pd.Gkv, kInitThreads, 0, s>>>(desc, posp, colsum, ids, special, ns,
                                                      punct, np, pd.n, pd.HL, acc, role);
  return cudaGetLastError();
}

cudaError_t launch_refresh(const ProfileDims& pd, fg_head_desc* desc, void* Kp, void* Vp,
                           int32_t* posp, float* acc, const uint8_t* role, int t, int cap,
                           cudaStream_t s) {
  if (pd.dtype == FG_FP32)
    return pd.d == 64 ? run_refresh<float, 64>(pd.Gkv, desc, Kp, Vp, posp, acc, role, t, cap, s)
                      : run_refresh<float, 128>(pd.Gkv, desc, Kp, Vp, posp, acc, role, t, cap, s);
  return pd.d == 64
             ? run_refresh<__nv_bfloat16, 64>(pd.Gkv, desc, Kp, Vp, posp, acc, role, t, cap, s)
             : run_refresh<__nv_bfloat16, 128>(pd.Gkv, desc, Kp, Vp, posp, acc, role, t, cap, s);
}

}  // namespace fg
