// Compaction: K_C, V_C = f(K, V, C) (Model Tells You What to Discard,
// Method, second paragraph) into one pooled, ragged, per-head layout.
//
// Pool layout of head g (rows of d elements, K and V pools share it):
//   [off, off + static_cap)        never-evicted segment: the kept static
//                                  prompt rows in position order, then room
//                                  for max_new_tokens appended rows;
//   [win_off, win_off + w)         SPFL heads only: the window ring, the row
//                                  of position t at slot t mod w.
// One cache per key/value head holds the union of its query heads' caches.
// The plan kernel lays caches out by an exclusive scan of their row counts
// and also emits the decode work list (one item per kRowsPerWork rows of the
// prompt's never-evicted rows, the last one also taking the rows appended
// while generating, plus one per kRowsPerWork rows of the ring).
#include "fg_common.cuh"
#include "fg_internal.h"

namespace fg {
namespace {

constexpr int kPlanThreads = 1024;
constexpr int kCompactThreads = 256;

// Union of a key/value head's members (query heads g0 .. g0 + R - 1): the
// group policy is the largest member policy (the placement rules are nested
// along the shortlist) and the never-evicted prompt set is the union of the
// members' (a position any member keeps so).
__device__ __forceinline__ int union_code(const uint8_t* __restrict__ keep, size_t g0, int R, int n,
                                          int j) {
  int any_static = 0, any_window = 0;
  for (int m = 0; m < R; ++m) {
    const int c = keep[(g0 + m) * (size_t)n + j];
    any_static |= c == FG_KEEP_STATIC;
    any_window |= c == FG_KEEP_WINDOW;
  }
  return any_static ? FG_KEEP_STATIC : (any_window ? FG_KEEP_WINDOW : FG_KEEP_DROP);
}

__global__ void __launch_bounds__(256) group_kernel(const int8_t* __restrict__ policy,
                                                    const uint8_t* __restrict__ keep, int n,
                                                    int H, int R, int2* __restrict__ cinfo) {
  __shared__ int red[8];
  const int c = blockIdx.x;
  const int Hkv = H / R;
  const size_t g0 = (size_t)(c / Hkv) * H + (size_t)(c % Hkv) * R;
  int cnt = 0;
  for (int j = threadIdx.x; j < n; j += blockDim.x)
    cnt += union_code(keep, g0, R, n, j) == FG_KEEP_STATIC;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = cnt;
  __syncthreads();
  if (threadIdx.x == 0) {
    int tot = 0, pol = 0;
    for (int i = 0; i < (int)(blockDim.x >> 5); ++i) tot += red[i];
    for (int m = 0; m < R; ++m) pol = max(pol, (int)policy[g0 + m]);
    cinfo[c] = make_int2(pol, tot);
  }
}

// Decode work items of a cache at `rpw` rows per item: the never-evicted
// segment's prompt rows (at least one item; the last one also takes the rows
// appended later) and the window ring.
__device__ __forceinline__ int cache_items(int n_static, int wg, int rpw) {
  return max(1, cdiv(n_static, rpw)) + cdiv(wg, rpw);
}

// Item size: kRowsPerWork, or kRowsPerWorkWide when the plan would have at
// least `wide_at` items at the small size (plenty of CTAs either way; the
// wide items halve the fixed cost per item).
__global__ void __launch_bounds__(kPlanThreads) plan_kernel(
    const int2* __restrict__ cinfo, int G, int w, int reserve, int wide_at,
    fg_head_desc* __restrict__ desc, long long* __restrict__ totals) {
  __shared__ long long scr64[33];
  __shared__ int scr32[33];
  int small_items = 0;
  for (int base = 0; base < G; base += blockDim.x) {
    const int g = base + threadIdx.x;
    int works = 0;
    if (g < G) {
      const int2 ci = cinfo[g];
      works = cache_items(ci.y, ci.x == FG_POLICY_SPFL ? w : 0, kRowsPerWork);
    }
    int wtot;
    block_exclusive_scan(works, scr32, &wtot);
    small_items += wtot;
  }
  const int rpw = small_items >= wide_at ? kRowsPerWorkWide : kRowsPerWork;
  long long row_base = 0;
  int work_base = 0;
  for (int base = 0; base < G; base += blockDim.x) {
    const int g = base + threadIdx.x;
    long long rows = 0;
    int works = 0, p = 0, n_static = 0, cap = 0, wg = 0;
    if (g < G) {
      const int2 ci = cinfo[g];
      p = ci.x;
      n_static = ci.y;
      cap = n_static + reserve;
      wg = (p == FG_POLICY_SPFL) ? w : 0;
      rows = (long long)cap + wg;
      works = cache_items(n_static, wg, rpw);
    }
    long long rtot;
    int wtot;
    const long long roff = row_base + block_exclusive_scan(rows, scr64, &rtot);
    const int woff = work_base + block_exclusive_scan(works, scr32, &wtot);
    if (g < G) {
      fg_head_desc hd;
      hd.off = roff;
      hd.n_static = n_static;
      hd.static_cap = cap;
      hd.win_off = roff + cap;
      hd.w = wg;
      hd.policy = p;
      hd.work_off = woff;
      hd.n_work = works;
      desc[g] = hd;
    }
    row_base += rtot;
    work_base += wtot;
  }
  if (threadIdx.x == 0) {
    totals[0] = row_base;
    totals[1] = work_base;
    totals[2] = rpw;
  }
}

__global__ void worklist_kernel(const fg_head_desc* __restrict__ desc, int G,
                                int2* __restrict__ work) {
  const int g = blockIdx.x * blockDim.x + threadIdx.x;
  if (g >= G) return;
  const fg_head_desc hd = desc[g];
  for (int i = 0; i < hd.n_work; ++i) work[hd.work_off + i] = make_int2(g, i);
}

// One CTA per (cache, chunk of `chunk` prompt positions): the CTA first
// counts the never-evicted rows before its chunk (their count is the first
// row it fills), then scans its positions in tiles of 256 and copies each
// tile's kept rows with 16-byte vectors, one row per LPR lanes.  A window
// position's ring slot (position mod w) is written by the CTA that owns the
// position: its position if the row lives in the window, else the empty
// marker; chunk 0 also marks the segment's reserve rows empty.
// Chunk length: 512 positions, or n / 8 for long prompts, so that a cache has
// at most eight chunks and the counting of earlier rows (linear in the
// chunk's start) stays a small part of the work.
constexpr int kCompactChunk = 512;
constexpr int kMaxCompactChunks = 8;
inline int compact_chunk(int n) {
  return max(kCompactChunk, cdiv(cdiv(n, kMaxCompactChunks), 256) * 256);
}

template <typename T, int D>
__global__ void __launch_bounds__(kCompactThreads) compact_kernel(
    const T* __restrict__ K, const T* __restrict__ V, const uint8_t* __restrict__ keep,
    const fg_head_desc* __restrict__ desc, int n, int chunk, int H, int R, T* __restrict__ Kp,
    T* __restrict__ Vp, int32_t* __restrict__ posp) {
  constexpr int E = Vec16<T>::kElems;
  constexpr int LPR = D / E;  // 16-byte vectors per row
  __shared__ int scr[33];
  __shared__ int src_pos[kCompactThreads];
  __shared__ long long dst_row[kCompactThreads];
  const int g = blockIdx.y;  // key/value head
  const int j0 = blockIdx.x * chunk, j1 = min(j0 + chunk, n);
  const fg_head_desc hd = desc[g];
  const int Hkv = H / R;
  const size_t g0 = (size_t)(g / Hkv) * H + (size_t)(g % Hkv) * R;  // its first query head
  if (blockIdx.x == 0)  // empty markers on the reserve rows of the segment
    for (int r = hd.n_static + threadIdx.x; r < hd.static_cap; r += blockDim.x)
      posp[hd.off + r] = -1;
  int before = 0;  // never-evicted rows at positions < j0
  for (int j = threadIdx.x; j < j0; j += blockDim.x)
    before += union_code(keep, g0, R, n, j) == FG_KEEP_STATIC ? 1 : 0;
  int static_seen;
  block_exclusive_scan(before, scr, &static_seen);
  const T* Kg = K + (size_t)g * n * D;
  const T* Vg = V + (size_t)g * n * D;
  for (int base = j0; base < j1; base += blockDim.x) {
    const int j = base + threadIdx.x;
    const int code = j < j1 ? union_code(keep, g0, R, n, j) : FG_KEEP_DROP;
    const int is_static = code == FG_KEEP_STATIC;
    const int is_kept = code != FG_KEEP_DROP;
    int st_total, kept_total;
    const int st_rank = static_seen + block_exclusive_scan(is_static, scr, &st_total);
    const int slot = block_exclusive_scan(is_kept, scr, &kept_total);
    if (hd.w > 0 && j < j1 && j >= n - hd.w && code != FG_KEEP_WINDOW)
      posp[hd.win_off + j % hd.w] = -1;  // a window position kept elsewhere (or not at all)
    if (is_kept) {
      long long dst;
      if (is_static) dst = hd.off + st_rank;
      else dst = hd.win_off + (hd.w > 0 ? j % hd.w : 0);
      posp[dst] = j;
      src_pos[slot] = j;
      dst_row[slot] = dst;
    }
    static_seen += st_total;
    __syncthreads();
#pragma unroll 4
    for (int v = threadIdx.x; v < kept_total * LPR; v += blockDim.x) {
      const int r = v / LPR, c = (v % LPR) * E;
      const size_t s = (size_t)src_pos[r] * D + c;
      const size_t d = (size_t)dst_row[r] * D + c;
      const uint4 kv = ldg_stream(Kg + s);
      const uint4 vv = ldg_stream(Vg + s);
      *reinterpret_cast<uint4*>(Kp + d) = kv;
      *reinterpret_cast<uint4*>(Vp + d) = vv;
    }
    __syncthreads();
  }
}

template <typename T, int D>
cudaError_t run_compact(const ProfileDims& pd, const void* K, const void* V, const uint8_t* keep,
                        const fg_head_desc* desc, void* Kp, void* Vp, int32_t* posp,
                        cudaStream_t s) {
  const int chunk = compact_chunk(pd.n);
  const dim3 grid(cdiv(pd.n, chunk), pd.Gkv);
  compact_kernel<T, D><<<grid, kCompactThreads, 0, s>>>((const T*)K, (const T*)V, keep, desc,
                                                        pd.n, chunk, pd.H, pd.R, (T*)Kp, (T*)Vp,
                                                        posp);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_group(const ProfileDims& pd, const int8_t* policy, const uint8_t* keep,
                         int2* cinfo, cudaStream_t s) {
  group_kernel<<<pd.Gkv, 256, 0, s>>>(policy, keep, pd.n, pd.H, pd.R, cinfo);
  return cudaGetLastError();
}

cudaError_t launch_plan(int Gkv, int w, int reserve, int wide_at, const int2* cinfo,
                        fg_head_desc* desc, int2* work, long long* totals, cudaStream_t s) {
  plan_kernel<<<1, kPlanThreads, 0, s>>>(cinfo, Gkv, w, reserve, wide_at, desc, totals);
  worklist_kernel<<<cdiv(Gkv, 256), 256, 0, s>>>(desc, Gkv, work);
  return cudaGetLastError();
}

cudaError_t launch_compact(const ProfileDims& pd, const void* K, const void* V,
                           const uint8_t* keep, const fg_head_desc* desc, void* Kp, void* Vp,
                           int32_t* posp, cudaStream_t s) {
  if (pd.dtype == FG_FP32)
    return pd.d == 64 ? run_compact<float, 64>(pd, K, V, keep, desc, Kp, Vp, posp, s)
                      : run_compact<float, 128>(pd, K, V, keep, desc, Kp, Vp, posp, s);
  return pd.d == 64 ? run_compact<__nv_bfloat16, 64>(pd, K, V, keep, desc, Kp, Vp, posp, s)
                    : run_compact<__nv_bfloat16, 128>(pd, K, V, keep, desc, Kp, Vp, posp, s);
}

}  // namespace fg
