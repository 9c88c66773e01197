// Launchers shared between the C-ABI translation unit and the kernel files.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "fastgen.h"

namespace fg {

// Decode work item: kRowsPerWork (or, in plans with many items,
// kRowsPerWorkWide) consecutive cache rows of one head; the last item of a
// never-evicted segment also covers the rows appended later.  Buffer sizes
// are bounded with kRowsPerWork, the smaller size.
constexpr int kRowsPerWork = 256;
constexpr int kRowsPerWorkWide = 512;

struct ProfileDims {
  int G, HL, B, n, d, dtype;
  int H, Hkv, R;   // heads and key/value heads per layer; group size R = H / Hkv
  int Gkv, HLkv;   // key/value head instances; L * Hkv
  int w, k;
  float T, sl2;  // sl2 = scale * log2(e): scores are kept in base-2 units
};

// Key/value head serving query head g.
__host__ __device__ inline int kv_head(int g, int H, int R) { return (g / H) * (H / R) + (g % H) / R; }

// Token class per prompt position: bit 0 special, bit 1 punctuation.  Also
// zeroes the work counters of the profiler passes (counters[0], [1] and [3],
// when non-null).
cudaError_t launch_token_class(const int32_t* ids, int count, const int32_t* special, int ns,
                               const int32_t* punct, int np, uint8_t* cls, int32_t* counters,
                               cudaStream_t s);

// Row stride of the lse2 workspace: n rounded up to whole 128-row tiles.
inline int lse_ld(int n) { return (n + 127) / 128 * 128; }

// Pass 1 (row log-sum-exp, base 2; lse2 rows of stride ld) and pass 2
// (column and band sums), plain SIMT fp32 arithmetic.
cudaError_t launch_profile_simt(const ProfileDims& pd, const void* Q, const void* K, float* lse2,
                                int ld, float* colsum, float* bandcol, cudaStream_t s);

// The same two passes on the tcgen05 tensor cores (bf16, d = 64 or 128).
// heads / n_heads (device): when heads is non-null only the *n_heads listed
// heads are profiled.  sched: two ints of scratch (the passes' work
// counters).  A device-side wait that times out ORs 2 into *err.
// stall_pass (1 or 2; 0 in normal use) keeps that pass's producer from
// starting, so its waits run out: a test of the error path.
bool profile_tc_supported(const ProfileDims& pd);
cudaError_t launch_profile_tc(const ProfileDims& pd, const void* Q, const void* K, float* lse2,
                              int ld, float* colsum, float* bandcol, const int32_t* heads,
                              const int32_t* n_heads, int32_t* sched, int32_t* err,
                              int stall_pass, cudaStream_t s);

// Pass 3: the prompt attention output out [G, n, d] = A V, from pass 1's
// negated base-2 row LSEs.  bf16 on the tensor cores (sched: one zeroed work
// counter; a timed-out wait ORs 2 into *err), fp32 on SIMT lanes.
cudaError_t launch_attn_tc(const ProfileDims& pd, const void* Q, const void* K, const void* V,
                           const float* lse2, int ld, void* out, int32_t* sched, int32_t* err,
                           cudaStream_t s);
cudaError_t launch_attn_simt(const ProfileDims& pd, const void* Q, const void* K, const void* V,
                             const float* lse2, int ld, void* out, cudaStream_t s);

// Heads whose saved policy contains C_frequent, and their count.
cudaError_t launch_head_list(const int8_t* fixed, int G, int32_t* heads, int32_t* count,
                             cudaStream_t s);

// Top-k frequent set, candidate masses, policy, keep codes.  With `fixed`
// (a saved policy per head) the saved entry is used: mass, cost and policy
// are not written, and an out-of-range saved value ORs 4 into *err.
cudaError_t launch_select(const ProfileDims& pd, const float* colsum, const float* bandcol,
                          const uint8_t* cls, const int8_t* fixed, int8_t* policy, float* mass,
                          int32_t* cost, uint8_t* keep, int32_t* kept, int32_t* err,
                          cudaStream_t s);

// Per key/value head c: the group policy (largest member policy) and the size
// of the union of the members' never-evicted prompt sets, as int2 cinfo[c].
cudaError_t launch_group(const ProfileDims& pd, const int8_t* policy, const uint8_t* keep,
                         int2* cinfo, cudaStream_t s);

// Writes one descriptor per cache from cinfo and builds the decode work list
// (every cache gets at least one item).
// Item size: kRowsPerWorkWide when the plan has >= wide_at items at
// kRowsPerWork; totals = {pool rows, items, rows per item}.
cudaError_t launch_plan(int Gkv, int w, int reserve, int wide_at, const int2* cinfo,
                        fg_head_desc* desc, int2* work, long long* totals, cudaStream_t s);

cudaError_t launch_compact(const ProfileDims& pd, const void* K, const void* V,
                           const uint8_t* keep, const fg_head_desc* desc, void* Kp, void* Vp,
                           int32_t* posp, cudaStream_t s);

struct DecodeArgs {
  fg_head_desc* desc;  // per cache (key/value head)
  const int2* work;
  int n_work;
  void* Kp;
  void* Vp;
  int32_t* posp;
  const void* q;
  const void* k_new;
  const void* v_new;
  const int32_t* new_ids;
  const int32_t* special;
  int ns;
  const int32_t* punct;
  int np;
  int pos;
  int rpw;  // rows per work item of the plan
  void* out;
  float* part_ml;   // [n_work, R, 2]
  float* part_acc;  // [n_work, R, d]
  int32_t* dev_err;
  // accumulated attention of every pool row (refresh of C_frequent; no groups):
  // when non-null the split kernel writes each row's score to row_sc, the
  // combine each head's final (M, L) to head_ml, and a third kernel adds each
  // row's weight to row_acc
  float* row_acc = nullptr;
  float* row_sc = nullptr;
  float* head_ml = nullptr;  // [G, 2]: each head's final (M, L) of the step
};

cudaError_t launch_decode(const ProfileDims& pd, const DecodeArgs& a, cudaStream_t s);

// Refresh of C_frequent (opt-in).  Init: per pool row, acc = the prompt column
// sum of its position (0 for empty rows) and role = 1 for never-evicted rows
// kept for frequency.  Refresh: one CTA per cache re-chooses the frequent
// members among them and the window rows (cap: shared key slots, a power of
// two >= k + w; t: the step's position).
constexpr int kRefreshMaxCandidates = 16384;
cudaError_t launch_refresh_init(const ProfileDims& pd, const fg_head_desc* desc,
                                const int32_t* posp, const float* colsum, const int32_t* ids,
                                const int32_t* special, int ns, const int32_t* punct, int np,
                                float* acc, uint8_t* role, cudaStream_t s);
cudaError_t launch_refresh(const ProfileDims& pd, fg_head_desc* desc, void* Kp, void* Vp,
                           int32_t* posp, float* acc, const uint8_t* role, int t, int cap,
                           cudaStream_t s);

}  // namespace fg
