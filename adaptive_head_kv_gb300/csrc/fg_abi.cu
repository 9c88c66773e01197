// C ABI of the FastGen hot path: argument checks, workspace carving and the
// launch sequence of each call.  All memory belongs to the caller.
#include <math.h>
#include <stdint.h>

#include "fg_common.cuh"
#include "fg_internal.h"

namespace {

using fg::cdiv;

constexpr size_t kAlign = 256;
constexpr int kMaxIdSet = 4096;

size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }
bool aligned(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }

int ratio_count(float r, int n) { return (int)ceil((double)r * (double)n); }

fg_status check_params(const fg_params* p) {
  if (!p) return FG_EINVAL;
  if (p->B < 1 || p->L < 1 || p->H < 1 || p->n < 1) return FG_EINVAL;
  const long long G = (long long)p->B * p->L * p->H;
  if (G > 0x7fffffffLL || (long long)G * p->n > (1LL << 40)) return FG_EINVAL;
  if (p->d != 64 && p->d != 128) return FG_EDTYPE;
  if (p->dtype != FG_BF16 && p->dtype != FG_FP32) return FG_EDTYPE;
  if (!(p->T > 0.f && p->T <= 1.f)) return FG_EINVAL;
  if (!(p->r_l >= 0.f && p->r_l <= 1.f) || !(p->r_f >= 0.f && p->r_f <= 1.f)) return FG_EINVAL;
  if (!(p->scale >= 0.f) || isinf(p->scale)) return FG_EINVAL;
  if (p->Hkv < 0 || (p->Hkv > 0 && p->H % p->Hkv != 0)) return FG_EINVAL;
  const int R = p->Hkv > 0 ? p->H / p->Hkv : 1;
  if (R != 1 && R != 2 && R != 4 && R != 8) return FG_EDTYPE;
  return FG_OK;
}

fg::ProfileDims dims(const fg_params* p) {
  fg::ProfileDims pd;
  pd.B = p->B;
  pd.HL = p->L * p->H;
  pd.G = p->B * pd.HL;
  pd.H = p->H;
  pd.Hkv = p->Hkv > 0 ? p->Hkv : p->H;
  pd.R = p->H / pd.Hkv;
  pd.HLkv = p->L * pd.Hkv;
  pd.Gkv = p->B * pd.HLkv;
  pd.n = p->n;
  pd.d = p->d;
  pd.dtype = p->dtype;
  pd.w = ratio_count(p->r_l, p->n);
  pd.k = ratio_count(p->r_f, p->n);
  pd.T = p->T;
  const float s = p->scale > 0.f ? p->scale : (float)(1.0 / sqrt((double)p->d));
  pd.sl2 = s * fg::kLog2e;
  return pd;
}

fg_status check_ids(const int32_t* set, int32_t cnt) {
  if (cnt < 0 || cnt > kMaxIdSet) return FG_EINVAL;
  if (cnt > 0 && !set) return FG_EINVAL;
  return FG_OK;
}

fg_status cuda_status(cudaError_t e) { return e == cudaSuccess ? FG_OK : FG_ECUDA; }

size_t elem_bytes(const fg_params* p) { return p->dtype == FG_BF16 ? 2 : 4; }

// plan buffer: [Gkv descriptors][Gkv x int2 group info][2 x int64 totals][work list]
size_t plan_desc_bytes(int Gkv) { return align_up((size_t)Gkv * sizeof(fg_head_desc)); }
size_t plan_cinfo_bytes(int Gkv) { return align_up((size_t)Gkv * sizeof(int2)); }
size_t plan_work_offset(int Gkv) { return plan_desc_bytes(Gkv) + plan_cinfo_bytes(Gkv) + kAlign; }
int kv_count(const fg_params* p) { return p->B * p->L * (p->Hkv > 0 ? p->Hkv : p->H); }
int group_size(const fg_params* p) { return p->Hkv > 0 ? p->H / p->Hkv : 1; }
size_t plan_max_work(const fg_params* p, int32_t max_new) {
  const size_t Gkv = (size_t)kv_count(p);
  const int w = ratio_count(p->r_l, p->n);
  return Gkv * (size_t)(cdiv(p->n + max_new, fg::kRowsPerWork) + cdiv(w, fg::kRowsPerWork));
}

}  // namespace

extern "C" {

const char* fastgen_status_string(fg_status s) {
  switch (s) {
    case FG_OK: return "ok";
    case FG_EINVAL: return "invalid argument";
    case FG_EDTYPE: return "unsupported dtype or head dim";
    case FG_EWORKSPACE: return "workspace, plan or pool buffer too small";
    case FG_ECAPACITY: return "a head ran out of reserved cache rows";
    case FG_ECUDA: return "CUDA error";
    case FG_EDEVICE: return "a device-side wait timed out; results of that call are invalid";
  }
  return "unknown status";
}

int32_t fastgen_version(void) { return 100; }

size_t fastgen_profile_workspace_bytes(const fg_params* p) {
  if (check_params(p) != FG_OK) return 0;
  const size_t G = (size_t)p->B * p->L * p->H, n = p->n;
  return align_up(G * fg::lse_ld(p->n) * sizeof(float)) + align_up(G * n * sizeof(float)) +
         align_up((size_t)p->B * n) + kAlign + align_up(G * sizeof(int32_t));
}

// Shared by fastgen_profile (fixed == NULL), fastgen_profile_with_policy and
// fastgen_profile_attn (V and out non-NULL: the prompt attention output too).
static fg_status profile_call(const fg_params* p, const void* Q, const void* K, const void* V,
                              void* out, const int32_t* token_ids, const int32_t* special_ids,
                              int32_t n_special, const int32_t* punct_ids, int32_t n_punct,
                              const int8_t* fixed, int8_t* policy, float* mass, int32_t* cost,
                              float* colsum, uint8_t* keep, int32_t* kept, void* workspace,
                              size_t workspace_bytes, int32_t* dev_err, void* stream,
                              int stall_pass = 0) {
  fg_status st = check_params(p);
  if (st != FG_OK) return st;
  if ((st = check_ids(special_ids, n_special)) != FG_OK) return st;
  if ((st = check_ids(punct_ids, n_punct)) != FG_OK) return st;
  if (!Q || !K || !token_ids || !colsum || !keep || !kept || !workspace || !dev_err)
    return FG_EINVAL;
  if (!fixed && (!policy || !mass || !cost)) return FG_EINVAL;
  if ((V == nullptr) != (out == nullptr)) return FG_EINVAL;
  if (V && (!aligned(V, 16) || !aligned(out, 16))) return FG_EINVAL;
  if (!aligned(Q, 16) || !aligned(K, 16) || !aligned(workspace, kAlign) ||
      !aligned(colsum, 4) || !aligned(kept, 4) || !aligned(token_ids, 4) ||
      !aligned(dev_err, 4) || (!fixed && (!aligned(mass, 4) || !aligned(cost, 4))))
    return FG_EINVAL;
  if (workspace_bytes < fastgen_profile_workspace_bytes(p)) return FG_EWORKSPACE;
  const fg::ProfileDims pd = dims(p);
  const size_t Gn = (size_t)pd.G * pd.n;
  const int ld = fg::lse_ld(pd.n);
  // workspace: [lse2 G x ld][bandcol G x n][token classes B x n][256: counters][head list G]
  char* ws = (char*)workspace;
  float* lse2 = (float*)ws;
  size_t off = align_up((size_t)pd.G * ld * sizeof(float));
  float* bandcol = (float*)(ws + off);
  off += align_up(Gn * sizeof(float));
  uint8_t* cls = (uint8_t*)(ws + off);
  off += align_up((size_t)pd.B * pd.n);
  int32_t* sched = (int32_t*)(ws + off);  // [0], [1] zeroed by the class kernel; [2] head count
  off += kAlign;
  int32_t* heads = (int32_t*)(ws + off);
  cudaStream_t s = (cudaStream_t)stream;
  cudaError_t e = fg::launch_token_class(token_ids, pd.B * pd.n, special_ids, n_special,
                                         punct_ids, n_punct, cls, sched, s);
  const bool tc = fg::profile_tc_supported(pd);
  if (e == cudaSuccess && fixed && tc) e = fg::launch_head_list(fixed, pd.G, heads, sched + 2, s);
  if (e == cudaSuccess) {
    if (tc)
      e = fg::launch_profile_tc(pd, Q, K, lse2, ld, colsum, bandcol, fixed ? heads : nullptr,
                                fixed ? sched + 2 : nullptr, sched, dev_err, stall_pass, s);
    else  // the fp32 path scores every head
      e = fg::launch_profile_simt(pd, Q, K, lse2, ld, colsum, bandcol, s);
  }
  if (e == cudaSuccess && V)
    e = tc ? fg::launch_attn_tc(pd, Q, K, V, lse2, ld, out, sched + 3, dev_err, s)
           : fg::launch_attn_simt(pd, Q, K, V, lse2, ld, out, s);
  if (e == cudaSuccess)
    e = fg::launch_select(pd, colsum, bandcol, cls, fixed, policy, mass, cost, keep, kept,
                          dev_err, s);
  return cuda_status(e);
}

fg_status fastgen_profile(const fg_params* p, const void* Q, const void* K,
                          const int32_t* token_ids, const int32_t* special_ids,
                          int32_t n_special, const int32_t* punct_ids, int32_t n_punct,
                          int8_t* policy, float* mass, int32_t* cost, float* colsum,
                          uint8_t* keep, int32_t* kept, void* workspace,
                          size_t workspace_bytes, int32_t* dev_err, void* stream) {
  return profile_call(p, Q, K, nullptr, nullptr, token_ids, special_ids, n_special, punct_ids,
                      n_punct, nullptr, policy, mass, cost, colsum, keep, kept, workspace,
                      workspace_bytes, dev_err, stream);
}

fg_status fastgen_profile_attn(const fg_params* p, const void* Q, const void* K, const void* V,
                               const int32_t* token_ids, const int32_t* special_ids,
                               int32_t n_special, const int32_t* punct_ids, int32_t n_punct,
                               int8_t* policy, float* mass, int32_t* cost, float* colsum,
                               uint8_t* keep, int32_t* kept, void* out, void* workspace,
                               size_t workspace_bytes, int32_t* dev_err, void* stream) {
  if (!V || !out) return FG_EINVAL;
  return profile_call(p, Q, K, V, out, token_ids, special_ids, n_special, punct_ids, n_punct,
                      nullptr, policy, mass, cost, colsum, keep, kept, workspace,
                      workspace_bytes, dev_err, stream);
}

fg_status fastgen_profile_with_policy(const fg_params* p, const void* Q, const void* K,
                                      const int32_t* token_ids, const int32_t* special_ids,
                                      int32_t n_special, const int32_t* punct_ids,
                                      int32_t n_punct, const int8_t* policy, float* colsum,
                                      uint8_t* keep, int32_t* kept, void* workspace,
                                      size_t workspace_bytes, int32_t* dev_err, void* stream) {
  if (!policy) return FG_EINVAL;
  return profile_call(p, Q, K, nullptr, nullptr, token_ids, special_ids, n_special, punct_ids,
                      n_punct, policy, nullptr, nullptr, nullptr, colsum, keep, kept, workspace,
                      workspace_bytes, dev_err, stream);
}

fg_status fastgen_profile_stall_test(const fg_params* p, const void* Q, const void* K,
                                     const int32_t* token_ids, const int32_t* special_ids,
                                     int32_t n_special, const int32_t* punct_ids, int32_t n_punct,
                                     int8_t* policy, float* mass, int32_t* cost, float* colsum,
                                     uint8_t* keep, int32_t* kept, void* workspace,
                                     size_t workspace_bytes, int32_t* dev_err, int32_t stall_pass,
                                     void* stream) {
  if (stall_pass != 1 && stall_pass != 2) return FG_EINVAL;
  if (!p || p->dtype != FG_BF16) return FG_EDTYPE;  // the bounded waits are the tensor-core passes'
  return profile_call(p, Q, K, nullptr, nullptr, token_ids, special_ids, n_special, punct_ids,
                      n_punct, nullptr, policy, mass, cost, colsum, keep, kept, workspace,
                      workspace_bytes, dev_err, stream, stall_pass);
}

size_t fastgen_plan_bytes(const fg_params* p, int32_t max_new_tokens) {
  if (check_params(p) != FG_OK || max_new_tokens < 0) return 0;
  return plan_work_offset(kv_count(p)) + plan_max_work(p, max_new_tokens) * sizeof(int2);
}

fg_status fastgen_compact_plan(const fg_params* p, const int8_t* policy, const uint8_t* keep,
                               int32_t max_new_tokens, void* plan, size_t plan_bytes,
                               fg_plan_info* info, void* stream) {
  fg_status st = check_params(p);
  if (st != FG_OK) return st;
  if (!policy || !keep || !plan || !info || max_new_tokens < 0) return FG_EINVAL;
  if (!aligned(plan, kAlign)) return FG_EINVAL;
  if ((long long)p->n + max_new_tokens > 0x7fffffffLL - fg::kRowsPerWork) return FG_EINVAL;
  if (plan_bytes < fastgen_plan_bytes(p, max_new_tokens)) return FG_EWORKSPACE;
  const fg::ProfileDims pd = dims(p);
  char* base = (char*)plan;
  fg_head_desc* desc = (fg_head_desc*)base;
  int2* cinfo = (int2*)(base + plan_desc_bytes(pd.Gkv));
  long long* totals = (long long*)(base + plan_desc_bytes(pd.Gkv) + plan_cinfo_bytes(pd.Gkv));
  int2* work = (int2*)(base + plan_work_offset(pd.Gkv));
  cudaStream_t s = (cudaStream_t)stream;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return FG_ECUDA;
  // wide items once there are 64 small ones per SM (16 waves of 4 CTAs)
  const int wide_at = 64 * sms;
  cudaError_t e = fg::launch_group(pd, policy, keep, cinfo, s);
  if (e == cudaSuccess)
    e = fg::launch_plan(pd.Gkv, pd.w, max_new_tokens, wide_at, cinfo, desc, work, totals, s);
  long long h[3] = {0, 0, 0};
  if (e == cudaSuccess) e = cudaMemcpyAsync(h, totals, sizeof(h), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return FG_ECUDA;
  if (h[1] > (long long)plan_max_work(p, max_new_tokens) || h[1] > 0x7fffffffLL ||
      (h[2] != fg::kRowsPerWork && h[2] != fg::kRowsPerWorkWide))
    return FG_ECUDA;
  info->pool_rows = h[0];
  info->n_work = (int32_t)h[1];
  info->rows_per_work = (int32_t)h[2];
  return FG_OK;
}

fg_status fastgen_compact(const fg_params* p, const void* K, const void* V, const uint8_t* keep,
                          const void* plan, const fg_plan_info* info, void* K_pool,
                          void* V_pool, int32_t* pos_pool, int64_t pool_rows, void* stream) {
  fg_status st = check_params(p);
  if (st != FG_OK) return st;
  if (!K || !V || !keep || !plan || !info || !K_pool || !V_pool || !pos_pool) return FG_EINVAL;
  if (!aligned(K, 16) || !aligned(V, 16) || !aligned(K_pool, 16) || !aligned(V_pool, 16) ||
      !aligned(plan, kAlign) || !aligned(pos_pool, 4))
    return FG_EINVAL;
  if (pool_rows < info->pool_rows) return FG_EWORKSPACE;
  const fg::ProfileDims pd = dims(p);
  cudaError_t e = fg::launch_compact(pd, K, V, keep, (const fg_head_desc*)plan, K_pool, V_pool,
                                     pos_pool, (cudaStream_t)stream);
  return cuda_status(e);
}

fg_status fastgen_plan_compact(const fg_params* p, const int8_t* policy, const uint8_t* keep,
                               int32_t max_new_tokens, void* plan, size_t plan_bytes,
                               const void* K, const void* V, void* K_pool, void* V_pool,
                               int32_t* pos_pool, int64_t pool_rows, fg_plan_info* info,
                               void* stream) {
  if (!K || !V || !K_pool || !V_pool || !pos_pool) return FG_EINVAL;
  fg_status st = fastgen_compact_plan(p, policy, keep, max_new_tokens, plan, plan_bytes, info,
                                      stream);
  if (st != FG_OK) return st;
  if (pool_rows < info->pool_rows) return FG_EWORKSPACE;  // info tells the caller what to allocate
  return fastgen_compact(p, K, V, keep, plan, info, K_pool, V_pool, pos_pool, pool_rows, stream);
}

size_t fastgen_decode_workspace_bytes(const fg_params* p, const fg_plan_info* info) {
  if (check_params(p) != FG_OK || !info || info->n_work < 0) return 0;
  const size_t nw = (size_t)info->n_work * group_size(p);  // one partial per item and query
  return align_up(nw * 2 * sizeof(float)) + align_up(nw * p->d * sizeof(float));
}

// Shared by fastgen_decode_attn and fastgen_decode_attn_refresh (row_acc and
// row_sc non-null: every row's attention weight is added to its score).
static fg_status decode_call(const fg_params* p, void* plan, const fg_plan_info* info,
                             void* K_pool, void* V_pool, int32_t* pos_pool, const void* q,
                             const void* k_new, const void* v_new, const int32_t* new_ids,
                             const int32_t* special_ids, int32_t n_special,
                             const int32_t* punct_ids, int32_t n_punct, int32_t pos, void* out,
                             void* workspace, size_t workspace_bytes, int32_t* dev_err,
                             float* row_acc, float* row_sc, float* head_ml, void* stream) {
  fg_status st = check_params(p);
  if (st != FG_OK) return st;
  if ((st = check_ids(special_ids, n_special)) != FG_OK) return st;
  if ((st = check_ids(punct_ids, n_punct)) != FG_OK) return st;
  if (!plan || !info || !K_pool || !V_pool || !pos_pool || !q || !k_new || !v_new ||
      !new_ids || !out || !workspace || !dev_err)
    return FG_EINVAL;
  if (!aligned(plan, kAlign) || !aligned(K_pool, 16) || !aligned(V_pool, 16) ||
      !aligned(q, 16) || !aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(out, 16) ||
      !aligned(workspace, kAlign) || !aligned(dev_err, 4) || !aligned(pos_pool, 4))
    return FG_EINVAL;
  if (pos < p->n || info->n_work < 0) return FG_EINVAL;
  if (info->rows_per_work != fg::kRowsPerWork && info->rows_per_work != fg::kRowsPerWorkWide)
    return FG_EINVAL;
  if (workspace_bytes < fastgen_decode_workspace_bytes(p, info)) return FG_EWORKSPACE;
  const fg::ProfileDims pd = dims(p);
  char* base = (char*)plan;
  fg::DecodeArgs a;
  a.rpw = info->rows_per_work;
  a.desc = (fg_head_desc*)base;
  a.work = (const int2*)(base + plan_work_offset(pd.Gkv));
  a.n_work = info->n_work;
  a.Kp = K_pool;
  a.Vp = V_pool;
  a.posp = pos_pool;
  a.q = q;
  a.k_new = k_new;
  a.v_new = v_new;
  a.new_ids = new_ids;
  a.special = special_ids;
  a.ns = n_special;
  a.punct = punct_ids;
  a.np = n_punct;
  a.pos = pos;
  a.out = out;
  char* ws = (char*)workspace;
  a.part_ml = (float*)ws;
  a.part_acc = (float*)(ws + align_up((size_t)info->n_work * pd.R * 2 * sizeof(float)));
  a.dev_err = dev_err;
  a.row_acc = row_acc;
  a.row_sc = row_sc;
  a.head_ml = head_ml;
  if (info->n_work == 0) {
    cudaError_t e = cudaMemsetAsync(out, 0, (size_t)pd.G * pd.d * elem_bytes(p),
                                    (cudaStream_t)stream);
    return cuda_status(e);
  }
  return cuda_status(fg::launch_decode(pd, a, (cudaStream_t)stream));
}

fg_status fastgen_decode_attn(const fg_params* p, void* plan, const fg_plan_info* info,
                              void* K_pool, void* V_pool, int32_t* pos_pool, const void* q,
                              const void* k_new, const void* v_new, const int32_t* new_ids,
                              const int32_t* special_ids, int32_t n_special,
                              const int32_t* punct_ids, int32_t n_punct, int32_t pos,
                              void* out, void* workspace, size_t workspace_bytes,
                              int32_t* dev_err, void* stream) {
  return decode_call(p, plan, info, K_pool, V_pool, pos_pool, q, k_new, v_new, new_ids,
                     special_ids, n_special, punct_ids, n_punct, pos, out, workspace,
                     workspace_bytes, dev_err, nullptr, nullptr, nullptr, stream);
}

// Refresh state: [acc f32 x pool_rows][sc f32 x pool_rows][role u8 x pool_rows]
// [(M, L) f32 x 2 x G].
size_t fastgen_refresh_state_bytes(const fg_params* p, const fg_plan_info* info) {
  if (check_params(p) != FG_OK || !info || info->pool_rows < 0) return 0;
  const size_t rows = (size_t)info->pool_rows, G = (size_t)p->B * p->L * p->H;
  return 2 * align_up(rows * sizeof(float)) + align_up(rows) + align_up(G * 2 * sizeof(float));
}

static fg_status check_refresh(const fg_params* p, const fg_plan_info* info, const void* state,
                               size_t state_bytes) {
  fg_status st = check_params(p);
  if (st != FG_OK) return st;
  if (group_size(p) != 1) return FG_EINVAL;  // one query per cache only
  if ((long long)ratio_count(p->r_l, p->n) + ratio_count(p->r_f, p->n) >
      fg::kRefreshMaxCandidates)
    return FG_EINVAL;
  if (!info || !state || !aligned(state, kAlign)) return FG_EINVAL;
  if (state_bytes < fastgen_refresh_state_bytes(p, info)) return FG_EWORKSPACE;
  return FG_OK;
}

fg_status fastgen_refresh_init(const fg_params* p, const void* plan, const fg_plan_info* info,
                               const int32_t* pos_pool, const float* colsum,
                               const int32_t* token_ids, const int32_t* special_ids,
                               int32_t n_special, const int32_t* punct_ids, int32_t n_punct,
                               void* state, size_t state_bytes, void* stream) {
  fg_status st = check_refresh(p, info, state, state_bytes);
  if (st != FG_OK) return st;
  if ((st = check_ids(special_ids, n_special)) != FG_OK) return st;
  if ((st = check_ids(punct_ids, n_punct)) != FG_OK) return st;
  if (!plan || !pos_pool || !colsum || !token_ids || !aligned(plan, kAlign) ||
      !aligned(pos_pool, 4) || !aligned(colsum, 4) || !aligned(token_ids, 4))
    return FG_EINVAL;
  const fg::ProfileDims pd = dims(p);
  const size_t rows = (size_t)info->pool_rows;
  char* sb = (char*)state;
  float* acc = (float*)sb;
  uint8_t* role = (uint8_t*)(sb + 2 * align_up(rows * sizeof(float)));
  return cuda_status(fg::launch_refresh_init(pd, (const fg_head_desc*)plan, pos_pool, colsum,
                                             token_ids, special_ids, n_special, punct_ids,
                                             n_punct, acc, role, (cudaStream_t)stream));
}

fg_status fastgen_decode_attn_refresh(const fg_params* p, void* plan, const fg_plan_info* info,
                                      void* K_pool, void* V_pool, int32_t* pos_pool,
                                      const void* q, const void* k_new, const void* v_new,
                                      const int32_t* new_ids, const int32_t* special_ids,
                                      int32_t n_special, const int32_t* punct_ids,
                                      int32_t n_punct, int32_t pos, int32_t period, void* out,
                                      void* state, size_t state_bytes, void* workspace,
                                      size_t workspace_bytes, int32_t* dev_err, void* stream) {
  fg_status st = check_refresh(p, info, state, state_bytes);
  if (st != FG_OK) return st;
  if (period < 1) return FG_EINVAL;
  const size_t rows = (size_t)info->pool_rows;
  char* sb = (char*)state;
  float* acc = (float*)sb;
  float* sc = (float*)(sb + align_up(rows * sizeof(float)));
  const uint8_t* role = (const uint8_t*)(sb + 2 * align_up(rows * sizeof(float)));
  float* head_ml = (float*)(sb + 2 * align_up(rows * sizeof(float)) + align_up(rows));
  st = decode_call(p, plan, info, K_pool, V_pool, pos_pool, q, k_new, v_new, new_ids,
                   special_ids, n_special, punct_ids, n_punct, pos, out, workspace,
                   workspace_bytes, dev_err, acc, sc, head_ml, stream);
  if (st != FG_OK || info->n_work == 0) return st;
  if ((pos - p->n + 1) % period != 0) return FG_OK;
  const fg::ProfileDims pd = dims(p);
  int cap = 2;
  while (cap < pd.k + pd.w) cap <<= 1;
  return cuda_status(fg::launch_refresh(pd, (fg_head_desc*)plan, K_pool, V_pool, pos_pool, acc,
                                        role, pos, cap, (cudaStream_t)stream));
}

fg_status fastgen_read_error(const int32_t* dev_err, void* stream) {
  if (!dev_err) return FG_EINVAL;
  int32_t h = 0;
  cudaStream_t s = (cudaStream_t)stream;
  if (cudaMemcpyAsync(&h, dev_err, sizeof(h), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess)
    return FG_ECUDA;
  if (h & 2) return FG_EDEVICE;
  if (h & 4) return FG_EINVAL;
  return (h & 1) ? FG_ECAPACITY : FG_OK;
}

}  // extern "C"
