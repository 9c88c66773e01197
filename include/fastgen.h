/*
 * fastgen.h -- C ABI of the GB300 (sm_103a) FastGen hot path.
 *
 * FastGen ("Model Tells You What to Discard: Adaptive KV Cache Compression
 * for LLMs", ICLR 2024; hyper.ai paper summaries in Chinese and Korean/English,
 * section Method) compresses the KV cache per attention head in two phases:
 *   1. prompt encoding: profile every head on A = softmax(Q K^T) and pick the
 *      cheapest hybrid policy of the shortlist {special, special+punct,
 *      special+punct+frequent, special+punct+frequent+local, full} whose kept
 *      attention is within the recover ratio T (eq. (C*));
 *   2. generation: keep a head-specific cache K_C, V_C = f(K, V, C), append
 *      new keys/values to it by the same policy, and attend over it.
 *
 * The library covers three calls of that path: fastgen_profile (phase 1;
 * fastgen_profile_attn also returns the prompt attention output,
 * fastgen_profile_with_policy reuses a saved head-policy map),
 * fastgen_compact_plan + fastgen_compact (building K_C, V_C) and
 * fastgen_decode_attn (one generation step for every head;
 * fastgen_decode_attn_refresh also refreshes the frequent sets, an opt-in
 * variant).
 *
 * Conventions shared by every entry point
 *   - Query heads are a flat index g = (b*L + l)*H + h over G = B*L*H
 *     instances.  Keys and values have Hkv heads per layer (grouped-query
 *     attention when Hkv < H): key/value head c = (b*L + l)*Hkv + h / (H/Hkv)
 *     serves query head g, over Gkv = B*L*Hkv instances.  Each key/value head
 *     keeps one compressed cache, shared by the query heads of its group.
 *   - All array arguments are DEVICE pointers owned by the caller unless
 *     marked HOST; the library never allocates, frees or keeps memory
 *     between calls, and has no global state.  Scratch memory is passed in
 *     as `workspace`.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Calls
 *     are asynchronous on it unless stated otherwise.
 *   - Argument errors are detected on the host before any launch and
 *     returned as a negative fg_status; nothing is launched then.  Launch
 *     failures return FG_ECUDA.  No call traps, asserts or aborts on device.
 *   - Element types: Q/K/V/q/out and the K/V pools are bf16 (FG_BF16) or
 *     fp32 (FG_FP32) per fg_params.dtype; head dim d is 64 or 128; every
 *     K/V/Q row is contiguous (row-major [.., d]) and 16-byte aligned.
 */
#ifndef FASTGEN_H
#define FASTGEN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FG_OK = 0,
  FG_EINVAL = -1,      /* bad size, ratio, threshold, null or misaligned pointer */
  FG_EDTYPE = -2,      /* dtype or head dim not supported */
  FG_EWORKSPACE = -3,  /* workspace / plan / pool buffer too small */
  FG_ECAPACITY = -4,   /* a head ran out of reserved cache rows while appending */
  FG_ECUDA = -5,       /* a CUDA runtime call or launch failed */
  FG_EDEVICE = -6      /* a kernel's bounded wait timed out (reported through dev_err) */
} fg_status;

typedef enum { FG_BF16 = 0, FG_FP32 = 1 } fg_dtype;

/* Policy ids, in the shortlist order of eq. (C*). */
enum {
  FG_POLICY_S = 0,    /* special */
  FG_POLICY_SP = 1,   /* special + punct */
  FG_POLICY_SPF = 2,  /* special + punct + frequent */
  FG_POLICY_SPFL = 3, /* special + punct + frequent + local */
  FG_POLICY_FULL = 4  /* full cache */
};

/* Keep-mask codes written by fastgen_profile. */
enum {
  FG_KEEP_DROP = 0,   /* position not in the compressed cache */
  FG_KEEP_STATIC = 1, /* kept for the whole generation (special/punct/frequent, or full) */
  FG_KEEP_WINDOW = 2  /* kept only while inside the local window (SPFL heads) */
};

typedef struct {
  int32_t B, L, H; /* batch, layers, heads per layer: G = B*L*H */
  int32_t n;       /* prompt length, >= 1 */
  int32_t d;       /* head dim: 64 or 128 */
  int32_t dtype;   /* fg_dtype */
  float T;         /* recover ratio, 0 < T <= 1 (eq. (C*)) */
  float r_l;       /* local ratio in [0, 1]: window w = ceil(r_l * n) */
  float r_f;       /* frequent ratio in [0, 1]: k = ceil(r_f * n) keys */
  float scale;     /* score scale s in softmax(s Q K^T); 0 selects 1/sqrt(d) */
  int32_t Hkv;     /* key/value heads per layer; 0 selects H (no grouping).  H must be
                      a multiple of Hkv with a group size H/Hkv of 1, 2, 4 or 8. */
} fg_params;

/* One key/value head's compressed cache inside the pooled K/V buffers. */
typedef struct {
  int64_t off;        /* first pool row of the never-evicted segment */
  int32_t n_static;   /* rows currently used in that segment */
  int32_t static_cap; /* rows reserved for it */
  int64_t win_off;    /* first pool row of the window ring */
  int32_t w;          /* ring rows (window size; 0 unless policy is SPFL) */
  int32_t policy;     /* FG_POLICY_* */
  int32_t work_off;   /* first decode work item of this head */
  int32_t n_work;     /* decode work items of this head */
} fg_head_desc;

typedef struct {
  int64_t pool_rows;     /* rows the K, V and position pools must hold */
  int32_t n_work;        /* decode work items of the plan */
  int32_t rows_per_work; /* cache rows covered by one decode work item (the last item of a
                            never-evicted segment also covers the rows appended later) */
} fg_plan_info;

/* Human-readable text of a status code (static storage). */
const char* fastgen_status_string(fg_status s);

/* Library version as major*10000 + minor*100 + patch. */
int32_t fastgen_version(void);

/* ------------------------------------------------------------------------
 * Phase 1: prompt profiling (Method: A = softmax(QK^T), base policies,
 * shortlist, eq. (C*)).
 *
 * For every head g, with s the scale and the causal mask (row i sees j <= i):
 *   A_ij      = softmax_j(s q_i . k_j)
 *   colsum_j  = sum_i A_ij                       (cumulative attention score)
 *   Spec/Punc = prompt positions whose token id is in special_ids / punct_ids
 *   Freq      = top-k keys by colsum, k = ceil(r_f n), ties to the lower index
 *   Local_i   = {j : i - w < j <= i}, w = ceil(r_l n)
 *   mass[g,p] = (1/n) sum_i sum_{j in K_i^p} A_ij for the nested per-row sets
 *               K^0 = Spec, K^1 = K^0 u Punc, K^2 = K^1 u Freq,
 *               K_i^3 = K^2 u Local_i; mass[g,4] = 1.  1 - mass is the mean
 *               half-L1 distance of eq. (C*).
 *   cost[g,p] = cache rows kept at the end of the prompt: |K^p| for p <= 2,
 *               |K^2 u {n-w .. n-1}| for p = 3, n for p = 4.
 *   policy[g] = the first p (= cheapest) with mass[g,p] >= T.
 *   keep[g,j] = FG_KEEP_* code of position j in the chosen policy's cache.
 *   kept[g]   = cost[g, policy[g]].
 * Ratios are evaluated as ceil(r * n) exactly on the float value of r.
 *
 * With groups, every query head is profiled on its own against its group's
 * keys (the per-head outputs below are per query head).
 *
 * Arguments:
 *   Q [G, n, d] and K [Gkv, n, d], dtype, row-major, 16-byte aligned.
 *   token_ids   [B, n] int32 prompt token ids.
 *   special_ids [n_special] int32, punct_ids [n_punct] int32 (0 <= counts <= 4096;
 *               a count of 0 allows a NULL pointer).
 *   policy [G] int8, mass [G,5] float, cost [G,5] int32, colsum [G,n] float,
 *   keep [G,n] uint8, kept [G] int32: outputs.
 *   workspace: >= fastgen_profile_workspace_bytes(p) bytes, 256-byte aligned.
 *   dev_err: device int32 the call ORs with 2 if a kernel's bounded wait on
 *            its own pipeline timed out (about 1 s); read with
 *            fastgen_read_error (FG_EDEVICE).  Never set in normal operation.
 * bf16 inputs run on the tcgen05 tensor cores (fp32 accumulation); fp32
 * inputs on fp32 SIMT arithmetic.
 * Errors: FG_EINVAL for G, n < 1, T outside (0,1], ratios outside [0,1],
 * null/misaligned pointers; FG_EDTYPE for other d or dtype; FG_EWORKSPACE.
 * ------------------------------------------------------------------------ */
size_t fastgen_profile_workspace_bytes(const fg_params* p);

fg_status fastgen_profile(const fg_params* p, const void* Q, const void* K,
                          const int32_t* token_ids, const int32_t* special_ids,
                          int32_t n_special, const int32_t* punct_ids, int32_t n_punct,
                          int8_t* policy, float* mass, int32_t* cost, float* colsum,
                          uint8_t* keep, int32_t* kept, void* workspace,
                          size_t workspace_bytes, int32_t* dev_err, void* stream);

/* ------------------------------------------------------------------------
 * Phase 1 with the prompt attention output (Method, first paragraph: the
 * prompt-encoding phase runs attention over the prompt; A = softmax(QK^T)).
 *
 * Everything fastgen_profile writes, plus
 *   out[g, i, :] = sum_{j <= i} A_ij v_j        (V [Gkv, n, d] like K)
 * for every query head g and prompt position i, in the dtype of Q/K/V,
 * row-major [G, n, d], 16-byte aligned.  A third pass reuses the row
 * log-sum-exps of the first, so each weight A_ij is final when it is formed
 * (no rescaling); bf16 inputs run it on the tcgen05 tensor cores (P rounded
 * to bf16 for the P V product, fp32 accumulation), fp32 inputs on fp32 SIMT
 * arithmetic.  Same workspace as fastgen_profile.
 * Errors: those of fastgen_profile; FG_EINVAL for NULL or misaligned V/out.
 * ------------------------------------------------------------------------ */
fg_status fastgen_profile_attn(const fg_params* p, const void* Q, const void* K, const void* V,
                               const int32_t* token_ids, const int32_t* special_ids,
                               int32_t n_special, const int32_t* punct_ids, int32_t n_punct,
                               int8_t* policy, float* mass, int32_t* cost, float* colsum,
                               uint8_t* keep, int32_t* kept, void* out, void* workspace,
                               size_t workspace_bytes, int32_t* dev_err, void* stream);

/* ------------------------------------------------------------------------
 * Phase 1 with a saved head-policy map (policy reuse across prompts: the
 * overview page's saved head-type map read with the Method's reuse of the
 * prompt-time policy).
 *
 * policy [G] int8 (device, input) fixes each head's shortlist entry
 * (FG_POLICY_*), e.g. the policy output of an earlier fastgen_profile saved
 * by the caller.  For this prompt the call writes, per head g, the keep codes
 * and kept count of that entry's final cache, with the definitions of
 * fastgen_profile (Spec/Punc from token_ids, the last w positions, the top-k
 * keys of THIS prompt's colsum).  No masses are formed and no choice is made.
 * The column sums are computed only for heads whose entry contains
 * C_frequent (FG_POLICY_SPF, FG_POLICY_SPFL); with bf16 inputs the other heads
 * skip both profiler passes.  colsum rows of the other heads are left
 * unspecified (fp32 inputs score every head).
 *
 * Arguments as for fastgen_profile, without policy/mass/cost outputs; the
 * same workspace size.  keep/kept and the policy map then feed
 * fastgen_compact_plan / fastgen_compact as usual.
 * A saved value outside 0..4 is read as FG_POLICY_FULL and ORs 4 into
 * dev_err (fastgen_read_error returns FG_EINVAL).
 * Errors: those of fastgen_profile; FG_EINVAL for a NULL policy.
 * ------------------------------------------------------------------------ */
fg_status fastgen_profile_with_policy(const fg_params* p, const void* Q, const void* K,
                                      const int32_t* token_ids, const int32_t* special_ids,
                                      int32_t n_special, const int32_t* punct_ids,
                                      int32_t n_punct, const int8_t* policy, float* colsum,
                                      uint8_t* keep, int32_t* kept, void* workspace,
                                      size_t workspace_bytes, int32_t* dev_err, void* stream);

/* ------------------------------------------------------------------------
 * Compaction, step 1: the pool layout (Method: K_C, V_C = f(K, V, C)).
 *
 * From policy [G] and keep [G, n] (outputs of fastgen_profile) it writes,
 * into the device buffer `plan` (>= fastgen_plan_bytes bytes, 256-byte
 * aligned): Gkv fg_head_desc records followed by the decode work list.  The
 * cache of key/value head c holds the union of its query heads' caches (a
 * position is never-evicted if any member keeps it so, else in the window if
 * any member's window holds it) and follows the largest member policy; without
 * groups that is the head's own cache.  Each cache gets a never-evicted
 * segment of (kept static rows + max_new_tokens) rows and, for SPFL, a ring
 * of w rows for the sliding window.  The totals are written to *info (HOST
 * pointer).  This call is SYNCHRONOUS: it waits on `stream` to return them.
 * ------------------------------------------------------------------------ */
size_t fastgen_plan_bytes(const fg_params* p, int32_t max_new_tokens);

fg_status fastgen_compact_plan(const fg_params* p, const int8_t* policy, const uint8_t* keep,
                               int32_t max_new_tokens, void* plan, size_t plan_bytes,
                               fg_plan_info* info, void* stream);

/* ------------------------------------------------------------------------
 * Compaction, step 2: gather the kept prompt rows into the pools.
 *
 * K, V [Gkv, n, d] dtype; keep [G, n] from fastgen_profile; plan and *info
 * (HOST pointer) from fastgen_compact_plan.  Writes K_pool, V_pool
 * [pool_rows, d] dtype and pos_pool [pool_rows] int32 (absolute position of
 * each row, -1 = empty).  Never-evicted rows are stored in position order;
 * window rows sit at ring slot (position mod w).
 * Errors: FG_EWORKSPACE if pool_rows < info->pool_rows.
 * ------------------------------------------------------------------------ */
fg_status fastgen_compact(const fg_params* p, const void* K, const void* V, const uint8_t* keep,
                          const void* plan, const fg_plan_info* info, void* K_pool,
                          void* V_pool, int32_t* pos_pool, int64_t pool_rows, void* stream);

/* ------------------------------------------------------------------------
 * Compaction, both steps in one call: fastgen_compact_plan, then, if the
 * caller's pools hold info->pool_rows rows, fastgen_compact at once (no
 * return to the caller between the plan's host read-back and the gather
 * launch).  Arguments as for those two calls; `info` is always filled when
 * the plan succeeded.  Returns FG_EWORKSPACE without launching the gather when
 * pool_rows < info->pool_rows (the caller allocates that many rows and calls
 * fastgen_compact).  Synchronous like fastgen_compact_plan.
 * ------------------------------------------------------------------------ */
fg_status fastgen_plan_compact(const fg_params* p, const int8_t* policy, const uint8_t* keep,
                               int32_t max_new_tokens, void* plan, size_t plan_bytes,
                               const void* K, const void* V, void* K_pool, void* V_pool,
                               int32_t* pos_pool, int64_t pool_rows, fg_plan_info* info,
                               void* stream);

/* ------------------------------------------------------------------------
 * Generation step for every head (Method: head-specific caches, appends,
 * policy reused from the prompt).
 *
 * The new token at absolute position pos (>= n) with id new_ids[b] is placed
 * by its head's policy: full -> appended; special/punct-containing policies
 * append it to the never-evicted segment when its id is special (or, except
 * for the special-only policy, punctuation); SPFL heads otherwise put it in
 * the window ring at slot pos mod w, evicting the row that left the window.
 * The frequent set stays as profiled.  Then
 *   out[g] = sum_{j in cache_g} softmax_j(s q_g . k_j) v_j   (zeros if empty)
 * over the cache after placement.
 *
 * Arguments: plan and *info (HOST pointer) from fastgen_compact_plan; pools
 * from fastgen_compact (updated in place); q [G, d], k_new, v_new [Gkv, d]
 * dtype; new_ids [B] int32; id sets as in fastgen_profile; out [G, d] dtype
 * (every query head attends over its group's cache);
 * workspace >= fastgen_decode_workspace_bytes(p, info).  dev_err: device
 * int32 that the call ORs with 1 when a head had no free reserved row (that
 * token is then not stored); read it with fastgen_read_error.
 * ------------------------------------------------------------------------ */
size_t fastgen_decode_workspace_bytes(const fg_params* p, const fg_plan_info* info);

fg_status fastgen_decode_attn(const fg_params* p, void* plan, const fg_plan_info* info,
                              void* K_pool, void* V_pool, int32_t* pos_pool, const void* q,
                              const void* k_new, const void* v_new, const int32_t* new_ids,
                              const int32_t* special_ids, int32_t n_special,
                              const int32_t* punct_ids, int32_t n_punct, int32_t pos,
                              void* out, void* workspace, size_t workspace_bytes,
                              int32_t* dev_err, void* stream);

/* ------------------------------------------------------------------------
 * Decode-time refresh of C_frequent (opt-in variant; Method: C_frequent keeps
 * the tokens with the largest cumulative attention scores, and the stability
 * paragraph examines accumulated attention scores at the prompt and at later
 * decoding steps).  The pages reuse the prompt-time policy and state no
 * update rule; this variant is the library's own rule and is off unless
 * these calls are used.
 *
 * Rule: every cached row j carries an accumulated score acc_j: its prompt
 * column sum colsum_j at the end of the prompt (0 for a generated token when
 * it is placed) plus, at every generation step, the attention weight the
 * step's query gives it.  After every `period`-th step, a local-hybrid
 * (FG_POLICY_SPFL) cache re-chooses its frequent members (the never-evicted
 * rows kept for frequency, i.e. not special or punctuation tokens) as the
 * |F| rows of largest acc among those members and the rows of the local
 * window, ties to the lower position; |F| is fixed at the prompt, so the
 * cache never grows.  A member that loses its place leaves the cache unless
 * it is still inside the window (then it stays until it is w positions old);
 * a window row that wins a place stays for good; dropped rows never return.
 * Other policies have no window rows to promote and are left as profiled.
 *
 * Limits: no groups (Hkv == H, else FG_EINVAL); ceil(r_f n) + ceil(r_l n)
 * <= 16384 (the candidates of one cache are ranked in shared memory, else
 * FG_EINVAL).
 *
 * fastgen_refresh_state_bytes: size of the caller-owned state (per pool
 *   row: acc float, the step's score float, a role byte; per head: the step's
 *   softmax maximum and sum), 256-byte aligned.
 * fastgen_refresh_init: after fastgen_compact, sets acc from colsum [G, n]
 *   (fastgen_profile's output) and marks the frequent slots from token_ids
 *   [B, n] and the id sets.  Asynchronous on `stream`.
 * fastgen_decode_attn_refresh: fastgen_decode_attn (same arguments and
 *   outputs) that also accumulates every cached row's weight into acc and,
 *   when (pos - n + 1) is a multiple of `period` (>= 1), runs the refresh
 *   after the step.  With a period longer than the generation it gives
 *   fastgen_decode_attn's outputs bit for bit.
 * Errors: those of fastgen_decode_attn; FG_EINVAL for the limits above, a
 * period < 1 or a NULL/misaligned state; FG_EWORKSPACE for a short state.
 * ------------------------------------------------------------------------ */
size_t fastgen_refresh_state_bytes(const fg_params* p, const fg_plan_info* info);

fg_status fastgen_refresh_init(const fg_params* p, const void* plan, const fg_plan_info* info,
                               const int32_t* pos_pool, const float* colsum,
                               const int32_t* token_ids, const int32_t* special_ids,
                               int32_t n_special, const int32_t* punct_ids, int32_t n_punct,
                               void* state, size_t state_bytes, void* stream);

fg_status fastgen_decode_attn_refresh(const fg_params* p, void* plan, const fg_plan_info* info,
                                      void* K_pool, void* V_pool, int32_t* pos_pool,
                                      const void* q, const void* k_new, const void* v_new,
                                      const int32_t* new_ids, const int32_t* special_ids,
                                      int32_t n_special, const int32_t* punct_ids,
                                      int32_t n_punct, int32_t pos, int32_t period, void* out,
                                      void* state, size_t state_bytes, void* workspace,
                                      size_t workspace_bytes, int32_t* dev_err, void* stream);

/* ------------------------------------------------------------------------
 * fastgen_decode_attn for callers that cannot allocate device memory.
 * (The paper has no counterpart: this is a deployment convenience.)
 *
 * Some callers cannot call cudaMalloc when they decode: a serving engine that
 * gives all free device memory to its own pool at start-up (a new allocation
 * fails or undercuts that pool), a plug-in whose host framework owns every
 * allocation, or a latency-bound loop that cannot pay for cudaMalloc's
 * implicit synchronisation.  This variant takes the same arguments as
 * fastgen_decode_attn minus `workspace`/`workspace_bytes` and allocates
 * nothing: its scratch (the split-K partial results) is a fixed array of
 * FASTGEN_NOALLOC_SCRATCH_BYTES inside the library.
 *   - When the array is set aside: the array lives in its own CUDA module of
 *     the library, which CUDA loads on a device the first time this entry
 *     point looks the array up there.  Under CUDA's default lazy module
 *     loading that is the first call of this entry point on the device (with
 *     CUDA_MODULE_LOADING=EAGER it is the creation of the device's context);
 *     from then on the device holds the array until the process exits.  So
 *     make the first call at set-up: before the caller's own pool takes the
 *     device's free memory, and before any stream capture.
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress, with the device current) and caches it for the
 *     life of the process: the cache assumes the device's primary context is
 *     never destroyed (no cudaDeviceReset between calls).
 *   - Every call shares the one array: calls that overlap on the GPU (other
 *     streams, other host threads) race and produce wrong results, so issue
 *     them in order on one stream.  Nothing in the array has to start at
 *     zero: a call writes every entry it later reads.
 *   - Size limit: the plan fits when fastgen_decode_workspace_bytes(p, info)
 *     <= FASTGEN_NOALLOC_SCRATCH_BYTES, i.e. roughly
 *     info->n_work * (H / Hkv) * (d + 2) * 4 bytes <= 8 MiB: about 16,000
 *     work items at d = 128 without groups, 8,000 with groups of 2, 2,000
 *     with groups of 8 (one work item covers info->rows_per_work = 256 or 512
 *     rows of one cache).  The 7B attention shape (1024 heads, 2048-token
 *     prompt, 256 new tokens: about 5,000 items) fits; the 13B and 65B
 *     shapes (tens of thousands of items) do not.  Larger plans return FG_EWORKSPACE before
 *     anything is launched; other errors as fastgen_decode_attn.
 * ------------------------------------------------------------------------ */
#define FASTGEN_NOALLOC_SCRATCH_BYTES (8u * 1024u * 1024u)

fg_status fastgen_decode_attn_noalloc(const fg_params* p, void* plan, const fg_plan_info* info,
                                      void* K_pool, void* V_pool, int32_t* pos_pool,
                                      const void* q, const void* k_new, const void* v_new,
                                      const int32_t* new_ids, const int32_t* special_ids,
                                      int32_t n_special, const int32_t* punct_ids,
                                      int32_t n_punct, int32_t pos, void* out,
                                      int32_t* dev_err, void* stream);

/* ------------------------------------------------------------------------
 * Test support for the bounded-wait error path (the paper has no
 * counterpart).  fastgen_profile, except that the producer warp of tensor-core
 * pass `stall_pass` (1: row log-sum-exps, 2: column sums) never starts: the
 * pass's other warps wait for work that never comes, each wait runs out after
 * its limit (about 1 s), and every CTA unwinds with no copy or MMA in flight
 * and ORs 2 into *dev_err (fastgen_read_error then gives FG_EDEVICE).  The
 * stalled pass's outputs are left as they were; the context stays usable and
 * later calls on the stream run normally.  bf16 inputs only (FG_EDTYPE
 * otherwise); FG_EINVAL for another stall_pass; other errors as
 * fastgen_profile.
 * ------------------------------------------------------------------------ */
fg_status fastgen_profile_stall_test(const fg_params* p, const void* Q, const void* K,
                                     const int32_t* token_ids, const int32_t* special_ids,
                                     int32_t n_special, const int32_t* punct_ids, int32_t n_punct,
                                     int8_t* policy, float* mass, int32_t* cost, float* colsum,
                                     uint8_t* keep, int32_t* kept, void* workspace,
                                     size_t workspace_bytes, int32_t* dev_err, int32_t stall_pass,
                                     void* stream);

/* Synchronously reads a device flag written by fastgen_profile,
 * fastgen_profile_with_policy or fastgen_decode_attn and maps it to a status
 * (FG_OK, FG_ECAPACITY, FG_EINVAL for an out-of-range saved policy, or
 * FG_EDEVICE).  Waits on `stream`. */
fg_status fastgen_read_error(const int32_t* dev_err, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* FASTGEN_H */
