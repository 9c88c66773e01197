"""FastGen oracle: a plain float64 CPU statement of the adaptive KV-cache path.

TEST INFRASTRUCTURE ONLY.  Nothing in the product imports this module; only
the tests, ``__graft_entry__.smoke()`` and the bench's CPU-baseline arm may
call it.  It shares no code with the CUDA path.

Sources (the FastGen paper, "Model Tells You What to Discard: Adaptive KV
Cache Compression for LLMs", ICLR 2024, as summarised on the hyper.ai pages
in Chinese and Korean/English; same text on both):
  * Method, first paragraph: two phases.  Prompt encoding profiles every
    attention head; generation keeps a head-specific KV cache to which new
    keys/values are appended.
  * Method, eq. (C*): C* = argmin_C CacheMemoryCost(C) subject to
    |A - softmax(Q K_C^T)| <= 1 - T, with A = softmax(Q K^T).
  * Method, base policies: C_special (special tokens such as the
    begin-of-sequence marker), C_punct (punctuation), C_local (recent tokens
    within a relative distance set by r_l), C_frequent (the tokens with the
    largest cumulative attention scores, share r_f), C_full.
  * Method, eq. for the shortlist: {special, special+punct,
    special+punct+frequent, special+punct+frequent+local, full}, hybrids
    being unions of base caches.
  * Method, stability paragraph: the policy chosen at the prompt is reused
    for all generated tokens.

Readings of points the pages leave open (each is listed in the design notes):
  R1 scores are scaled by s = 1/sqrt(d) unless a scale is given; the prompt
     map is causal (row i sees keys j <= i).
  R2 the distance in eq. (C*) is half the L1 norm per query row, averaged
     uniformly over all n rows.  Renormalising A over a kept set K_i gives
     (1/2)||A_i - Ahat_i||_1 = 1 - m_i with m_i the kept mass, so the
     constraint is mean_i m_i >= T.
  R3 w = ceil(r_l * n) and k = ceil(r_f * n), evaluated exactly on the
     float32 value of the ratio.
  R4 the local set of query row i is {j : i - w < j <= i}; the final cache of
     a local-containing policy keeps the last w prompt positions.
  R5 the frequent set is the top-k of colsum_j = sum_i A_ij over all prompt
     keys, ties going to the lower index.
  R6 policy = the cheapest shortlist entry whose mass is >= T; equal cost goes
     to the earlier entry; the full cache has mass exactly 1.
  R7 decoding: a new token is cached by a head iff its policy is full, or
     its policy contains special and the token is special, or it contains
     punct and the token is punctuation, or the policy contains local (the
     token then lives in the window).  Special/punct/frequent members never
     leave the cache; window members leave it once they are w positions old.
     The frequent set is frozen at the prompt.  The query attends over the
     cache after the new token is placed; an empty cache yields zeros.
  R11 a saved head-policy map (the overview page's offline head-type map,
     read together with the Method's policy reuse) fixes each head's
     shortlist entry for a later prompt; that prompt's caches are the
     entry's final sets built from the prompt itself (its special and
     punctuation ids, its last w positions, the top-k of its own cumulative
     attention scores).  Only entries containing C_frequent need the scores;
     no masses are formed and no choice is made.
"""
from __future__ import annotations

import math

import numpy as np

# shortlist order of eq. (C*)'s policy set
POLICIES = ("special", "special+punct", "special+punct+frequent",
            "special+punct+frequent+local", "full")
P_S, P_SP, P_SPF, P_SPFL, P_FULL = range(5)

# cache-membership codes of the keep mask
DROP, KEEP_STATIC, KEEP_WINDOW = 0, 1, 2


def default_scale(d: int) -> float:
    """R1: 1/sqrt(d), the scale of the Llama attention the workloads copy."""
    return 1.0 / math.sqrt(d)


def ratio_count(r: float, n: int) -> int:
    """R3: ceil(r * n) on the float32 value of r (exact in float64)."""
    r32 = float(np.float32(r))
    return int(math.ceil(r32 * n))


def attention_map(Q: np.ndarray, K: np.ndarray, scale: float) -> np.ndarray:
    """A = softmax(s Q K^T) with the causal mask (Method, eq. (C*); R1)."""
    Q = np.asarray(Q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    n = Q.shape[0]
    S = scale * (Q @ K.T)
    S[np.triu_indices(n, 1)] = -np.inf
    S = S - S.max(axis=1, keepdims=True)
    E = np.exp(S)
    return E / E.sum(axis=1, keepdims=True)


def cumulative_scores(A: np.ndarray) -> np.ndarray:
    """colsum_j = sum_i A_ij: the cumulative attention score of key j that
    C_frequent ranks by (Method, base policies; R5)."""
    return A.sum(axis=0)


def token_sets(ids, special_ids, punct_ids):
    """Boolean masks of C_special and C_punct members among positions."""
    ids = np.asarray(ids)
    return np.isin(ids, np.asarray(special_ids)), np.isin(ids, np.asarray(punct_ids))


def frequent_set(colsum: np.ndarray, k: int) -> np.ndarray:
    """C_frequent: the k keys of largest colsum, lower index first on ties (R5)."""
    order = np.argsort(-colsum, kind="stable")
    m = np.zeros(colsum.shape[0], dtype=bool)
    m[order[:k]] = True
    return m


def local_rows(n: int, w: int) -> np.ndarray:
    """C_local per query row i: {j : i - w < j <= i} (R4), as an [n, n] mask."""
    i = np.arange(n)[:, None]
    j = np.arange(n)[None, :]
    return (j <= i) & (j > i - w)


def candidate_row_masks(n, spec, punc, freq, w):
    """Per-row kept sets K_i^p of the first four shortlist entries (unions of
    base caches; Method, shortlist equation)."""
    k0 = np.broadcast_to(spec, (n, n))
    k1 = np.broadcast_to(spec | punc, (n, n))
    k2 = np.broadcast_to(spec | punc | freq, (n, n))
    k3 = k2 | local_rows(n, w)
    return [k0, k1, k2, k3]


def kept_mass(A: np.ndarray, row_mask: np.ndarray) -> float:
    """mean_i sum_{j in K_i} A_ij, which is 1 - mean_i (1/2)||A_i - Ahat_i||_1 (R2)."""
    n = A.shape[0]
    return float((A * row_mask).sum() / n)


def final_sets(n, spec, punc, freq, w):
    """Positions kept at the end of the prompt by each shortlist entry, as
    keep-code vectors (DROP / KEEP_STATIC / KEEP_WINDOW)."""
    out = []
    static = [spec, spec | punc, spec | punc | freq]
    for s in static:
        out.append(np.where(s, KEEP_STATIC, DROP).astype(np.uint8))
    win = np.arange(n) >= n - w
    k3 = np.where(static[2], KEEP_STATIC, np.where(win, KEEP_WINDOW, DROP)).astype(np.uint8)
    out.append(k3)
    out.append(np.full(n, KEEP_STATIC, dtype=np.uint8))
    return out


def choose_policy(mass, cost, T: float) -> int:
    """eq. (C*): the cheapest entry with mass >= T; ties go to the earlier entry."""
    feasible = [p for p in range(5) if mass[p] >= T]
    return min(feasible, key=lambda p: (cost[p], p))


def profile_head(Q, K, ids, special_ids, punct_ids, T, r_l, r_f, scale=None):
    """Profile one head over its prompt (Method: prompt-encoding phase).

    Q, K: [n, d] (any float dtype; upcast to float64).  ids: [n] token ids.
    Returns dict(policy, mass[5], cost[5], colsum[n], keep[n] uint8, kept,
    w, k, A).
    """
    Q = np.asarray(Q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    n, d = Q.shape
    s = default_scale(d) if scale is None else scale
    w, k = ratio_count(r_l, n), ratio_count(r_f, n)
    A = attention_map(Q, K, s)
    colsum = cumulative_scores(A)
    spec, punc = token_sets(ids[:n], special_ids, punct_ids)
    freq = frequent_set(colsum, k)
    masks = candidate_row_masks(n, spec, punc, freq, w)
    mass = [kept_mass(A, m) for m in masks] + [1.0]
    finals = final_sets(n, spec, punc, freq, w)
    cost = [int((f != DROP).sum()) for f in finals]
    p = choose_policy(mass, cost, T)
    return dict(policy=p, mass=np.array(mass), cost=np.array(cost),
                colsum=colsum, keep=finals[p], kept=cost[p], w=w, k=k, A=A,
                freq=freq)


def masses_from_column_scores(colsum, bandcol, spec, punc, freq):
    """Column form of the four candidate masses (exact algebra on eq. (C*)'s
    per-row sums): for p <= 2 the kept mass is sum_{j in K^p} colsum_j / n;
    for the local hybrid it is [sum_j bandcol_j + sum_{j in K^2}
    (colsum_j - bandcol_j)] / n, with bandcol_j = sum_{i=j}^{j+w-1} A_ij.
    Used to cross-check the per-row definition."""
    n = colsum.shape[0]
    k2 = spec | punc | freq
    m0 = colsum[spec].sum() / n
    m1 = colsum[spec | punc].sum() / n
    m2 = colsum[k2].sum() / n
    m3 = (bandcol.sum() + (colsum[k2] - bandcol[k2]).sum()) / n
    return np.array([m0, m1, m2, m3, 1.0])


def band_scores(A: np.ndarray, w: int) -> np.ndarray:
    """bandcol_j = sum_{i=j}^{min(j+w-1, n-1)} A_ij."""
    n = A.shape[0]
    i = np.arange(n)[:, None]
    j = np.arange(n)[None, :]
    band = (i >= j) & (i < j + w)
    return (A * band).sum(axis=0)


def compact_head(K, V, keep):
    """K_C, V_C = f(K, V, C) (Method, second paragraph): the kept prompt
    rows in position order, split into never-evicted members and window
    members.  Returns (static_pos, window_pos, K_static, V_static, K_win, V_win)."""
    keep = np.asarray(keep)
    sp = np.nonzero(keep == KEEP_STATIC)[0]
    wp = np.nonzero(keep == KEEP_WINDOW)[0]
    K = np.asarray(K)
    V = np.asarray(V)
    return sp, wp, K[sp], V[sp], K[wp], V[wp]


def stores_static(policy: int, is_special: bool, is_punct: bool) -> bool:
    """R7: does a generated token join the never-evicted part of the cache?"""
    if policy == P_FULL:
        return True
    if policy == P_S:
        return is_special
    return is_special or is_punct


def attend(q, Kc, Vc, scale):
    """Single-query attention softmax(s q K_c^T) V_c over a cache (zeros if empty)."""
    q = np.asarray(q, dtype=np.float64)
    if Kc.shape[0] == 0:
        return np.zeros(q.shape[0])
    s = scale * (np.asarray(Kc, dtype=np.float64) @ q)
    e = np.exp(s - s.max())
    return (e / e.sum()) @ np.asarray(Vc, dtype=np.float64)


def decode_positions(policy, static_pos, w, t):
    """Cache positions seen by the query at position t (after placement):
    the never-evicted members plus, for the local hybrid, the window
    (t - w, t] (R7)."""
    pos = set(int(p) for p in static_pos)
    if policy == P_SPFL:
        pos.update(range(max(t - w + 1, 0), t + 1))
    return np.array(sorted(pos), dtype=np.int64)


def decode_head(policy, keep, n, w, ids, Qall, Kall, Vall, special_ids, punct_ids,
                steps, scale=None):
    """Token generation with the head-specific cache (Method, first and
    stability paragraphs): for t = n .. n+steps-1, place token t by R7 and
    attend with q_t.  Qall/Kall/Vall: [n + steps, d]; ids: [n + steps].
    Returns (out [steps, d], final cache positions)."""
    Kall = np.asarray(Kall, dtype=np.float64)
    Vall = np.asarray(Vall, dtype=np.float64)
    Qall = np.asarray(Qall, dtype=np.float64)
    d = Kall.shape[1]
    s = default_scale(d) if scale is None else scale
    sset, pset = set(int(x) for x in special_ids), set(int(x) for x in punct_ids)
    static = [int(j) for j in np.nonzero(np.asarray(keep) == KEEP_STATIC)[0]]
    out = np.zeros((steps, d))
    pos = np.array(static, dtype=np.int64)
    for step in range(steps):
        t = n + step
        tau = int(ids[t])
        if stores_static(policy, tau in sset, tau in pset):
            static.append(t)
        pos = decode_positions(policy, static, w, t)
        out[step] = attend(Qall[t], Kall[pos], Vall[pos], s)
    return out, pos


# ---------------------------------------------------------------------------
# Grouped-query attention (the kdj.com article lists combining FastGen with
# grouped-query attention as future work; the pages fix no rule for it).
# Reading R10: query heads are profiled one by one exactly as above, each
# against its group's shared K; the group keeps one cache, the union of its
# members' final caches (a position is never-evicted if any member keeps it
# so, else in the window if any member's window holds it); a generated token
# is placed by the rule of the group's largest policy (the shortlist entries
# are nested, so that rule keeps every token any member would keep); every
# member attends over the shared cache.
# ---------------------------------------------------------------------------

def union_keep(keeps):
    """Union of the members' keep codes (never-evicted beats window)."""
    keeps = np.asarray(keeps)
    static = (keeps == KEEP_STATIC).any(axis=0)
    window = (keeps == KEEP_WINDOW).any(axis=0)
    return np.where(static, KEEP_STATIC, np.where(window, KEEP_WINDOW, DROP)).astype(np.uint8)


def profile_group(Qs, K, ids, special_ids, punct_ids, T, r_l, r_f, scale=None):
    """Profiles every query head of a group against the shared K.  Returns
    (member results, group keep codes, group policy)."""
    members = [profile_head(Q, K, ids, special_ids, punct_ids, T, r_l, r_f, scale) for Q in Qs]
    keep = union_keep([m["keep"] for m in members])
    return members, keep, max(m["policy"] for m in members)


def decode_group(policy, keep, n, w, ids, Qalls, Kall, Vall, special_ids, punct_ids, steps,
                 scale=None):
    """Generation over a group's shared cache: the token at each position is
    placed by the group policy's rule and every member attends with its own
    query.  Returns (out [members, steps, d], final cache positions)."""
    Kall = np.asarray(Kall, dtype=np.float64)
    Vall = np.asarray(Vall, dtype=np.float64)
    d = Kall.shape[1]
    s = default_scale(d) if scale is None else scale
    sset, pset = set(int(x) for x in special_ids), set(int(x) for x in punct_ids)
    static = [int(j) for j in np.nonzero(np.asarray(keep) == KEEP_STATIC)[0]]
    out = np.zeros((len(Qalls), steps, d))
    pos = np.array(static, dtype=np.int64)
    for step in range(steps):
        t = n + step
        tau = int(ids[t])
        if stores_static(policy, tau in sset, tau in pset):
            static.append(t)
        pos = decode_positions(policy, static, w, t)
        for m, Qall in enumerate(Qalls):
            out[m, step] = attend(np.asarray(Qall, dtype=np.float64)[t], Kall[pos], Vall[pos], s)
    return out, pos


# --- policy reuse with a saved head-policy map (R11) ----------------------

def keep_for_policy(policy, ids, special_ids, punct_ids, r_l, r_f, n, colsum=None):
    """Keep codes of shortlist entry `policy` on a prompt of n tokens (R11).

    The cache is the entry's final set (final_sets): special / punctuation
    positions from the prompt's ids, the last w = ceil(r_l n) positions for
    the local part, and the top k = ceil(r_f n) keys of the prompt's own
    cumulative attention scores `colsum` for the frequent part.  `colsum` is
    required exactly when the entry contains C_frequent.
    """
    n = int(n)
    spec, punc = token_sets(np.asarray(ids)[:n], special_ids, punct_ids)
    w, k = ratio_count(r_l, n), ratio_count(r_f, n)
    if policy in (P_SPF, P_SPFL):
        if colsum is None:
            raise ValueError("entries containing C_frequent need the column sums")
        freq = frequent_set(np.asarray(colsum, dtype=np.float64), k)
    else:
        freq = np.zeros(n, dtype=bool)
    return final_sets(n, spec, punc, freq, w)[policy]


def profile_with_policy(policy, Q, K, ids, special_ids, punct_ids, r_l, r_f, scale=None):
    """One head of a later prompt under a saved policy (R11): the attention
    map and its column sums are formed only when the entry needs C_frequent.
    Returns dict(keep, kept, colsum or None)."""
    Q = np.asarray(Q, dtype=np.float64)
    n, d = Q.shape
    colsum = None
    if policy in (P_SPF, P_SPFL):
        s = default_scale(d) if scale is None else scale
        colsum = cumulative_scores(attention_map(Q, np.asarray(K, dtype=np.float64), s))
    keep = keep_for_policy(policy, ids, special_ids, punct_ids, r_l, r_f, n, colsum)
    return dict(keep=keep, kept=int((keep != DROP).sum()), colsum=colsum)


# --- prompt attention output --------------------------------------------------

def prompt_attention(Q, K, V, scale=None):
    """The prompt-encoding attention output of one head, O = A V with
    A = softmax(s Q K^T) under the causal mask (Method, first paragraph and
    A = softmax(QK^T); reading R1 for s and the mask).  [n, d_v] float64."""
    Q = np.asarray(Q, dtype=np.float64)
    s = default_scale(Q.shape[1]) if scale is None else scale
    A = attention_map(Q, np.asarray(K, dtype=np.float64), s)
    return A @ np.asarray(V, dtype=np.float64)



# --- long prompts: the same profile with the map formed a block of rows at a time

def attention_rows(Q, K, scale, lo, hi):
    """Rows lo..hi-1 of A = softmax(s Q K^T) under the causal mask, each row
    formed as in attention_map: row i depends only on q_i and k_0..k_i, so
    the rows are returned over the key columns 0..hi-1 (every later key is
    masked out of all of them).  [hi - lo, hi] float64."""
    S = scale * (Q[lo:hi] @ K[:hi].T)
    i = np.arange(lo, hi)[:, None]
    j = np.arange(hi)[None, :]
    S[j > i] = -np.inf
    S = S - S.max(axis=1, keepdims=True)
    E = np.exp(S)
    return E / E.sum(axis=1, keepdims=True)


def local_rows_block(lo, hi, w):
    """Rows lo..hi-1 of the C_local mask {j : i - w < j <= i} (R4) over the
    key columns 0..hi-1."""
    i = np.arange(lo, hi)[:, None]
    j = np.arange(hi)[None, :]
    return (j <= i) & (j > i - w)


def profile_head_long(Q, K, ids, special_ids, punct_ids, T, r_l, r_f, scale=None, block=512):
    """profile_head for prompts whose [n, n] map does not fit in memory.

    The definitions are those of profile_head (Method: A = softmax(QK^T),
    base policies, shortlist, eq. (C*); readings R1-R6); only the map is
    formed `block` query rows at a time, twice: the first sweep adds the
    rows into the cumulative scores colsum_j = sum_i A_ij, which fix
    C_frequent; the second sums each row's attention over the per-row kept
    sets K_i^p of the four compressed entries.  Returns the dict of
    profile_head without A."""
    Q = np.asarray(Q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    n, d = Q.shape
    s = default_scale(d) if scale is None else scale
    w, k = ratio_count(r_l, n), ratio_count(r_f, n)
    colsum = np.zeros(n)
    for lo in range(0, n, block):
        hi = min(lo + block, n)
        colsum[:hi] += attention_rows(Q, K, s, lo, hi).sum(axis=0)
    spec, punc = token_sets(ids[:n], special_ids, punct_ids)
    freq = frequent_set(colsum, k)
    static = [spec, spec | punc, spec | punc | freq]
    kept = np.zeros(4)
    for lo in range(0, n, block):
        hi = min(lo + block, n)
        A = attention_rows(Q, K, s, lo, hi)
        for p in range(3):  # sum_i sum_j A_ij [j in K^p]
            kept[p] += (A @ static[p][:hi].astype(np.float64)).sum()
        kept[3] += (A * (static[2][None, :hi] | local_rows_block(lo, hi, w))).sum()
    mass = [float(x / n) for x in kept] + [1.0]
    finals = final_sets(n, spec, punc, freq, w)
    cost = [int((f != DROP).sum()) for f in finals]
    p = choose_policy(mass, cost, T)
    return dict(policy=p, mass=np.array(mass), cost=np.array(cost), colsum=colsum,
                keep=finals[p], kept=cost[p], w=w, k=k, freq=freq)


# --- decode-time refresh of C_frequent (reading R13, off unless asked for) ---
# The pages define C_frequent by the largest cumulative attention scores and,
# in the stability paragraph, track accumulated attention over the prompt and
# later decoding steps; they reuse the prompt-time policy and state no rule
# for updating the frequent set while generating.  R13 is this build's own
# rule for such an update, available only on request (period > 0):
#   * every cached row j carries an accumulated score acc_j: its prompt
#     column sum colsum_j at the end of the prompt (0 for a generated token
#     when it is placed), plus, at every step, the attention weight the
#     step's query gives it (the softmax over the cache after placement);
#   * after every `period`-th generation step, the frequent members F (the
#     never-evicted rows kept for frequency, i.e. not special or punctuation
#     tokens) are re-chosen as the |F| rows of largest acc among F and the
#     non-special, non-punctuation rows of the current local window (ties to
#     the lower position); |F| never changes, so neither does the cache size;
#   * a member that loses its place leaves the cache, unless it is inside
#     the window, where it stays until it is w positions old like any window
#     row; a window row that wins a place stays in the cache for good;
#     dropped rows never return.
# Only local-hybrid caches have window rows to promote: for the other
# entries the refresh leaves the cache as profiled.

def accumulate_scores(acc, pos, weights):
    """acc_j += the step's attention weight of cached row j (R13)."""
    for j, a in zip(pos, weights):
        acc[int(j)] = acc.get(int(j), 0.0) + float(a)


def refresh_frequent(freq, window_candidates, acc):
    """R13: the |F| rows of largest accumulated score among the frequent
    members and the window candidates, ties to the lower position."""
    cand = sorted(set(freq) | set(window_candidates), key=lambda j: (-acc[j], j))
    return set(cand[:len(freq)])


def refresh_cache_positions(policy, static_sp, freq, w, t):
    """Cache positions at step t under R13: never-evicted special/punct
    members, the frequent members and, for the local hybrid, the window."""
    pos = set(int(p) for p in static_sp) | set(int(p) for p in freq)
    if policy == P_SPFL:
        pos.update(range(max(t - w + 1, 0), t + 1))
    return np.array(sorted(pos), dtype=np.int64)


def attention_weights(q, Kc, scale):
    """softmax(s q K_c^T) over the cache rows (the weights attend() applies)."""
    s = scale * (np.asarray(Kc, dtype=np.float64) @ np.asarray(q, dtype=np.float64))
    e = np.exp(s - s.max())
    return e / e.sum()


def decode_head_refresh(policy, keep, n, w, ids, Qall, Kall, Vall, special_ids, punct_ids,
                        steps, colsum, period, scale=None):
    """decode_head with the frequent set refreshed every `period` steps by
    R13 (period 0: never, which is decode_head).  colsum: the prompt's
    cumulative scores [n].  Returns dict(out [steps, d], pos: positions seen
    at the last step, final: the cache after the last refresh, acc: final
    accumulated scores of the cached rows, gaps: per refresh, the score gap
    between the last member kept and the best candidate left out, relative
    to max(1, score) (inf when nothing was left out))."""
    Kall = np.asarray(Kall, dtype=np.float64)
    Vall = np.asarray(Vall, dtype=np.float64)
    Qall = np.asarray(Qall, dtype=np.float64)
    d = Kall.shape[1]
    s = default_scale(d) if scale is None else scale
    sset, pset = set(int(x) for x in special_ids), set(int(x) for x in punct_ids)
    keep = np.asarray(keep)
    is_sp = lambda j: int(ids[j]) in sset or int(ids[j]) in pset
    static = [int(j) for j in np.nonzero(keep == KEEP_STATIC)[0]]
    uses_f = policy in (P_SPF, P_SPFL)
    static_sp = [j for j in static if is_sp(j) or not uses_f]
    freq = set(j for j in static if uses_f and not is_sp(j))
    acc = {int(j): float(colsum[j]) for j in np.nonzero(keep != DROP)[0]}
    out = np.zeros((steps, d))
    gaps = []
    pos = refresh_cache_positions(policy, static_sp, freq, w, n - 1)
    for step in range(steps):
        t = n + step
        tau = int(ids[t])
        if stores_static(policy, tau in sset, tau in pset):
            static_sp.append(t)
        pos = refresh_cache_positions(policy, static_sp, freq, w, t)
        if len(pos):
            acc.setdefault(t, 0.0)
            a = attention_weights(Qall[t], Kall[pos], s)
            out[step] = a @ Vall[pos]
            accumulate_scores(acc, pos, a)
        if period > 0 and uses_f and (step + 1) % period == 0:
            window = range(max(t - w + 1, 0), t + 1) if policy == P_SPFL else range(0)
            cands = [j for j in window if not is_sp(j)]
            new = refresh_frequent(freq, cands, acc)
            ranked = sorted(set(freq) | set(cands), key=lambda j: (-acc[j], j))
            kf = len(freq)
            if 0 < kf < len(ranked):
                hi, lo = acc[ranked[kf - 1]], acc[ranked[kf]]
                gaps.append((hi - lo) / max(1.0, hi))
            else:
                gaps.append(math.inf)
            freq = new
    final = refresh_cache_positions(policy, static_sp, freq, w, n + steps - 1)
    return dict(out=out, pos=pos, final=final,
                acc={int(j): acc[int(j)] for j in final}, gaps=gaps)
