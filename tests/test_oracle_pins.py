"""Pins of the oracle against what the FastGen pages and plain mathematics fix.

None of these checks re-types the oracle's own formulas: each compares it
with an independent route (hand-derived fixtures under tests/golden/, exact
fractions, 40-digit mpmath, pure-Python loops over the literal definitions,
a library sort, closed forms and invariants).  The last test plants plausible
mistakes in the oracle, one at a time, and requires that some pin fails.
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest

from oracle import fastgen_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ---------------------------------------------------------------------------
# independent, literal restatements used by the pins (pure Python loops)
# ---------------------------------------------------------------------------

def _py_attention(Q, K, scale):
    n = len(Q)
    A = [[0.0] * n for _ in range(n)]
    for i in range(n):
        s = [scale * sum(Q[i][c] * K[j][c] for c in range(len(Q[i]))) for j in range(i + 1)]
        m = max(s)
        e = [math.exp(x - m) for x in s]
        z = math.fsum(e)
        for j in range(i + 1):
            A[i][j] = e[j] / z
    return A


def _py_kept_sets(n, ids, special, punct, colsum, w, k):
    """Per-row kept sets of the four compressed shortlist entries, written
    from the policy descriptions with explicit loops."""
    spec = {j for j in range(n) if ids[j] in special}
    punc = {j for j in range(n) if ids[j] in punct}
    freq = set(sorted(range(n), key=lambda j: (-colsum[j], j))[:k])
    rows = []
    for i in range(n):
        local = {j for j in range(n) if i - w < j <= i}
        rows.append([spec, spec | punc, spec | punc | freq, spec | punc | freq | local])
    finals = [spec, spec | punc, spec | punc | freq,
              spec | punc | freq | set(range(max(n - w, 0), n)), set(range(n))]
    return rows, finals


def _py_half_l1(Q, K, scale, A, kept_rows_p):
    """mean over rows of (1/2)||A_i - softmax(q_i K_C^T)_i||_1, with the
    reconstruction built literally from the scores restricted to K_C."""
    n = len(Q)
    total = 0.0
    for i in range(n):
        kept = sorted(j for j in kept_rows_p[i] if j <= i)
        ahat = [0.0] * n
        if kept:
            s = [scale * sum(Q[i][c] * K[j][c] for c in range(len(Q[i]))) for j in kept]
            m = max(s)
            e = [math.exp(x - m) for x in s]
            z = math.fsum(e)
            for t, j in enumerate(kept):
                ahat[j] = e[t] / z
        total += 0.5 * math.fsum(abs(A[i][j] - ahat[j]) for j in range(n))
    return total / n


def _tiny_heads():
    """Small heads with varied structure: random, BOS-heavy, local-ish, ties."""
    rng = np.random.default_rng(1234)
    heads = []
    for trial in range(10):
        n = int(rng.integers(2, 15))
        d = 4
        Q = rng.standard_normal((n, d))
        K = rng.standard_normal((n, d))
        ids = rng.integers(2, 12, size=n)
        ids[0] = 1
        if trial % 3 == 1:  # make position 0 dominant
            u = rng.standard_normal(d)
            K[0] += 3 * u
            Q += 3 * u
        if trial % 3 == 2:  # nearly local
            K = Q + 0.1 * rng.standard_normal((n, d))
        r_l = [0.0, 0.2, 0.35, 0.5, 1.0][trial % 5]
        r_f = [0.3, 0.0, 0.5, 0.15, 1.0][trial % 5]
        heads.append((Q, K, ids, r_l, r_f))
    return heads


SPECIAL, PUNCT = [1], [5, 6]


# ---------------------------------------------------------------------------
# the pins
# ---------------------------------------------------------------------------

def pin_golden_three_token_map():
    g = _load("three_token_map.json")
    Q = np.array(g["q"])[:, None]
    K = np.array(g["k"])[:, None]
    A = O.attention_map(Q, K, g["scale"])
    for i, (row, den) in enumerate(zip(g["A_num"], g["A_den"])):
        for j, num in enumerate(row):
            assert abs(A[i, j] - num / den) < 1e-14, (i, j, A[i, j])
    colsum = O.cumulative_scores(A)
    for j, num in enumerate(g["colsum_num_over_21"]):
        assert abs(colsum[j] - num / 21) < 1e-14
    for T, want in g["policy_for_T"].items():
        r = O.profile_head(Q, K, np.array(g["ids"]), g["special_ids"], g["punct_ids"],
                           float(T), g["r_l"], g["r_f"], scale=g["scale"])
        assert r["w"] == g["w"] and r["k"] == g["k_count"]
        assert list(np.nonzero(r["freq"])[0]) == g["frequent"]
        assert list(r["cost"]) == g["cost"], r["cost"]
        for p, num in enumerate(g["mass_num_over_63"]):
            assert abs(r["mass"][p] - num / 63) < 1e-14, (p, r["mass"])
        assert r["policy"] == want, (T, r["policy"], want)
    # the half-L1 distance of the special-only cache on row 1 is 2/3
    row1 = A[1, :2]
    ahat = np.array([1.0, 0.0])
    assert abs(0.5 * np.abs(row1 - ahat).sum() - float(Fraction(g["half_l1_policy_S_row1"]))) < 1e-14


def pin_mpmath_attention():
    mp = pytest.importorskip("mpmath")
    mp.mp.dps = 40
    rng = np.random.default_rng(7)
    n, d = 8, 4
    Q = rng.standard_normal((n, d))
    K = rng.standard_normal((n, d))
    s = 1 / math.sqrt(d)
    A = O.attention_map(Q, K, s)
    for i in range(n):
        sc = [mp.mpf(s) * mp.fsum(mp.mpf(Q[i, c]) * mp.mpf(K[j, c]) for c in range(d))
              for j in range(i + 1)]
        z = mp.fsum(mp.exp(x) for x in sc)
        for j in range(n):
            want = mp.exp(sc[j]) / z if j <= i else mp.mpf(0)
            assert abs(A[i, j] - float(want)) < 1e-15, (i, j)
    # the default scale is 1/sqrt(d): profile_head's colsum equals the
    # column sums of the 40-digit map
    r = O.profile_head(Q, K, np.arange(n) + 100, SPECIAL, PUNCT, 0.9, 0.25, 0.25)
    for j in range(n):
        col = 0.0
        for i in range(j, n):
            sc = [mp.mpf(s) * mp.fsum(mp.mpf(Q[i, c]) * mp.mpf(K[jj, c]) for c in range(d))
                  for jj in range(i + 1)]
            col += float(mp.exp(sc[j]) / mp.fsum(mp.exp(x) for x in sc))
        assert abs(r["colsum"][j] - col) < 1e-13


def pin_half_l1_literal():
    """1 - mass_p equals the literal mean half-L1 distance of eq. (C*)."""
    for Q, K, ids, r_l, r_f in _tiny_heads():
        n, d = Q.shape
        s = 1 / math.sqrt(d)
        r = O.profile_head(Q, K, ids, SPECIAL, PUNCT, 0.9, r_l, r_f)
        A = _py_attention(Q.tolist(), K.tolist(), s)
        colsum = [math.fsum(A[i][j] for i in range(n)) for j in range(n)]
        w = math.ceil(float(np.float32(r_l)) * n)
        k = math.ceil(float(np.float32(r_f)) * n)
        rows, finals = _py_kept_sets(n, list(ids), set(SPECIAL), set(PUNCT), colsum, w, k)
        for p in range(4):
            dist = _py_half_l1(Q.tolist(), K.tolist(), s, A, [rw[p] for rw in rows])
            assert abs((1 - r["mass"][p]) - dist) < 1e-12, (p, 1 - r["mass"][p], dist)
        assert list(r["cost"]) == [len(f) for f in finals], (r["cost"], finals)


def pin_bruteforce_argmin():
    """The chosen policy is the argmin of cost over every entry whose literal
    distance is within 1 - T (enumerating all five)."""
    for Q, K, ids, r_l, r_f in _tiny_heads():
        n, d = Q.shape
        s = 1 / math.sqrt(d)
        A = _py_attention(Q.tolist(), K.tolist(), s)
        colsum = [math.fsum(A[i][j] for i in range(n)) for j in range(n)]
        w = math.ceil(float(np.float32(r_l)) * n)
        k = math.ceil(float(np.float32(r_f)) * n)
        rows, finals = _py_kept_sets(n, list(ids), set(SPECIAL), set(PUNCT), colsum, w, k)
        dist = [_py_half_l1(Q.tolist(), K.tolist(), s, A, [rw[p] for rw in rows]) for p in range(4)]
        dist.append(0.0)
        for T in (0.05, 0.5, 0.8, 0.9, 0.95, 0.99):
            if any(abs(x - (1 - T)) < 1e-9 for x in dist):
                continue
            feas = [p for p in range(5) if dist[p] <= 1 - T]
            want = min(feas, key=lambda p: (len(finals[p]), p))
            got = O.profile_head(Q, K, ids, SPECIAL, PUNCT, T, r_l, r_f)["policy"]
            assert got == want, (T, got, want, dist)


def pin_invariants():
    for Q, K, ids, r_l, r_f in _tiny_heads():
        n = Q.shape[0]
        r = O.profile_head(Q, K, ids, SPECIAL, PUNCT, 0.9, r_l, r_f)
        A = r["A"]
        assert np.allclose(A.sum(axis=1), 1.0, atol=1e-13, rtol=0)
        assert np.all(A[np.triu_indices(n, 1)] == 0)
        assert abs(r["colsum"].sum() - n) < 1e-12
        assert r["mass"][4] == 1.0
        full = O.kept_mass(A, np.ones((n, n), dtype=bool))
        assert abs(full - 1.0) < 1e-13
        assert np.all(np.diff(r["mass"]) >= -1e-15), r["mass"]
        assert np.all(np.diff(r["cost"]) >= 0), r["cost"]
        assert r["kept"] == r["cost"][r["policy"]] == int((r["keep"] != 0).sum())


def pin_planted_heads():
    """On the tiny workload a planted special-token head selects the
    special-only cache and a planted local head a local-containing one."""
    from synth import CONFIGS, head_types, make_head, make_ids, punct_ids, special_ids

    cfg = CONFIGS["tiny"]
    ids, types = make_ids(cfg), head_types(cfg)
    got = {}
    for g in range(cfg.G):
        Q, K, _ = make_head(cfg, 0, g, ids, types)
        r = O.profile_head(Q[:cfg.n], K[:cfg.n], ids[0], special_ids(), punct_ids(),
                           float(np.float32(cfg.T)), cfg.r_l, cfg.r_f)
        got[("special", "punct", "local", "broad")[types[0, g]]] = r["policy"]
    assert got["special"] == O.P_S, got
    assert got["local"] == O.P_SPFL, got


def pin_column_identity():
    """Per-row masses equal the column form, and the band sums equal their
    loop definition."""
    for Q, K, ids, r_l, r_f in _tiny_heads():
        n = Q.shape[0]
        r = O.profile_head(Q, K, ids, SPECIAL, PUNCT, 0.9, r_l, r_f)
        A, w = r["A"], r["w"]
        band = O.band_scores(A, w)
        for j in range(n):
            want = math.fsum(A[i, j] for i in range(j, min(j + w, n)))
            assert abs(band[j] - want) < 1e-14
        spec, punc = O.token_sets(ids, SPECIAL, PUNCT)
        col = O.masses_from_column_scores(r["colsum"], band, spec, punc, r["freq"])
        assert np.allclose(col, r["mass"], atol=1e-12, rtol=0), (col, r["mass"])


def pin_topk_sort():
    rng = np.random.default_rng(99)
    for trial in range(50):
        n = int(rng.integers(1, 40))
        c = rng.integers(0, 5, size=n).astype(np.float64) / 4  # many ties
        k = int(rng.integers(0, n + 1))
        want = set(sorted(range(n), key=lambda j: (-c[j], j))[:k])
        got = set(np.nonzero(O.frequent_set(c, k))[0].tolist())
        assert got == want, (c, k, got, want)


def pin_T_limits():
    for Q, K, ids, r_l, r_f in _tiny_heads():
        r = O.profile_head(Q, K, ids, SPECIAL, PUNCT, 1e-30, r_l, r_f)
        if r["mass"][0] > 0:
            assert r["policy"] == O.P_S
        r1 = O.profile_head(Q, K, ids, SPECIAL, PUNCT, 1.0, r_l, r_f)
        first_exact = min(p for p in range(5) if r1["mass"][p] == 1.0)
        assert r1["policy"] == first_exact


def pin_ratio_count():
    assert O.ratio_count(0.3, 128) == 39
    assert O.ratio_count(0.3, 2048) == 615
    assert O.ratio_count(0.25, 128) == 32
    assert O.ratio_count(0.0, 77) == 0
    assert O.ratio_count(1.0, 77) == 77
    assert O.ratio_count(0.1, 8192) == 820


def pin_decode_textbook_full():
    """A full-cache head attends over the whole history with plain softmax."""
    rng = np.random.default_rng(5)
    n, steps, d = 5, 4, 3
    Qa, Ka, Va = (rng.standard_normal((n + steps, d)) for _ in range(3))
    ids = np.array([1, 2, 3, 4, 5, 6, 7, 8, 9])
    keep = np.full(n, O.KEEP_STATIC, dtype=np.uint8)
    out, pos = O.decode_head(O.P_FULL, keep, n, 0, ids, Qa, Ka, Va, SPECIAL, PUNCT, steps)
    s = 1 / math.sqrt(d)
    for st in range(steps):
        t = n + st
        lg = [s * sum(Qa[t, c] * Ka[j, c] for c in range(d)) for j in range(t + 1)]
        m = max(lg)
        e = [math.exp(x - m) for x in lg]
        z = math.fsum(e)
        want = [math.fsum(e[j] / z * Va[j, c] for j in range(t + 1)) for c in range(d)]
        assert np.allclose(out[st], want, atol=1e-14, rtol=0)
    assert list(pos) == list(range(n + steps))


def pin_decode_small_caches():
    rng = np.random.default_rng(11)
    q = rng.standard_normal(6)
    Kc, Vc = rng.standard_normal((9, 6)), rng.standard_normal((9, 6))
    perm = rng.permutation(9)
    a = O.attend(q, Kc, Vc, 0.4)
    b = O.attend(q, Kc[perm], Vc[perm], 0.4)
    assert np.allclose(a, b, atol=1e-14, rtol=0)
    assert np.array_equal(O.attend(q, Kc[:1], Vc[:1], 0.4), Vc[0])
    assert np.array_equal(O.attend(q, Kc[:0], Vc[:0], 0.4), np.zeros(6))
    # two rows with logits 0 and ln 3 weigh 1/4 and 3/4
    q2 = np.array([math.log(3.0)])
    K2 = np.array([[0.0], [1.0]])
    V2 = np.array([[4.0], [8.0]])
    assert abs(O.attend(q2, K2, V2, 1.0)[0] - 7.0) < 1e-14


def pin_decode_window_golden():
    g = _load("decode_window.json")
    n, w = g["n"], g["w"]
    ids = np.zeros(11, dtype=np.int64) + 9
    for t, v in g["ids"].items():
        ids[int(t)] = v
    d = 2
    rng = np.random.default_rng(0)
    Qa, Ka, Va = (rng.standard_normal((11, d)) for _ in range(3))
    for p, per_t in g["expected"].items():
        p = int(p)
        keep = np.zeros(n, dtype=np.uint8)
        if p == O.P_FULL:
            keep[:] = O.KEEP_STATIC
        else:
            keep[g["static_prompt"]] = O.KEEP_STATIC
            if p == O.P_SPFL:
                keep[n - w:] = np.where(keep[n - w:] == 0, O.KEEP_WINDOW, keep[n - w:])
        for t, want in per_t.items():
            steps = int(t) - n + 1
            _, pos = O.decode_head(p, keep, n, w, ids, Qa, Ka, Va, g["special_ids"],
                                   g["punct_ids"], steps)
            assert list(pos) == want, (p, t, list(pos), want)


def pin_compact_order():
    rng = np.random.default_rng(3)
    K, V = rng.standard_normal((10, 2)), rng.standard_normal((10, 2))
    keep = np.array([1, 0, 2, 1, 0, 0, 2, 2, 1, 0], dtype=np.uint8)
    sp, wp, Ks, Vs, Kw, Vw = O.compact_head(K, V, keep)
    assert list(sp) == [0, 3, 8] and list(wp) == [2, 6, 7]
    assert np.array_equal(Ks, K[[0, 3, 8]]) and np.array_equal(Vw, V[[2, 6, 7]])


PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin):
    pin()


# ---------------------------------------------------------------------------
# planted mistakes: each must make at least one pin fail
# ---------------------------------------------------------------------------

def _mut_no_causal(Q, K, scale):
    S = scale * (np.asarray(Q, float) @ np.asarray(K, float).T)
    E = np.exp(S - S.max(axis=1, keepdims=True))
    return E / E.sum(axis=1, keepdims=True)


def _mut_rowsum(A):
    return A.sum(axis=1)


def _mut_ties_high(colsum, k):
    order = np.argsort(colsum, kind="stable")[::-1]
    m = np.zeros(colsum.shape[0], dtype=bool)
    m[order[:k]] = True
    return m


def _mut_local_wide(n, w):
    i = np.arange(n)[:, None]
    j = np.arange(n)[None, :]
    return (j <= i) & (j >= i - w)


def _mut_mass_nm1(A, row_mask):
    n = A.shape[0]
    return float((A * row_mask).sum() / max(n - 1, 1))


def _mut_choose_high(mass, cost, T):
    feasible = [p for p in range(5) if mass[p] >= T]
    return max(feasible, key=lambda p: (-cost[p], p))


def _mut_finals_short(n, spec, punc, freq, w):
    out = O._orig_final_sets(n, spec, punc, freq, max(w - 1, 0))
    return out


def _mut_sp_no_punct(policy, is_special, is_punct):
    if policy == O.P_FULL:
        return True
    return is_special


def _mut_window_open(policy, static_pos, w, t):
    pos = set(int(p) for p in static_pos)
    if policy == O.P_SPFL:
        pos.update(range(max(t - w + 1, 0), t))
    return np.array(sorted(pos), dtype=np.int64)


def _mut_attend_noscale(q, Kc, Vc, scale):
    return O._orig_attend(q, Kc, Vc, 1.0)


def _mut_round(r, n):
    return int(round(float(np.float32(r)) * n))


def _mut_scale_one(d):
    return 1.0


def _mut_band_short(A, w):
    return O._orig_band_scores(A, max(w - 1, 0))


MUTANTS = {
    "no_causal_mask": ("attention_map", _mut_no_causal),
    "colsum_over_rows": ("cumulative_scores", _mut_rowsum),
    "topk_ties_high": ("frequent_set", _mut_ties_high),
    "local_window_wide": ("local_rows", _mut_local_wide),
    "mass_over_n_minus_1": ("kept_mass", _mut_mass_nm1),
    "choose_costliest_tie": ("choose_policy", _mut_choose_high),
    "final_window_short": ("final_sets", _mut_finals_short),
    "decode_sp_ignores_punct": ("stores_static", _mut_sp_no_punct),
    "decode_window_excludes_t": ("decode_positions", _mut_window_open),
    "decode_missing_scale": ("attend", _mut_attend_noscale),
    "ratio_rounds": ("ratio_count", _mut_round),
    "scale_one": ("default_scale", _mut_scale_one),
    "band_short": ("band_scores", _mut_band_short),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name, monkeypatch):
    attr, fn = MUTANTS[name]
    for orig in ("final_sets", "attend", "band_scores"):
        monkeypatch.setattr(O, "_orig_" + orig, getattr(O, orig), raising=False)
    monkeypatch.setattr(O, attr, fn)
    failed = []
    for pin in PINS:
        try:
            pin()
        except (AssertionError, ValueError, IndexError):
            failed.append(pin.__name__)
    assert failed, f"mutant {name} passed every pin"
