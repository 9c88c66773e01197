"""Pins of the oracle's policy reuse with a saved head-policy map (reading
R11: a saved map fixes each head's shortlist entry; a later prompt's cache is
that entry's final set built from the prompt itself).

Independent routes: position-by-position Python loops over the definitions
of the base caches, a brute-force top-k with ties to the lower index, the
literal pure-Python attention map, and planted mistakes that must fail.
"""
import math

import numpy as np
import pytest

from oracle import fastgen_oracle as O
from test_oracle_pins import _py_attention

SPECIAL = [1, 2]
PUNCT = [7, 8, 9]


def _prompt(n, seed):
    rng = np.random.default_rng(seed)
    ids = rng.integers(10, 50, size=n)
    ids[0] = 1  # begin-of-sequence
    for j in rng.choice(np.arange(1, n), size=n // 5, replace=False):
        ids[j] = rng.choice(SPECIAL + PUNCT)
    return ids


def _expected(policy, ids, n, w, top):
    """Keep codes by a loop over positions, from the base-cache definitions."""
    out = []
    for j in range(n):
        s = int(ids[j]) in SPECIAL
        p = int(ids[j]) in PUNCT
        f = j in top
        if policy == O.P_S:
            st = s
        elif policy == O.P_SP:
            st = s or p
        elif policy in (O.P_SPF, O.P_SPFL):
            st = s or p or f
        else:
            st = True
        if st:
            out.append(O.KEEP_STATIC)
        elif policy == O.P_SPFL and j >= n - w:
            out.append(O.KEEP_WINDOW)
        else:
            out.append(O.DROP)
    return out


def _brute_topk(colsum, k):
    return set(sorted(range(len(colsum)), key=lambda j: (-float(colsum[j]), j))[:k])


def pin_closed_forms():
    n, r_l, r_f = 37, 0.3, 0.2
    w, k = math.ceil(np.float32(r_l) * n), math.ceil(np.float32(r_f) * n)
    ids = _prompt(n, 3)
    colsum = np.random.default_rng(5).random(n) * 3
    top = _brute_topk(colsum, k)
    for p in range(5):
        got = O.keep_for_policy(p, ids, SPECIAL, PUNCT, r_l, r_f, n, colsum)
        assert list(got) == _expected(p, ids, n, w, top), O.POLICIES[p]


def pin_ties_to_lower_index():
    n, r_f = 12, 0.25  # k = 3
    ids = np.full(n, 20)
    colsum = np.array([1, 5, 2, 5, 5, 0, 5, 1, 1, 0, 2, 2], dtype=np.float64)
    got = O.keep_for_policy(O.P_SPF, ids, SPECIAL, PUNCT, 0.0, r_f, n, colsum)
    assert list(np.nonzero(got == O.KEEP_STATIC)[0]) == [1, 3, 4]


def test_closed_forms_of_every_entry():
    pin_closed_forms()


def test_frequent_ties_go_to_the_lower_index():
    pin_ties_to_lower_index()


def test_scores_needed_only_for_frequent_entries():
    n = 9
    ids = _prompt(n, 1)
    for p in (O.P_S, O.P_SP, O.P_FULL):
        O.keep_for_policy(p, ids, SPECIAL, PUNCT, 0.3, 0.3, n)  # no colsum: fine
        r = O.profile_with_policy(p, np.ones((n, 4)), np.ones((n, 4)), ids, SPECIAL, PUNCT,
                                  0.3, 0.3)
        assert r["colsum"] is None
    for p in (O.P_SPF, O.P_SPFL):
        with pytest.raises(ValueError):
            O.keep_for_policy(p, ids, SPECIAL, PUNCT, 0.3, 0.3, n)


def test_frequent_entry_uses_the_literal_column_sums():
    """The scores of an F entry are the column sums of the literal causal map."""
    rng = np.random.default_rng(11)
    n, d = 14, 4
    Q, K = rng.standard_normal((n, d)), rng.standard_normal((n, d))
    ids = _prompt(n, 2)
    A = _py_attention(Q.tolist(), K.tolist(), 1 / math.sqrt(d))
    cs = [math.fsum(A[i][j] for i in range(n)) for j in range(n)]
    r = O.profile_with_policy(O.P_SPFL, Q, K, ids, SPECIAL, PUNCT, 0.25, 0.3)
    assert np.allclose(r["colsum"], cs, rtol=0, atol=1e-12)
    w, k = math.ceil(np.float32(0.25) * n), math.ceil(np.float32(0.3) * n)
    assert list(r["keep"]) == _expected(O.P_SPFL, ids, n, w, _brute_topk(cs, k))
    assert r["kept"] == sum(1 for c in r["keep"] if c != O.DROP)


def test_saved_choice_reproduces_the_profiled_cache():
    """Applying each head's own profiled policy to the same prompt gives the
    cache that profiling chose."""
    rng = np.random.default_rng(4)
    n, d = 40, 8
    ids = _prompt(n, 4)
    seen = set()
    for T in np.linspace(0.05, 0.99, 12):
        Q = rng.standard_normal((n, d)) * 2
        K = rng.standard_normal((n, d))
        r = O.profile_head(Q, K, ids, SPECIAL, PUNCT, float(T), 0.3, 0.3)
        again = O.profile_with_policy(r["policy"], Q, K, ids, SPECIAL, PUNCT, 0.3, 0.3)
        assert np.array_equal(again["keep"], r["keep"])
        seen.add(r["policy"])
    assert len(seen) >= 3, seen


@pytest.mark.parametrize("mistake", ["window_off_by_one", "ties_to_higher", "s_keeps_punct"])
def test_planted_mistakes_fail_a_pin(monkeypatch, mistake):
    if mistake == "window_off_by_one":
        real = O.final_sets
        monkeypatch.setattr(O, "final_sets", lambda n, s, p, f, w: real(n, s, p, f, w + 1))
    elif mistake == "ties_to_higher":
        def bad(colsum, k):
            order = np.lexsort((-np.arange(colsum.shape[0]), -colsum))
            m = np.zeros(colsum.shape[0], dtype=bool)
            m[order[:k]] = True
            return m
        monkeypatch.setattr(O, "frequent_set", bad)
    else:
        real_sets = O.token_sets
        monkeypatch.setattr(O, "token_sets",
                            lambda ids, sp, pu: (lambda a: (a[0] | a[1], a[1]))(real_sets(ids, sp, pu)))
    failed = 0
    for pin in (pin_closed_forms, pin_ties_to_lower_index):
        try:
            pin()
        except AssertionError:
            failed += 1
    assert failed >= 1, mistake
