"""Pins of the grouped-query extension of the oracle: a group of one is the
per-head path; the union, the group rule and the shared-cache attention
against hand-derived cases."""
import json
import os

import numpy as np

from oracle import fastgen_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_group_of_one_is_the_head_path():
    rng = np.random.default_rng(2)
    n, d, steps = 12, 4, 5
    Q, K, V = (rng.standard_normal((n + steps, d)) for _ in range(3))
    ids = rng.integers(2, 9, size=n + steps)
    ids[0] = 1
    r = O.profile_head(Q[:n], K[:n], ids, [1], [5], 0.9, 0.3, 0.3)
    members, keep, pol = O.profile_group([Q[:n]], K[:n], ids, [1], [5], 0.9, 0.3, 0.3)
    assert pol == r["policy"] and np.array_equal(keep, r["keep"])
    out1, pos1 = O.decode_head(r["policy"], r["keep"], n, r["w"], ids, Q, K, V, [1], [5], steps)
    outg, posg = O.decode_group(pol, keep, n, r["w"], ids, [Q], K, V, [1], [5], steps)
    assert np.array_equal(outg[0], out1) and np.array_equal(pos1, posg)


def test_union_codes():
    a = np.array([1, 0, 2, 0, 2, 1], dtype=np.uint8)
    b = np.array([0, 0, 1, 2, 2, 0], dtype=np.uint8)
    assert list(O.union_keep([a, b])) == [1, 0, 1, 2, 2, 1]
    assert np.array_equal(O.union_keep([a, a]), a)


def test_group_rule_matches_window_golden():
    """A special-only member and a local-hybrid member sharing a cache behave
    as the local hybrid on the union of their prompt caches."""
    g = json.load(open(os.path.join(GOLDEN, "decode_window.json")))
    n, w = g["n"], g["w"]
    ids = np.zeros(11, dtype=np.int64) + 9
    for t, v in g["ids"].items():
        ids[int(t)] = v
    keep_s = np.zeros(n, dtype=np.uint8)
    keep_s[0] = O.KEEP_STATIC
    keep_l = np.zeros(n, dtype=np.uint8)
    keep_l[g["static_prompt"]] = O.KEEP_STATIC
    keep_l[n - w:] = np.where(keep_l[n - w:] == 0, O.KEEP_WINDOW, keep_l[n - w:])
    keep = O.union_keep([keep_s, keep_l])
    pol = max(O.P_S, O.P_SPFL)
    rng = np.random.default_rng(0)
    Qa, Qb, Ka, Va = (rng.standard_normal((11, 2)) for _ in range(4))
    for t, want in g["expected"]["3"].items():
        steps = int(t) - n + 1
        out, pos = O.decode_group(pol, keep, n, w, ids, [Qa, Qb], Ka, Va, g["special_ids"],
                                  g["punct_ids"], steps)
        assert list(pos) == want
        # every member attends over the shared positions with its own query
        s = O.default_scale(2)
        assert np.allclose(out[1, -1], O.attend(Qb[int(t)], Ka[pos], Va[pos], s), atol=0, rtol=0)


def test_union_contains_every_member_cache():
    rng = np.random.default_rng(9)
    n, d = 16, 4
    K = rng.standard_normal((n, d))
    Qs = [rng.standard_normal((n, d)) for _ in range(4)]
    Qs[0] = Qs[0] + 3 * K[0]  # one member leaning on the first token
    ids = rng.integers(2, 9, size=n)
    ids[0] = 1
    members, keep, pol = O.profile_group(Qs, K, ids, [1], [5], 0.9, 0.25, 0.25)
    for m in members:
        assert np.all((keep != O.DROP) >= (m["keep"] != O.DROP))
        assert np.all((keep == O.KEEP_STATIC) >= (m["keep"] == O.KEEP_STATIC))
    assert pol == max(m["policy"] for m in members)


def test_planted_mistakes_fail_a_pin(monkeypatch):
    """Plausible mistakes in the grouped extension, one at a time: each must
    fail one of the pins above."""
    pins = (test_group_of_one_is_the_head_path, test_union_codes,
            test_group_rule_matches_window_golden, test_union_contains_every_member_cache)
    real_union, real_profile, real_attend = O.union_keep, O.profile_group, O.attend

    def window_beats_static(keeps):
        keeps = np.asarray(keeps)
        window = (keeps == O.KEEP_WINDOW).any(axis=0)
        static = (keeps == O.KEEP_STATIC).any(axis=0)
        return np.where(window, O.KEEP_WINDOW, np.where(static, O.KEEP_STATIC, O.DROP)).astype(
            np.uint8)

    def smallest_policy(Qs, K, ids, sp, pu, T, r_l, r_f, scale=None):
        members, keep, _ = real_profile(Qs, K, ids, sp, pu, T, r_l, r_f, scale)
        return members, keep, min(m["policy"] for m in members)

    def intersection(keeps):
        keeps = np.asarray(keeps)
        return np.where((keeps != O.DROP).all(axis=0), real_union(keeps), O.DROP).astype(np.uint8)

    for name, attr, bad in (("window beats static", "union_keep", window_beats_static),
                            ("smallest member policy", "profile_group", smallest_policy),
                            ("intersection of caches", "union_keep", intersection)):
        monkeypatch.setattr(O, attr, bad)
        failed = 0
        for pin in pins:
            try:
                pin()
            except AssertionError:
                failed += 1
        monkeypatch.setattr(O, attr, {"union_keep": real_union,
                                      "profile_group": real_profile}[attr])
        assert failed >= 1, name
    assert O.attend is real_attend
