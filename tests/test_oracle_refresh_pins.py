"""Pins of the oracle's decode-time refresh of C_frequent (reading R13; the
pages give no refresh rule, so the rule is pinned to its own statement and
to mathematics): a hand-derived fixture with exact fractions, the frozen path
when no refresh happens, the accumulated score as a literal sum over steps,
the no-op on caches without a window, and the ranking property after a
refresh.  Plausible mistakes in each helper must fail one of these pins."""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest

from oracle import fastgen_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
SPECIAL, PUNCT = [1], [5, 6]


def _fixture():
    with open(os.path.join(GOLDEN, "refresh_window.json")) as f:
        g = json.load(f)
    total = len(g["ids"])
    K = np.array([[math.log(c)] for c in g["c"]])
    Q = np.ones((total, 1))
    V = np.arange(total, dtype=np.float64)[:, None]
    colsum = np.array([float(Fraction(x)) for x in g["colsum"]])
    return g, Q, K, V, colsum


def _heads(seed=17, count=12):
    """Small generation problems with every policy; ids drawn so that some
    generated tokens are special or punctuation."""
    rng = np.random.default_rng(seed)
    out = []
    for trial in range(count):
        n = int(rng.integers(3, 24))
        steps = int(rng.integers(1, 14))
        d = 3
        Qa, Ka, Va = (rng.standard_normal((n + steps, d)) for _ in range(3))
        ids = rng.integers(2, 12, size=n + steps)
        ids[0] = 1
        r_l = [0.2, 0.35, 0.5, 0.1][trial % 4]
        r_f = [0.3, 0.25, 0.5, 0.2][trial % 4]
        T = [0.5, 0.9, 0.99, 0.7][trial % 4]
        prof = O.profile_head(Qa[:n], Ka[:n], ids, SPECIAL, PUNCT, T, r_l, r_f)
        out.append((prof, n, steps, ids, Qa, Ka, Va))
    return out


def _local_head(seed):
    """A local-hybrid head with a non-empty window and frequent set: T is
    set between the masses of the entries without and with the window."""
    rng = np.random.default_rng(seed)
    n, steps, d = 16, 12, 3
    Qa, Ka, Va = (rng.standard_normal((n + steps, d)) for _ in range(3))
    ids = rng.integers(2, 12, size=n + steps)
    ids[0] = 1
    m = O.profile_head(Qa[:n], Ka[:n], ids, SPECIAL, PUNCT, 0.5, 0.25, 0.25)["mass"]
    prof = O.profile_head(Qa[:n], Ka[:n], ids, SPECIAL, PUNCT, (m[2] + m[3]) / 2, 0.25, 0.25)
    assert prof["policy"] == O.P_SPFL, m
    return prof, n, steps, ids, Qa, Ka, Va


def pin_golden_refresh():
    g, Q, K, V, colsum = _fixture()
    n, w = g["n"], g["w"]
    keep = np.array(g["keep"], dtype=np.uint8)
    for t, want in g["positions_seen"].items():
        steps = int(t) - n + 1
        r = O.decode_head_refresh(O.P_SPFL, keep, n, w, np.array(g["ids"]), Q, K, V,
                                  g["special_ids"], g["punct_ids"], steps, colsum, g["period"],
                                  scale=1.0)
        assert list(r["pos"]) == want, (t, list(r["pos"]), want)
    r = O.decode_head_refresh(O.P_SPFL, keep, n, w, np.array(g["ids"]), Q, K, V,
                              g["special_ids"], g["punct_ids"], g["steps"], colsum, g["period"],
                              scale=1.0)
    for st, want in enumerate(g["out"]):
        assert abs(r["out"][st, 0] - float(Fraction(want))) < 1e-13, (st, r["out"][st, 0])
    assert list(r["final"]) == g["final_cache"]
    assert sorted(r["acc"]) == sorted(int(j) for j in g["final_acc"])
    for j, want in g["final_acc"].items():
        assert abs(r["acc"][int(j)] - float(Fraction(want))) < 1e-13, (j, r["acc"][int(j)])
    f = O.decode_head_refresh(O.P_SPFL, keep, n, w, np.array(g["ids"]), Q, K, V,
                              g["special_ids"], g["punct_ids"], g["steps"], colsum, 0, scale=1.0)
    for st, want in enumerate(g["frozen_out"]):
        assert abs(f["out"][st, 0] - float(Fraction(want))) < 1e-13, (st, f["out"][st, 0])


def pin_period_zero_is_the_frozen_path():
    for prof, n, steps, ids, Qa, Ka, Va in _heads():
        want, pos = O.decode_head(prof["policy"], prof["keep"], n, prof["w"], ids, Qa, Ka, Va,
                                  SPECIAL, PUNCT, steps)
        for period in (0, steps + 1):  # off, or on but never reached
            r = O.decode_head_refresh(prof["policy"], prof["keep"], n, prof["w"], ids, Qa, Ka,
                                      Va, SPECIAL, PUNCT, steps, prof["colsum"], period)
            assert np.array_equal(r["out"], want), period
            assert np.array_equal(r["pos"], pos) and np.array_equal(r["final"], pos)


def pin_accumulated_score_is_the_literal_sum():
    """Without a refresh, acc_j = colsum_j + sum over steps of the weight a
    literal softmax loop gives row j (0 before a generated row is placed)."""
    for prof, n, steps, ids, Qa, Ka, Va in _heads(seed=23):
        w, s = prof["w"], 1 / math.sqrt(Qa.shape[1])
        r = O.decode_head_refresh(prof["policy"], prof["keep"], n, w, ids, Qa, Ka, Va, SPECIAL,
                                  PUNCT, steps, prof["colsum"], steps + 1)
        want = {}
        for j in range(n + steps):
            total = [float(prof["colsum"][j])] if j < n else []
            for st in range(steps):
                t = n + st
                _, pos = O.decode_head(prof["policy"], prof["keep"], n, w, ids, Qa, Ka, Va,
                                       SPECIAL, PUNCT, st + 1)
                pos = [int(x) for x in pos]
                if j not in pos:
                    continue
                lg = [s * math.fsum(Qa[t, c] * Ka[p, c] for c in range(Qa.shape[1]))
                      for p in pos]
                m = max(lg)
                z = math.fsum(math.exp(x - m) for x in lg)
                total.append(math.exp(lg[pos.index(j)] - m) / z)
            want[j] = math.fsum(total)
        for j, got in r["acc"].items():
            assert abs(got - want[j]) < 1e-12, (j, got, want[j])


def pin_no_window_means_no_change():
    """Entries without a window (special+punct+frequent) have no candidate
    outside their frequent set: the refresh leaves them as profiled."""
    rng = np.random.default_rng(31)
    n, steps, d = 14, 9, 3
    Qa, Ka, Va = (rng.standard_normal((n + steps, d)) for _ in range(3))
    ids = rng.integers(2, 12, size=n + steps)
    ids[0] = 1
    prof = O.profile_head(Qa[:n], Ka[:n], ids, SPECIAL, PUNCT, 0.9, 0.3, 0.3)
    keep = O.keep_for_policy(O.P_SPF, ids, SPECIAL, PUNCT, 0.3, 0.3, n, prof["colsum"])
    want, pos = O.decode_head(O.P_SPF, keep, n, prof["w"], ids, Qa, Ka, Va, SPECIAL, PUNCT, steps)
    r = O.decode_head_refresh(O.P_SPF, keep, n, prof["w"], ids, Qa, Ka, Va, SPECIAL, PUNCT,
                              steps, prof["colsum"], 1)
    assert np.array_equal(r["out"], want) and np.array_equal(r["final"], pos)


def pin_refresh_ranks_members_above_candidates():
    """Right after a refresh the frequent members outrank (or tie at a
    higher position with) every window candidate left out, their number is
    unchanged, and the cache never grows past the frozen path's."""
    for seed in range(6):
        prof, n, steps, ids, Qa, Ka, Va = _local_head(seed)
        w = prof["w"]
        sp = set(SPECIAL) | set(PUNCT)
        kf = sum(1 for j in np.nonzero(prof["keep"] == O.KEEP_STATIC)[0] if ids[j] not in sp)
        for period in (1, 2, 3):
            k = steps - steps % period  # the last refresh step
            r = O.decode_head_refresh(O.P_SPFL, prof["keep"], n, w, ids, Qa, Ka, Va, SPECIAL,
                                      PUNCT, k, prof["colsum"], period)
            t = n + k - 1
            window = set(range(max(t - w + 1, 0), t + 1))
            static_sp = {j for j in r["final"] if ids[j] in sp}
            members = set(r["final"]) - static_sp - window
            in_window = [j for j in window if ids[j] not in sp]
            # members outside the window plus the best-ranked window rows make up |F|
            cands = sorted(in_window, key=lambda j: (-r["acc"][j], j))
            assert len(members) <= kf
            chosen = members | set(cands[:kf - len(members)])
            assert len(chosen) == kf or len(cands) < kf - len(members)
            left = [j for j in in_window if j not in chosen]
            for m in chosen:
                for c in left:
                    assert (r["acc"][m], -m) > (r["acc"][c], -c), (m, c)
            _, frozen = O.decode_head(O.P_SPFL, prof["keep"], n, w, ids, Qa, Ka, Va, SPECIAL,
                                      PUNCT, k)
            assert len(r["final"]) <= len(frozen)


def pin_ties_go_to_the_lower_position():
    """Hand-made ties: equal scores keep the earlier position."""
    assert O.refresh_frequent({7}, [5, 9], {5: 1.0, 7: 1.0, 9: 1.0}) == {5}
    assert O.refresh_frequent({2, 8}, [3], {2: 0.5, 3: 0.5, 8: 0.5}) == {2, 3}
    assert O.refresh_frequent({4}, [6], {4: 0.25, 6: 0.75}) == {6}
    assert O.refresh_frequent(set(), [1, 2], {1: 3.0, 2: 4.0}) == set()


PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin):
    pin()


# --- planted mistakes ----------------------------------------------------------

def _mut_acc_double(acc, pos, weights):
    for j, a in zip(pos, weights):
        acc[int(j)] = acc.get(int(j), 0.0) + 2.0 * float(a)


def _mut_ties_high(freq, window_candidates, acc):
    cand = sorted(set(freq) | set(window_candidates), key=lambda j: (-acc[j], -j))
    return set(cand[:len(freq)])


def _mut_members_only(freq, window_candidates, acc):
    return set(freq)


def _mut_one_more(freq, window_candidates, acc):
    cand = sorted(set(freq) | set(window_candidates), key=lambda j: (-acc[j], j))
    return set(cand[:len(freq) + 1])


def _mut_lowest(freq, window_candidates, acc):
    cand = sorted(set(freq) | set(window_candidates), key=lambda j: (acc[j], j))
    return set(cand[:len(freq)])


def _mut_positions_without_freq(policy, static_sp, freq, w, t):
    pos = set(int(p) for p in static_sp)
    if policy == O.P_SPFL:
        pos.update(range(max(t - w + 1, 0), t + 1))
    return np.array(sorted(pos), dtype=np.int64)


def _mut_weights_unnormalised(q, Kc, scale):
    s = scale * (np.asarray(Kc, dtype=np.float64) @ np.asarray(q, dtype=np.float64))
    return np.exp(s - s.max())


MUTANTS = {
    "accumulates_twice": ("accumulate_scores", _mut_acc_double),
    "ties_to_higher_position": ("refresh_frequent", _mut_ties_high),
    "window_never_competes": ("refresh_frequent", _mut_members_only),
    "frequent_set_grows": ("refresh_frequent", _mut_one_more),
    "keeps_the_lowest": ("refresh_frequent", _mut_lowest),
    "members_not_attended": ("refresh_cache_positions", _mut_positions_without_freq),
    "weights_not_normalised": ("attention_weights", _mut_weights_unnormalised),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name, monkeypatch):
    attr, fn = MUTANTS[name]
    monkeypatch.setattr(O, attr, fn)
    failed = []
    for pin in PINS:
        try:
            pin()
        except (AssertionError, ValueError, IndexError, KeyError):
            failed.append(pin.__name__)
    assert failed, f"mutant {name} passed every pin"
