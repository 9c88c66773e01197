"""Pins of the oracle's long-prompt profile (profile_head_long), which forms
the attention map a block of query rows at a time so that 32k-token prompts
fit in host memory.  It must give exactly what the dense definition gives
(the hand-derived 3-token fixture, a literal loop of the causal softmax, the
dense profile_head on many small heads and block sizes, ragged last blocks
included), and plausible mistakes in it must fail one of these pins."""
import json
import math
import os

import numpy as np
import pytest

from oracle import fastgen_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
SPECIAL, PUNCT = [1], [5, 6]


def _heads():
    rng = np.random.default_rng(4321)
    out = []
    for trial in range(12):
        n = int(rng.integers(1, 40))
        d = 4
        Q = rng.standard_normal((n, d))
        K = rng.standard_normal((n, d))
        ids = rng.integers(2, 12, size=n)
        ids[0] = 1
        if trial % 3 == 1:
            u = rng.standard_normal(d)
            K[0] += 3 * u
            Q += 3 * u
        if trial % 3 == 2:
            K = Q + 0.1 * rng.standard_normal((n, d))
        r_l = [0.0, 0.2, 0.35, 0.5, 1.0, 0.1][trial % 6]
        r_f = [0.3, 0.0, 0.5, 0.15, 1.0, 0.2][trial % 6]
        out.append((Q, K, ids, r_l, r_f))
    return out


def pin_long_equals_dense():
    """Every output equals the dense profile's, for blocks of one row, of a
    few rows (ragged last block) and of the whole prompt."""
    for Q, K, ids, r_l, r_f in _heads():
        n = Q.shape[0]
        for T in (0.5, 0.9, 0.99):
            want = O.profile_head(Q, K, ids, SPECIAL, PUNCT, T, r_l, r_f)
            for block in (1, 3, 7, n):
                got = O.profile_head_long(Q, K, ids, SPECIAL, PUNCT, T, r_l, r_f, block=block)
                assert np.abs(got["colsum"] - want["colsum"]).max() < 1e-13, block
                assert np.abs(got["mass"] - want["mass"]).max() < 1e-13, (block, got["mass"])
                for key in ("policy", "kept", "w", "k"):
                    assert got[key] == want[key], (key, block)
                for key in ("cost", "keep", "freq"):
                    assert np.array_equal(got[key], want[key]), (key, block)


def pin_long_golden_three_token_map():
    """The hand-derived 3-token head (exact fractions) with blocks of 1 and 2 rows."""
    with open(os.path.join(GOLDEN, "three_token_map.json")) as f:
        g = json.load(f)
    Q = np.array(g["q"])[:, None]
    K = np.array(g["k"])[:, None]
    for block in (1, 2):
        for T, want in g["policy_for_T"].items():
            r = O.profile_head_long(Q, K, np.array(g["ids"]), g["special_ids"], g["punct_ids"],
                                    float(T), g["r_l"], g["r_f"], scale=g["scale"], block=block)
            for j, num in enumerate(g["colsum_num_over_21"]):
                assert abs(r["colsum"][j] - num / 21) < 1e-14, (block, j)
            for p, num in enumerate(g["mass_num_over_63"]):
                assert abs(r["mass"][p] - num / 63) < 1e-14, (block, p, r["mass"])
            assert list(r["cost"]) == g["cost"]
            assert list(np.nonzero(r["freq"])[0]) == g["frequent"]
            assert r["policy"] == want, (block, T, r["policy"])


def pin_attention_rows_literal():
    """A block of rows equals the causal softmax written as a loop."""
    rng = np.random.default_rng(8)
    n, d, s = 11, 3, 0.7
    Q, K = rng.standard_normal((n, d)), rng.standard_normal((n, d))
    for lo, hi in ((0, 1), (2, 6), (5, 11), (10, 11)):
        A = O.attention_rows(Q, K, s, lo, hi)
        assert A.shape == (hi - lo, hi)
        for i in range(lo, hi):
            lg = [s * math.fsum(Q[i, c] * K[j, c] for c in range(d)) for j in range(i + 1)]
            m = max(lg)
            e = [math.exp(x - m) for x in lg]
            z = math.fsum(e)
            for j in range(hi):
                want = e[j] / z if j <= i else 0.0
                assert abs(A[i - lo, j] - want) < 1e-15, (i, j)


def pin_local_rows_block_literal():
    for lo, hi, w in ((0, 5, 0), (0, 5, 1), (3, 9, 2), (4, 7, 10)):
        m = O.local_rows_block(lo, hi, w)
        for i in range(lo, hi):
            for j in range(hi):
                assert m[i - lo, j] == (i - w < j <= i), (lo, hi, w, i, j)


PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin):
    pin()


# --- planted mistakes: each must make at least one pin fail -----------------

def _mut_rows_no_mask(Q, K, scale, lo, hi):
    S = scale * (Q[lo:hi] @ K[:hi].T)
    S = S - S.max(axis=1, keepdims=True)
    E = np.exp(S)
    return E / E.sum(axis=1, keepdims=True)


def _mut_rows_diag_masked(Q, K, scale, lo, hi):
    S = scale * (Q[lo:hi] @ K[:hi].T)
    i = np.arange(lo, hi)[:, None]
    j = np.arange(hi)[None, :]
    S[(j >= i) & (j > 0)] = -np.inf
    S = S - S.max(axis=1, keepdims=True)
    E = np.exp(S)
    return E / E.sum(axis=1, keepdims=True)


def _mut_local_wide(lo, hi, w):
    i = np.arange(lo, hi)[:, None]
    j = np.arange(hi)[None, :]
    return (j <= i) & (j >= i - w)


def _mut_local_absolute(lo, hi, w):
    # the window measured from the block start instead of each row
    j = np.arange(hi)[None, :]
    i = np.arange(lo, hi)[:, None]
    return (j <= i) & (j > lo - w)


MUTANTS = {
    "rows_without_causal_mask": ("attention_rows", _mut_rows_no_mask),
    "rows_mask_the_diagonal": ("attention_rows", _mut_rows_diag_masked),
    "local_block_wide": ("local_rows_block", _mut_local_wide),
    "local_block_from_block_start": ("local_rows_block", _mut_local_absolute),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name, monkeypatch):
    attr, fn = MUTANTS[name]
    monkeypatch.setattr(O, attr, fn)
    failed = []
    for pin in PINS:
        try:
            pin()
        except (AssertionError, ValueError, IndexError):
            failed.append(pin.__name__)
    assert failed, f"mutant {name} passed every pin"
