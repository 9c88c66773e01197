"""Pins of the oracle's prompt attention output O = A V (causal A =
softmax(s Q K^T)): a hand-derived fixture, a literal pure-Python loop,
closed forms (constant value rows, one-hot values), causality, and planted
mistakes that must fail one of them."""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest

from oracle import fastgen_oracle as O
from test_oracle_pins import _py_attention

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def pin_golden():
    with open(os.path.join(GOLDEN, "three_token_output.json")) as f:
        g = json.load(f)
    Q = np.array(g["q"])[:, None]
    K = np.array(g["k"])[:, None]
    out = O.prompt_attention(Q, K, np.array(g["v"]), scale=g["scale"])
    for i, (row, den) in enumerate(zip(g["O_num"], g["O_den"])):
        for c, num in enumerate(row):
            assert abs(out[i, c] - float(Fraction(num, den))) < 1e-14, (i, c, out[i, c])


def pin_literal_loop():
    rng = np.random.default_rng(7)
    n, d, dv = 9, 3, 4
    Q, K, V = rng.standard_normal((n, d)), rng.standard_normal((n, d)), rng.standard_normal((n, dv))
    A = _py_attention(Q.tolist(), K.tolist(), 0.7)
    want = [[math.fsum(A[i][j] * V[j][c] for j in range(n)) for c in range(dv)] for i in range(n)]
    got = O.prompt_attention(Q, K, V, scale=0.7)
    assert np.allclose(got, want, rtol=0, atol=1e-13)


def pin_closed_forms():
    rng = np.random.default_rng(8)
    n, d = 11, 5
    Q, K = rng.standard_normal((n, d)) * 2, rng.standard_normal((n, d))
    # every value row equal: every output row is that row (rows of A sum to 1)
    c = rng.standard_normal(6)
    assert np.allclose(O.prompt_attention(Q, K, np.tile(c, (n, 1))), np.tile(c, (n, 1)),
                       rtol=0, atol=1e-13)
    # one-hot values (V = I): the output is the attention map itself, which
    # is causal and row-stochastic
    out = O.prompt_attention(Q, K, np.eye(n))
    assert np.allclose(np.triu(out, 1), 0.0) and np.allclose(out.sum(axis=1), 1.0)
    assert abs(out[0, 0] - 1.0) < 1e-15


def pin_causal():
    rng = np.random.default_rng(9)
    n, d = 10, 4
    Q, K, V = (rng.standard_normal((n, d)) for _ in range(3))
    V2 = V.copy()
    V2[6:] += 5.0
    a, b = O.prompt_attention(Q, K, V), O.prompt_attention(Q, K, V2)
    assert np.allclose(a[:6], b[:6], rtol=0, atol=0)
    assert not np.allclose(a[6:], b[6:])


PINS = (pin_golden, pin_literal_loop, pin_closed_forms, pin_causal)


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin()


@pytest.mark.parametrize("mistake", ["no_mask", "transposed_map", "unscaled"])
def test_planted_mistakes_fail_a_pin(monkeypatch, mistake):
    real = O.attention_map
    if mistake == "no_mask":
        def bad(Q, K, scale):
            S = scale * (Q @ K.T)
            E = np.exp(S - S.max(axis=1, keepdims=True))
            return E / E.sum(axis=1, keepdims=True)
    elif mistake == "transposed_map":
        def bad(Q, K, scale):
            return real(Q, K, scale).T
    else:
        def bad(Q, K, scale):
            return real(Q, K, 1.0)
    monkeypatch.setattr(O, "attention_map", bad)
    failed = 0
    for pin in PINS:
        try:
            pin()
        except AssertionError:
            failed += 1
    assert failed >= 1, mistake
