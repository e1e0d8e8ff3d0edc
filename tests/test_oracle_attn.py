"""Pins of the oracle's head-parallel attention block (CPU only)."""
import math

import numpy as np
import pytest

import oracle
from _golden import read_kv


def _problem(seed, b=2, s=5, h=8, heads=2):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal((b * s, h)), rng.standard_normal((h, 3 * h)) * 0.4,
            rng.standard_normal((h, h)) * 0.4, b, s, heads)


def _brute(X, Wqkv, Wo, heads, b, s):
    T, h = len(X), len(X[0])
    d = h // heads
    mm = lambda A, B: [[sum(A[i][k] * B[k][j] for k in range(len(B))) for j in range(len(B[0]))] for i in range(len(A))]
    QKV = mm(X, Wqkv)
    O = [[0.0] * h for _ in range(T)]
    for q in range(b):
        for j in range(heads):
            for i in range(s):
                r = q * s + i
                sc = []
                for k in range(i + 1):
                    c = q * s + k
                    sc.append(sum(QKV[r][j * d + e] * QKV[c][h + j * d + e] for e in range(d)) / math.sqrt(d))
                mx = max(sc)
                w = [math.exp(x - mx) for x in sc]
                tot = sum(w)
                for e in range(d):
                    O[r][j * d + e] = sum(w[k] / tot * QKV[q * s + k][2 * h + j * d + e] for k in range(i + 1))
    return np.array(mm(O, Wo))


def test_brute_force():
    X, Wqkv, Wo, b, s, heads = _problem(1)
    _, _, out = oracle.attn_fwd(X, Wqkv, Wo, heads, b, s)
    np.testing.assert_allclose(out, _brute(X.tolist(), Wqkv.tolist(), Wo.tolist(), heads, b, s), rtol=1e-12,
                               atol=1e-12)


@pytest.mark.parametrize("t", [1, 2, 4])
def test_head_sharding_invariance(t):
    X, Wqkv, Wo, b, s, heads = _problem(2, b=2, s=6, h=16, heads=4)
    _, _, out = oracle.attn_fwd(X, Wqkv, Wo, heads, b, s)
    sh, parts = oracle.attn_fwd_sharded(X, Wqkv, Wo, heads, b, s, t)
    assert np.linalg.norm(sh - out) <= 1e-12 * np.linalg.norm(out)
    if t > 1:
        assert not np.allclose(parts[0], out)


def test_zero_queries_average_the_prefix():
    # Q = 0: every score is 0, so each query averages the values of its causal prefix.
    rng = np.random.default_rng(3)
    b, s, h, heads = 1, 7, 6, 2
    Q = np.zeros((s, h))
    K = rng.standard_normal((s, h))
    V = rng.standard_normal((s, h))
    O = oracle.attention_heads(Q, K, V, heads, b, s)
    want = np.cumsum(V, axis=0) / np.arange(1, s + 1)[:, None]
    np.testing.assert_allclose(O, want, rtol=1e-13, atol=1e-14)


def test_causality():
    X, Wqkv, Wo, b, s, heads = _problem(4, b=1, s=8, h=8, heads=2)
    _, _, out = oracle.attn_fwd(X, Wqkv, Wo, heads, b, s)
    X2 = X.copy()
    X2[5:] += 3.0                           # change only tokens 5..7
    _, _, out2 = oracle.attn_fwd(X2, Wqkv, Wo, heads, b, s)
    np.testing.assert_array_equal(out[:5], out2[:5])
    assert not np.allclose(out[5:], out2[5:])


def test_causality_rejects_off_by_one_mask():
    # Planted mistake: a mask that also hides the diagonal changes the first token's output.
    rng = np.random.default_rng(5)
    s, h = 4, 4
    Q, K, V = (rng.standard_normal((s, h)) for _ in range(3))
    good = oracle.attention_heads(Q, K, V, 1, 1, s)
    S = Q @ K.T / 2.0
    S[np.triu(np.ones((s, s), dtype=bool), k=0)] = -np.inf   # k=0: diagonal masked too
    S[0, 0] = 0.0                                             # keep row 0 finite
    P = np.exp(S - S.max(axis=1, keepdims=True))
    wrong = (P / P.sum(axis=1, keepdims=True)) @ V
    assert not np.allclose(wrong, good)


def test_sampled_rows_match_full():
    X, Wqkv, Wo, b, s, heads = _problem(6, b=3, s=9, h=12, heads=3)
    _, O, out = oracle.attn_fwd(X, Wqkv, Wo, heads, b, s)
    rows = np.array([0, 8, 9, 17, 26])
    Or, outr = oracle.attn_fwd_rows(X, Wqkv, Wo, heads, b, s, rows)
    np.testing.assert_allclose(Or, O[rows], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(outr, out[rows], rtol=1e-12, atol=1e-13)


def test_head_width_arithmetic():
    g = read_kv("attention_heads.txt")
    heads, gpus, hidden = int(g["heads"][0]), int(g["gpus"][0]), int(g["hidden"][0])
    assert heads // gpus == int(g["heads_per_gpu"][0]) and hidden // heads == int(g["head_width"][0])
