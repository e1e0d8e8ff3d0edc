"""Pins of the oracle's vocab-parallel cross-entropy (CPU only)."""
import math

import numpy as np
import pytest

import oracle
from _golden import read_kv


def _brute(X, E, target, v_valid):
    # -log softmax(z)[target] by direct enumeration in pure Python.
    out = []
    for r in range(len(X)):
        z = [sum(X[r][k] * E[c][k] for k in range(len(X[r]))) for c in range(v_valid)]
        den = sum(math.exp(zc) for zc in z)
        out.append(-math.log(math.exp(z[target[r]]) / den))
    return out


@pytest.mark.parametrize("v", [2, 3, 4, 7, 16])
def test_brute_force_tiny_vocab(v):
    rng = np.random.default_rng(v)
    T, h = 5, min(8, v + 1)
    X = rng.standard_normal((T, h))
    E = rng.standard_normal((v, h)) * 0.7
    tgt = rng.integers(0, v, T)
    got = oracle.ce_loss(X, E, tgt, v)
    np.testing.assert_allclose(got, _brute(X.tolist(), E.tolist(), tgt.tolist(), v), rtol=1e-12, atol=1e-12)


def test_padding_rows_excluded():
    rng = np.random.default_rng(2)
    X = rng.standard_normal((4, 6))
    E = rng.standard_normal((12, 6))
    tgt = np.array([0, 3, 8, 9])
    a = oracle.ce_loss(X, E, tgt, 10)
    E2 = E.copy()
    E2[10:] = 100.0          # huge padding rows must not change anything
    np.testing.assert_array_equal(a, oracle.ce_loss(X, E2, tgt, 10))
    np.testing.assert_allclose(a, _brute(X.tolist(), E.tolist(), tgt.tolist(), 10), rtol=1e-12)


def test_zero_embedding_closed_form():
    # E = 0: every logit is 0, so the loss is ln(v_valid) exactly.
    g = read_kv("vocab_padding.txt")
    v, v_pad = int(g["v"][0]), int(g["v_pad"][0])
    X = np.random.default_rng(0).standard_normal((3, 4))
    E = np.zeros((v_pad, 4))
    tgt = np.array([0, 17, v - 1])
    np.testing.assert_allclose(oracle.ce_loss(X, E, tgt, v), math.log(v), rtol=1e-15)
    np.testing.assert_allclose(oracle.ce_loss(X, E, tgt, v_pad), math.log(v_pad), rtol=1e-15)
    assert math.log(v) == pytest.approx(10.82491, abs=1e-5)
    assert math.log(v_pad) == pytest.approx(10.84349, abs=1e-5)


def test_shift_invariance():
    # Appending a constant feature to X (1) and E (c) adds c to every logit.
    rng = np.random.default_rng(4)
    X = rng.standard_normal((6, 5))
    E = rng.standard_normal((20, 5))
    tgt = rng.integers(0, 20, 6)
    a = oracle.ce_loss(X, E, tgt, 20)
    X2 = np.concatenate([X, np.ones((6, 1))], axis=1)
    E2 = np.concatenate([E, np.full((20, 1), 37.5)], axis=1)
    np.testing.assert_allclose(oracle.ce_loss(X2, E2, tgt, 20), a, rtol=1e-12, atol=1e-12)


def test_dominant_target_zero_loss():
    X = np.array([[1.0, 0.0]])
    E = np.zeros((9, 2))
    E[4, 0] = 50.0
    assert oracle.ce_loss(X, E, np.array([4]), 9)[0] < 1e-19


@pytest.mark.parametrize("P", [1, 2, 4, 8, 16])
@pytest.mark.parametrize("v_valid", [64, 61, 40])
def test_partition_invariance(P, v_valid):
    rng = np.random.default_rng(P * 100 + v_valid)
    X = rng.standard_normal((7, 6))
    E = rng.standard_normal((64, 6))
    tgt = rng.integers(0, v_valid, 7)
    full = oracle.ce_loss(X, E, tgt, v_valid)
    np.testing.assert_allclose(oracle.ce_loss_partitioned(X, E, tgt, v_valid, P), full, rtol=1e-13, atol=1e-13)


def test_partitioned_rejects_missing_rescale():
    # Planted mistake: adding s_p without rescaling by exp(m_p - M) breaks the pin.
    rng = np.random.default_rng(9)
    X = rng.standard_normal((7, 6))
    E = rng.standard_normal((64, 6))
    tgt = rng.integers(0, 64, 7)
    m, s, zt = oracle.ce_partition_triples(X, E, tgt, 64, 4)
    z = np.nansum(np.where(np.isnan(zt), 0.0, zt), axis=0)
    wrong = m.max(axis=0) + np.log(s.sum(axis=0)) - z
    assert not np.allclose(wrong, oracle.ce_loss(X, E, tgt, 64))


def test_rejects_bad_target():
    with pytest.raises(ValueError):
        oracle.ce_loss(np.ones((1, 2)), np.ones((4, 2)), np.array([4]), 4)


def test_padding_rule():
    g = read_kv("vocab_padding.txt")
    v, t, mult = int(g["v"][0]), int(g["t"][0]), int(g["multiple"][0])
    v_pad = oracle.pad_vocab(v, t, mult)
    assert v_pad == int(g["v_pad"][0])
    assert v_pad - v == int(g["pad_rows"][0])
    assert (v_pad // t) % mult == 0
    assert oracle.pad_vocab(51200, 8) == 51200
    assert oracle.pad_vocab(1, 1) == 128
    b, s = int(g["b"][0]), int(g["s"][0])
    assert b * s * v_pad == int(g["n_logits"][0])
    assert b * s == int(g["n_losses"][0])
