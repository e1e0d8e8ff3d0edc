"""Pins of the oracle's GeLU (CPU only)."""
import math

import numpy as np
import pytest

import oracle
from _golden import read_columns


def _golden_gelu_ok(gelu_fn):
    for x, want in read_columns("gelu_values.txt"):
        if round(float(gelu_fn(x)), 3) != want:
            return False
    return True


def test_gelu_printed_values():
    # "Megatron-LM, annotated" section 2.2 prints these three values.
    for x, want in read_columns("gelu_values.txt"):
        assert round(float(oracle.gelu(x)), 3) == want


def test_gelu_printed_values_reject_tanh_form():
    # Planted mistake: the tanh approximation misses GELU(2) = 1.954 at 3 decimals.
    c = math.sqrt(2.0 / math.pi)
    tanh_gelu = lambda x: 0.5 * x * (1.0 + math.tanh(c * (x + 0.044715 * x ** 3)))
    assert not _golden_gelu_ok(tanh_gelu)


def test_gelu_closed_forms():
    assert oracle.gelu(0.0) == 0.0
    assert float(oracle.gelu_prime(0.0)) == pytest.approx(0.5, abs=1e-15)
    xs = np.linspace(-6, 6, 1201)
    # Phi(x) + Phi(-x) = 1  =>  GELU(x) - GELU(-x) = x
    np.testing.assert_allclose(oracle.gelu(xs) - oracle.gelu(-xs), xs, atol=1e-14)
    # far tails: GELU(x) -> x for large x, -> 0 for very negative x
    assert abs(float(oracle.gelu(12.0)) - 12.0) < 1e-20 + 1e-12
    assert abs(float(oracle.gelu(-12.0))) < 1e-30


def test_gelu_against_erfc_routine():
    # Phi(x) = erfc(-x / sqrt 2) / 2: a different library routine for the same function.
    for x in np.linspace(-5, 5, 101):
        want = x * 0.5 * math.erfc(-x / math.sqrt(2.0))
        assert float(oracle.gelu(x)) == pytest.approx(want, rel=1e-13, abs=1e-15)


def test_gelu_prime_finite_differences():
    xs = np.linspace(-6, 6, 241)
    eps = 1e-5
    fd = (oracle.gelu(xs + eps) - oracle.gelu(xs - eps)) / (2 * eps)
    np.testing.assert_allclose(oracle.gelu_prime(xs), fd, atol=1e-9)


def test_gelu_prime_rejects_sign_mistake():
    # Planted mistake: Phi(x) - x*phi(x) fails the finite-difference pin.
    xs = np.linspace(-3, 3, 61)
    eps = 1e-5
    fd = (oracle.gelu(xs + eps) - oracle.gelu(xs - eps)) / (2 * eps)
    wrong = oracle.std_normal_cdf(xs) - xs * oracle.std_normal_pdf(xs)
    assert np.max(np.abs(wrong - fd)) > 1e-2
