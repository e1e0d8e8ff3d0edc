"""GeLU in its exact (erf) form and its derivative, float64. Test infrastructure.

[p5] "Megatron-LM, annotated", §2.2: GELU(x) is x times the probability that a
standard normal variable falls below x, i.e. x * Phi(x) with
Phi(x) = (1 + erf(x / sqrt 2)) / 2; the page prints GELU(1) = 0.841,
GELU(-1) = -0.159, GELU(2) = 1.954 (three decimals), which the erf form gives
and the tanh approximation (GELU(2) -> 1.955) does not.

The derivative is the plain product rule on x * Phi(x): Phi(x) + x * phi(x),
phi the standard normal density. [p3] Proposition (Megatron MLP split), step 4,
uses GeLU'(U_i) in dL/dU_i; the page's own listing uses the tanh form, which
this oracle does not adopt (the erf form is the one the printed values pin).
"""
import math

import numpy as np
from scipy.special import erf

_INV_SQRT2 = 1.0 / math.sqrt(2.0)
_INV_SQRT_2PI = 1.0 / math.sqrt(2.0 * math.pi)


def std_normal_cdf(x):
    """Phi(x) = (1 + erf(x / sqrt(2))) / 2."""
    return 0.5 * (1.0 + erf(np.asarray(x, dtype=np.float64) * _INV_SQRT2))


def std_normal_pdf(x):
    """phi(x) = exp(-x^2 / 2) / sqrt(2 pi)."""
    x = np.asarray(x, dtype=np.float64)
    return np.exp(-0.5 * x * x) * _INV_SQRT_2PI


def gelu(x):
    """GELU(x) = x * Phi(x)."""
    x = np.asarray(x, dtype=np.float64)
    return x * std_normal_cdf(x)


def gelu_prime(x):
    """d/dx GELU(x) = Phi(x) + x * phi(x)."""
    x = np.asarray(x, dtype=np.float64)
    return std_normal_cdf(x) + x * std_normal_pdf(x)
