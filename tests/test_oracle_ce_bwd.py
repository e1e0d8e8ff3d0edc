"""Pins of the oracle's cross-entropy backward (CPU only)."""
import numpy as np
import pytest

import oracle


def _problem(seed, T=5, h=6, v=9, v_pad=12):
    rng = np.random.default_rng(seed)
    X = rng.standard_normal((T, h))
    E = rng.standard_normal((v_pad, h)) * 0.5
    tgt = rng.integers(0, v, T)
    dl = rng.standard_normal(T)
    return X, E, tgt, dl, v


def _objective(X, E, tgt, dl, v):
    return float(np.sum(dl * oracle.ce_loss(X, E, tgt, v)))


def _fd(fn, M, eps=1e-6):
    g = np.zeros_like(M)
    for i in np.ndindex(M.shape):
        old = M[i]
        M[i] = old + eps
        a = fn()
        M[i] = old - eps
        b = fn()
        M[i] = old
        g[i] = (a - b) / (2 * eps)
    return g


def _check(bwd):
    X, E, tgt, dl, v = _problem(1)
    out = bwd(X, E, tgt, dl, v)
    f = lambda: _objective(X, E, tgt, dl, v)
    return (np.max(np.abs(out["dX"] - _fd(f, X))) < 1e-7 and
            np.max(np.abs(out["dE"] - _fd(f, E))) < 1e-7)


def test_finite_differences():
    # padding rows (v <= c < v_pad) get exactly zero gradient
    assert _check(oracle.ce_bwd)
    X, E, tgt, dl, v = _problem(2)
    assert np.all(oracle.ce_bwd(X, E, tgt, dl, v)["dE"][v:] == 0.0)


def test_fd_rejects_missing_onehot():
    # planted mistake: softmax without subtracting the one-hot target
    def wrong(X, E, tgt, dl, v):
        d = oracle.ce_bwd(X, E, tgt, dl, v)
        oh = np.zeros_like(d["dZ"])
        oh[np.arange(len(tgt)), tgt] = dl
        dZ = d["dZ"] + oh
        dE = np.zeros_like(E)
        dE[:v] = dZ.T @ X
        return {"dX": dZ @ E[:v], "dE": dE}
    assert not _check(wrong)


def test_rows_of_dz_sum_to_zero():
    X, E, tgt, dl, v = _problem(3)
    dZ = oracle.ce_bwd(X, E, tgt, dl, v)["dZ"]
    np.testing.assert_allclose(dZ.sum(axis=1), 0.0, atol=1e-14)


def test_zero_embedding_closed_form():
    # E = 0: p = 1/v for every column, so dZ = dloss (1/v - onehot), dX = 0 and dE = dZ^T X.
    rng = np.random.default_rng(4)
    T, h, v = 4, 3, 7
    X = rng.standard_normal((T, h))
    E = np.zeros((8, h))
    tgt = np.array([0, 3, 6, 3])
    dl = np.array([1.0, -2.0, 0.5, 0.25])
    out = oracle.ce_bwd(X, E, tgt, dl, v)
    dZ = np.tile(dl[:, None] / v, (1, v))
    dZ[np.arange(T), tgt] -= dl
    np.testing.assert_allclose(out["dX"], 0.0, atol=1e-15)
    np.testing.assert_allclose(out["dE"][:v], dZ.T @ X, atol=1e-14)


def test_sampled_matches_full():
    X, E, tgt, dl, v = _problem(5, T=40, h=8, v=30, v_pad=32)
    full = oracle.ce_bwd(X, E, tgt, dl, v)
    rows = np.array([0, 7, 39])
    erows = np.array([0, 5, 29, 31])         # 31 is a padding row
    s = oracle.ce_bwd_sampled(X, E, tgt, dl, v, rows, erows)
    np.testing.assert_allclose(s["dX_rows"], full["dX"][rows], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(s["dE_rows"], full["dE"][erows], rtol=1e-12, atol=1e-13)
    lse = oracle.ce_logsumexp(X, E, v, block=7)
    z = X @ E[:v].T
    np.testing.assert_allclose(lse, np.log(np.exp(z).sum(axis=1)), rtol=1e-13)


def test_rejects_bad_target():
    with pytest.raises(ValueError):
        oracle.ce_bwd(np.ones((1, 2)), np.ones((4, 2)), np.array([4]), np.ones(1), 4)
