"""Pins of the oracle's MLP forward/backward (CPU only)."""
import math

import numpy as np
import pytest

import oracle
from _golden import read_kv


def _worked():
    g = read_kv("mlp_worked_example.txt")
    X = np.array([g["X"]])
    A = np.array([g["A_row0"], g["A_row1"]])
    B = np.array([g["B_row0"], g["B_row1"]])
    return g, X, A, B


def test_worked_example_forward():
    g, X, A, B = _worked()
    U, Y, Z = oracle.mlp_fwd(X, A, B)
    assert U[0].tolist() == g["XA"]
    assert [round(v, 3) for v in Y[0]] == g["gelu_XA_3dp"]
    assert [round(v, 3) for v in Z[0]] == g["Z_3dp"]


def test_worked_example_shards():
    g, X, A, B = _worked()
    Z, parts = oracle.mlp_sharded_fwd(X, A, B, t=2)
    assert [round(v, 3) + 0.0 for v in parts[0][0]] == g["col_shard_part1_3dp"]
    assert [round(v, 3) for v in parts[1][0]] == g["col_shard_part2_3dp"]
    assert [round(v, 3) for v in Z[0]] == g["Z_3dp"]


def test_worked_example_wrong_row_cut():
    g, X, A, B = _worked()
    right, wrong = oracle.first_layer_row_cut(X, A, t=2)
    assert [round(v, 3) for v in right[0]] == g["gelu_XA_3dp"]
    assert [round(v, 3) for v in wrong[0]] == g["row_cut_gelu_then_add_3dp"]
    assert np.max(np.abs(right - wrong)) > 0.5


def _gelu_py(x):
    return x * 0.5 * (1.0 + math.erf(x / math.sqrt(2.0)))


def _brute_force_fwd(X, A, B):
    T, h = len(X), len(X[0])
    f = len(A[0])
    Z = [[0.0] * h for _ in range(T)]
    for r in range(T):
        y = []
        for j in range(f):
            u = 0.0
            for k in range(h):
                u += X[r][k] * A[k][j]
            y.append(_gelu_py(u))
        for c in range(h):
            acc = 0.0
            for j in range(f):
                acc += y[j] * B[j][c]
            Z[r][c] = acc
    return np.array(Z)


def test_forward_brute_force():
    rng = np.random.default_rng(7)
    T, h, f = 3, 5, 12
    X = rng.standard_normal((T, h))
    A = rng.standard_normal((h, f)) * 0.5
    B = rng.standard_normal((f, h)) * 0.5
    _, _, Z = oracle.mlp_fwd(X, A, B)
    np.testing.assert_allclose(Z, _brute_force_fwd(X.tolist(), A.tolist(), B.tolist()), rtol=1e-12, atol=1e-13)


def _loss(X, A, B, G):
    return float(np.sum(oracle.mlp_fwd(X, A, B)[2] * G))


def _fd_grad(fn, M, eps=1e-6):
    g = np.zeros_like(M)
    it = np.nditer(M, flags=["multi_index"])
    for _ in it:
        i = it.multi_index
        old = M[i]
        M[i] = old + eps
        lp = fn()
        M[i] = old - eps
        lm = fn()
        M[i] = old
        g[i] = (lp - lm) / (2 * eps)
    return g


def _tiny_problem(seed=3, T=4, h=8, f=32):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal((T, h)), rng.standard_normal((h, f)) * 0.3,
            rng.standard_normal((f, h)) * 0.3, rng.standard_normal((T, h)))


def _check_bwd_fd(bwd_fn):
    X, A, B, G = _tiny_problem()
    out = bwd_fn(X, A, B, G)
    f = lambda: _loss(X, A, B, G)
    ok = True
    for name, M in (("dX", X), ("dA", A), ("dB", B)):
        fd = _fd_grad(f, M)
        ok &= np.max(np.abs(out[name] - fd)) < 1e-7
    return ok


def test_backward_finite_differences():
    # dL/dX, dL/dA, dL/dB of L = <G, Z(X, A, B)> by central differences in float64.
    assert _check_bwd_fd(oracle.mlp_bwd)


def test_backward_fd_rejects_dropped_gelu_prime():
    # Planted mistake: dA = X^T (G B^T) (GeLU' dropped) must fail the pin.
    def wrong_bwd(X, A, B, G):
        d = oracle.mlp_bwd(X, A, B, G)
        d = dict(d)
        d["dA"] = X.T @ (G @ B.T)
        return d
    assert not _check_bwd_fd(wrong_bwd)


def test_backward_fd_rejects_transposed_operand():
    # Planted mistake: dB = G^T Y (operands swapped, transposed result) fails.
    def wrong_bwd(X, A, B, G):
        d = dict(oracle.mlp_bwd(X, A, B, G))
        Y = oracle.gelu(X @ A)
        d["dB"] = (G.T @ Y).T[::-1].copy()
        return d
    assert not _check_bwd_fd(wrong_bwd)


@pytest.mark.parametrize("t", [1, 2, 4, 8, 16, 32])
def test_sharding_invariance(t):
    # Sharded result equals the unsplit one (to ~1e-15 on random matrices, per the
    # lesson-9 figure text); dX needs the sum over shards, one shard's part does not do.
    rng = np.random.default_rng(11)
    T, h, f = 6, 8, 32
    X, A, B, G = (rng.standard_normal((T, h)), rng.standard_normal((h, f)),
                  rng.standard_normal((f, h)), rng.standard_normal((T, h)))
    _, _, Z = oracle.mlp_fwd(X, A, B)
    Zs, parts = oracle.mlp_sharded_fwd(X, A, B, t)
    assert np.linalg.norm(Zs - Z) <= 1e-12 * np.linalg.norm(Z)
    ref = oracle.mlp_bwd(X, A, B, G)
    sh = oracle.mlp_sharded_bwd(X, A, B, G, t)
    for k in ("dX", "dA", "dB"):
        assert np.linalg.norm(sh[k] - ref[k]) <= 1e-12 * np.linalg.norm(ref[k])
    if t > 1:
        assert not np.allclose(sh["dX_parts"][0], ref["dX"])
        assert not np.allclose(parts[0], Z)


def test_sharding_rejects_bad_t():
    X, A, B, G = _tiny_problem()
    with pytest.raises(ValueError):
        oracle.mlp_sharded_fwd(X, A, B, 3)


def test_sampled_forms_match_full():
    rng = np.random.default_rng(5)
    T, h, f = 40, 16, 64
    X, A, B, G = (rng.standard_normal((T, h)), rng.standard_normal((h, f)) * 0.2,
                  rng.standard_normal((f, h)) * 0.2, rng.standard_normal((T, h)))
    rows = np.array([0, 3, 17, 39])
    cols = np.array([1, 30, 63])
    brows = np.array([0, 5, 62])
    U, Y, Z = oracle.mlp_fwd(X, A, B)
    Ur, Yr, Zr = oracle.mlp_fwd_rows(X, A, B, rows)
    np.testing.assert_allclose(Zr, Z[rows], rtol=1e-13, atol=1e-13)
    ref = oracle.mlp_bwd(X, A, B, G)
    s = oracle.mlp_bwd_sampled(X, A, B, G, rows, cols, brows)
    np.testing.assert_allclose(s["dX_rows"], ref["dX"][rows], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(s["dA_cols"], ref["dA"][:, cols], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(s["dB_rows"], ref["dB"][brows], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(s["dU_rows"], ref["dU"][rows], rtol=1e-12, atol=1e-12)
