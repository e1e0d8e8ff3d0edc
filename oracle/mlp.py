"""The MLP block Z = GeLU(X A) B, forward and backward, float64. Test infrastructure.

Notation of [p3] "Tensor and pipeline parallelism, and choosing a layout", §3,
Proposition (Megatron MLP split): X is [T, h], A is [h, f] (f = 4h), B is
[f, h]; A is split by columns and B by rows into t blocks of f/t; U = X A,
Y = GeLU(U), Z = Y B; G = dL/dZ.

``mlp_fwd`` / ``mlp_bwd`` are the unsplit definitions. The method reaches the
same numbers by sharding (the proposition's proof), so the unsplit layer is
the oracle the CUDA path is compared with. ``mlp_sharded_*`` walk the t shards
one by one exactly as proof steps 1-5 write them and exist to check that
invariance, not to be compared with the GPU. ``first_layer_row_cut`` is the
rejected split of [p1] §3.4 "Option 1" and [p5] §3.1 "Cut by rows".
"""
import numpy as np

from .gelu import gelu, gelu_prime


def _f64(a):
    return np.asarray(a, dtype=np.float64)


def mlp_fwd(X, A, B):
    """Unsplit forward: U = X A, Y = GeLU(U), Z = Y B. Returns (U, Y, Z)."""
    X, A, B = _f64(X), _f64(A), _f64(B)
    U = X @ A
    Y = gelu(U)
    Z = Y @ B
    return U, Y, Z


def mlp_bwd(X, A, B, G):
    """Unsplit backward of Z = GeLU(X A) B given G = dL/dZ.

    dY = G B^T; dU = dY * GeLU'(U); dB = Y^T G; dA = X^T dU; dX = dU A^T.
    Returns dict with dX, dA, dB, dU, U, Y.
    """
    X, A, B, G = _f64(X), _f64(A), _f64(B), _f64(G)
    U = X @ A
    Y = gelu(U)
    dY = G @ B.T
    dU = dY * gelu_prime(U)
    return {
        "dX": dU @ A.T,
        "dA": X.T @ dU,
        "dB": Y.T @ G,
        "dU": dU,
        "U": U,
        "Y": Y,
    }


def _shard_bounds(f: int, t: int):
    if t < 1 or f % t != 0:
        raise ValueError(f"shard count t={t} must divide f={f}")
    w = f // t
    return [(i * w, (i + 1) * w) for i in range(t)]


def mlp_sharded_fwd(X, A, B, t: int):
    """Forward shard by shard (proof steps 1-3): for i in 0..t-1,
    U_i = X A_i, Y_i = GeLU(U_i), Z_i = Y_i B_i; Z = sum_i Z_i (the g operator).

    Returns (Z, [Z_i]).
    """
    X, A, B = _f64(X), _f64(A), _f64(B)
    parts = []
    for lo, hi in _shard_bounds(A.shape[1], t):
        A_i = A[:, lo:hi]          # column block of A
        B_i = B[lo:hi, :]          # row block of B
        U_i = X @ A_i
        Y_i = gelu(U_i)
        parts.append(Y_i @ B_i)
    Z = parts[0].copy()
    for p in parts[1:]:
        Z += p
    return Z, parts


def mlp_sharded_bwd(X, A, B, G, t: int):
    """Backward shard by shard (proof steps 4-5).

    For shard i: dB_i = Y_i^T G, dY_i = G B_i^T, dU_i = dY_i * GeLU'(U_i),
    dA_i = X^T dU_i, and the shard's part of dX is dU_i A_i^T; dX is the sum of
    the parts (the f operator). dA and dB are the shards' blocks side by side.
    Returns dict with dX, dA, dB and dX_parts.
    """
    X, A, B, G = _f64(X), _f64(A), _f64(B), _f64(G)
    f = A.shape[1]
    dA = np.empty_like(A)
    dB = np.empty_like(B)
    dX_parts = []
    for lo, hi in _shard_bounds(f, t):
        A_i = A[:, lo:hi]
        B_i = B[lo:hi, :]
        U_i = X @ A_i
        Y_i = gelu(U_i)
        dB[lo:hi, :] = Y_i.T @ G
        dY_i = G @ B_i.T
        dU_i = dY_i * gelu_prime(U_i)
        dA[:, lo:hi] = X.T @ dU_i
        dX_parts.append(dU_i @ A_i.T)
    dX = dX_parts[0].copy()
    for p in dX_parts[1:]:
        dX += p
    return {"dX": dX, "dA": dA, "dB": dB, "dX_parts": dX_parts}


def first_layer_row_cut(X, A, t: int):
    """The rejected split of the first GEMM ([p1] §3.4 Option 1, [p5] §3.1).

    X is cut by columns and A by rows into t blocks; block i gives the partial
    product P_i = X_i A_i. Returns (gelu_of_sum, sum_of_gelus): the first is
    GeLU(sum_i P_i) (correct, needs a sum before the GeLU), the second is
    sum_i GeLU(P_i) (what applying GeLU locally would give, which is wrong).
    """
    X, A = _f64(X), _f64(A)
    h = A.shape[0]
    parts = []
    for lo, hi in _shard_bounds(h, t):
        parts.append(X[:, lo:hi] @ A[lo:hi, :])
    total = parts[0].copy()
    for p in parts[1:]:
        total += p
    gelu_first = gelu(parts[0])
    for p in parts[1:]:
        gelu_first = gelu_first + gelu(p)
    return gelu(total), gelu_first


# ---------------------------------------------------------------------------
# Sampled-index forms for large workloads. The block is separable: a row of Z
# or dX needs only its own row of X (and G); column j of dA needs column j of
# dU over all tokens; row j of dB needs column j of Y over all tokens. These
# are the same definitions restricted to the requested indices.
# ---------------------------------------------------------------------------

def mlp_fwd_rows(X, A, B, rows):
    """(U[rows], Y[rows], Z[rows]) of the unsplit forward."""
    Xr = _f64(X)[np.asarray(rows)]
    return mlp_fwd(Xr, A, B)


def mlp_bwd_sampled(X, A, B, G, rows, a_cols, b_rows):
    """dX[rows], dA[:, a_cols], dB[b_rows, :] and dU[rows] of the unsplit backward."""
    X, A, B, G = _f64(X), _f64(A), _f64(B), _f64(G)
    rows = np.asarray(rows)
    a_cols = np.asarray(a_cols)
    b_rows = np.asarray(b_rows)
    # rows of dX: dU[r] = (G[r] B^T) * GeLU'(X[r] A); dX[r] = dU[r] A^T
    U_r = X[rows] @ A
    dU_r = (G[rows] @ B.T) * gelu_prime(U_r)
    dX_r = dU_r @ A.T
    # columns of dA: dU[:, j] = (G B[j, :]^T) * GeLU'(X A[:, j]); dA[:, j] = X^T dU[:, j]
    U_c = X @ A[:, a_cols]
    dU_c = (G @ B[a_cols, :].T) * gelu_prime(U_c)
    dA_c = X.T @ dU_c
    # rows of dB: Y[:, j] = GeLU(X A[:, j]); dB[j, :] = Y[:, j]^T G
    Y_c = gelu(X @ A[:, b_rows])
    dB_r = Y_c.T @ G
    return {"dX_rows": dX_r, "dA_cols": dA_c, "dB_rows": dB_r, "dU_rows": dU_r}
