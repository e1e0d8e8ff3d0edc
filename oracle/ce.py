"""Vocab-parallel cross-entropy, float64. Test infrastructure.

[p1] §3.4 "Output Embedding Parallelism and the Fused Cross-Entropy
Optimization": logits of token r are z_r = X[r] E^T with E [v, h] (the tied
embedding, split along the vocabulary into row blocks E_i); the loss is the
softmax cross-entropy of z_r at the target id. The page's steps: per shard the
row max m_i, an all-reduce for the global max M, per shard the shifted sum
s_i = sum exp(z - M) and the target logit where the shard owns it, an
all-reduce of the sums, and the loss.

Reading adopted where the page is garbled (its last step drops the max shift):
loss = M + log(S) - z_target with S = sum_c exp(z_c - M), the standard
log-softmax cross-entropy. Columns c >= v_valid (vocabulary padding, [p5] §3.4)
are excluded from the softmax.

``ce_loss`` is the plain full-logit definition and is the oracle the GPU is
compared with. ``ce_partition_triples`` / ``ce_combine`` take the page's steps
per partition; they exist to check partition invariance. ``ce_combine`` uses
the single-pass form S = sum_p s_p exp(m_p - M) where s_p is taken about the
partition's own max m_p, which is the same number as the page's two-step form.
"""
import numpy as np


def _f64(a):
    return np.asarray(a, dtype=np.float64)


def ce_loss(X, E, target, v_valid: int):
    """Per-token loss [T] = logsumexp(z[:v_valid]) - z[target], z = X E^T."""
    X, E = _f64(X), _f64(E)
    target = np.asarray(target, dtype=np.int64)
    if np.any(target < 0) or np.any(target >= v_valid):
        raise ValueError("target id outside [0, v_valid)")
    z = X @ E[:v_valid].T                      # [T, v_valid]
    M = z.max(axis=1)
    S = np.exp(z - M[:, None]).sum(axis=1)
    z_t = z[np.arange(z.shape[0]), target]
    return M + np.log(S) - z_t


def ce_partition_triples(X, E, target, v_valid: int, P: int):
    """Per partition p of P equal column ranges of E's rows: (m_p, s_p, z_p).

    m_p = max of the partition's valid logits (-inf if it has none);
    s_p = sum exp(z - m_p) over them (0 if none); z_p = target logit where the
    target lies in the partition, else nan. Returns arrays [P, T].
    """
    X, E = _f64(X), _f64(E)
    target = np.asarray(target, dtype=np.int64)
    v_pad = E.shape[0]
    if P < 1 or v_pad % P != 0:
        raise ValueError("P must divide the padded vocabulary")
    w = v_pad // P
    T = X.shape[0]
    m = np.full((P, T), -np.inf)
    s = np.zeros((P, T))
    zt = np.full((P, T), np.nan)
    for p in range(P):
        lo, hi = p * w, min((p + 1) * w, v_valid)
        if hi <= lo:
            continue
        z = X @ E[lo:hi].T
        m[p] = z.max(axis=1)
        s[p] = np.exp(z - m[p][:, None]).sum(axis=1)
        own = (target >= lo) & (target < hi)
        zt[p, own] = z[np.nonzero(own)[0], target[own] - lo]
    return m, s, zt


def ce_combine(m, s, zt):
    """Combine partition triples: M = max_p m_p, S = sum_p s_p exp(m_p - M),
    z = the owning partition's target logit; loss = M + log S - z."""
    m, s, zt = _f64(m), _f64(s), _f64(zt)
    M = m.max(axis=0)
    S = np.zeros_like(M)
    for p in range(m.shape[0]):
        live = s[p] > 0
        S[live] += s[p][live] * np.exp(m[p][live] - M[live])
    z = np.nansum(np.where(np.isnan(zt), 0.0, zt), axis=0)
    return M + np.log(S) - z


def ce_loss_partitioned(X, E, target, v_valid: int, P: int):
    return ce_combine(*ce_partition_triples(X, E, target, v_valid, P))


def ce_bwd(X, E, target, dloss, v_valid: int):
    """Gradient of sum_r dloss[r] * loss[r] (loss as in ``ce_loss``) w.r.t. X and E.

    The plain derivative of softmax cross-entropy: with p = softmax(z) over the
    valid columns, dZ[r, c] = dloss[r] * (p[r, c] - [c == target[r]]);
    dX = dZ E[:v_valid]; dE[:v_valid] = dZ^T X and dE[v_valid:] = 0 (padding rows
    take no part in the loss). Returns dict with dX, dE, dZ.
    """
    X, E = _f64(X), _f64(E)
    target = np.asarray(target, dtype=np.int64)
    dloss = _f64(dloss)
    if np.any(target < 0) or np.any(target >= v_valid):
        raise ValueError("target id outside [0, v_valid)")
    z = X @ E[:v_valid].T
    M = z.max(axis=1, keepdims=True)
    p = np.exp(z - M)
    p /= p.sum(axis=1, keepdims=True)
    p[np.arange(z.shape[0]), target] -= 1.0
    dZ = dloss[:, None] * p
    dE = np.zeros_like(E)
    dE[:v_valid] = dZ.T @ X
    return {"dX": dZ @ E[:v_valid], "dE": dE, "dZ": dZ}


def ce_logsumexp(X, E, v_valid: int, block: int = 512):
    """Per-token log sum_c exp(z[r, c]) over the valid columns, computed a block of
    tokens at a time (same arithmetic as ``ce_loss``, bounded memory)."""
    X, E = _f64(X), _f64(E)
    out = np.empty(X.shape[0])
    Ev = E[:v_valid]
    for lo in range(0, X.shape[0], block):
        z = X[lo:lo + block] @ Ev.T
        M = z.max(axis=1)
        out[lo:lo + block] = M + np.log(np.exp(z - M[:, None]).sum(axis=1))
    return out


def ce_bwd_sampled(X, E, target, dloss, v_valid: int, rows, e_rows, lse=None):
    """dX[rows] and dE[e_rows] of ``ce_bwd`` without forming the full [T, v] matrix.

    A row of dX needs its token's logits over the vocabulary; a row c of dE needs
    column c of dZ over all tokens, i.e. z[:, c] and every token's log-sum-exp
    (``lse``, computed here by ``ce_logsumexp`` when not given).
    """
    X, E = _f64(X), _f64(E)
    target = np.asarray(target, dtype=np.int64)
    dloss = _f64(dloss)
    rows = np.asarray(rows)
    e_rows = np.asarray(e_rows)
    r = ce_bwd(X[rows], E, target[rows], dloss[rows], v_valid)
    if lse is None:
        lse = ce_logsumexp(X, E, v_valid)
    dE = np.zeros((len(e_rows), E.shape[1]))
    valid = e_rows < v_valid
    if np.any(valid):
        c = e_rows[valid]
        zc = X @ E[c].T                                   # [T, n]
        dZc = np.exp(zc - lse[:, None])
        dZc -= (target[:, None] == c[None, :])
        dZc *= dloss[:, None]
        dE[valid] = dZc.T @ X
    return {"dX_rows": r["dX"], "dE_rows": dE}
