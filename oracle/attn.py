"""Self-attention block with head parallelism, forward, float64. Test infrastructure.

[p1] §3.4 "Attention Head Parallelism in the Self-Attention Block" and [p5] §3.2
"The attention block": the key, query and value projections are split by columns
so that shard i holds whole heads; each shard runs softmax attention for its
heads alone; the output projection is split by rows and the shards' partial
outputs are summed (the g operator). GPT-2 is a decoder that reads left to right
([p5] §2.2), so the attention is causal; [p5] §3.2 gives the 8.3B model's
32 heads of width 96 on 8 shards (4 heads each).

Layout read here (the pages fix only the split, not the packing): Wqkv [h, 3h]
holds the Q, K and V projections side by side ([Wq | Wk | Wv]); head j owns
columns [j d, (j+1) d) of each, d = h / heads; Wo [h, h]; X [b s, h] holds b
sequences of s tokens. No dropout (the measured path has none).
"""
import numpy as np


def _f64(a):
    return np.asarray(a, dtype=np.float64)


def _softmax_rows(S):
    M = S.max(axis=1, keepdims=True)
    P = np.exp(S - M)
    return P / P.sum(axis=1, keepdims=True)


def attention_heads(Q, K, V, heads: int, b: int, s: int):
    """O [b s, h]: for each sequence and head, softmax(Q_j K_j^T / sqrt(d) + causal mask) V_j."""
    Q, K, V = _f64(Q), _f64(K), _f64(V)
    h = Q.shape[1]
    d = h // heads
    O = np.zeros_like(Q)
    causal = np.triu(np.ones((s, s), dtype=bool), k=1)   # key index > query index
    for q in range(b):
        rows = slice(q * s, (q + 1) * s)
        for j in range(heads):
            cols = slice(j * d, (j + 1) * d)
            S = Q[rows, cols] @ K[rows, cols].T / np.sqrt(d)
            S[causal] = -np.inf
            O[rows, cols] = _softmax_rows(S) @ V[rows, cols]
    return O


def attn_fwd(X, Wqkv, Wo, heads: int, b: int, s: int):
    """Unsplit block: QKV = X Wqkv; O = attention; out = O Wo. Returns (QKV, O, out)."""
    X, Wqkv, Wo = _f64(X), _f64(Wqkv), _f64(Wo)
    h = X.shape[1]
    QKV = X @ Wqkv
    O = attention_heads(QKV[:, :h], QKV[:, h:2 * h], QKV[:, 2 * h:], heads, b, s)
    return QKV, O, O @ Wo


def attn_fwd_sharded(X, Wqkv, Wo, heads: int, b: int, s: int, t: int):
    """Shard by shard: shard i takes its heads' columns of Wq, Wk, Wv, runs their
    attention and multiplies by its rows of Wo; out = sum over shards (g).
    Returns (out, [partial_i])."""
    X, Wqkv, Wo = _f64(X), _f64(Wqkv), _f64(Wo)
    h = X.shape[1]
    if t < 1 or heads % t != 0:
        raise ValueError("t must divide the number of heads")
    d = h // heads
    w = (heads // t) * d
    parts = []
    for i in range(t):
        cols = np.arange(i * w, (i + 1) * w)
        Wq_i, Wk_i, Wv_i = Wqkv[:, cols], Wqkv[:, h + cols], Wqkv[:, 2 * h + cols]
        O_i = attention_heads(X @ Wq_i, X @ Wk_i, X @ Wv_i, heads // t, b, s)
        parts.append(O_i @ Wo[cols, :])
    out = parts[0].copy()
    for p in parts[1:]:
        out += p
    return out, parts


def attn_fwd_rows(X, Wqkv, Wo, heads: int, b: int, s: int, rows):
    """out[rows] and O[rows]: a query row needs its own sequence's keys and values up
    to itself, so each sampled sequence's projections are formed once (up to its last
    sampled row) and the rows' attention is taken from them."""
    X, Wqkv, Wo = _f64(X), _f64(Wqkv), _f64(Wo)
    h = X.shape[1]
    d = h // heads
    rows = np.asarray(rows)
    O = np.zeros((len(rows), h))
    for q in np.unique(rows // s):
        sel = np.nonzero(rows // s == q)[0]
        last = int(rows[sel].max())
        q0 = q * s
        QKV = X[q0:last + 1] @ Wqkv
        for n in sel:
            i = int(rows[n]) - q0
            for j in range(heads):
                c = slice(j * d, (j + 1) * d)
                sc = QKV[:i + 1, h + j * d:h + (j + 1) * d] @ QKV[i, c] / np.sqrt(d)
                p = np.exp(sc - sc.max())
                O[n, c] = (p / p.sum()) @ QKV[:i + 1, 2 * h + j * d:2 * h + (j + 1) * d]
    return O, O @ Wo
