"""Vocab-parallel input embedding. Test infrastructure.

[p1] §3.4 "Input Embedding Parallelism": E [v, h] is split along the
vocabulary into t row blocks E_i; for a token id, shard i looks the row up if the
id lies in its range and yields a zero vector otherwise; an all-reduce (the g
operator) sums the shards' results, which reconstructs the embedded token.

``embed_sharded`` takes those steps literally. An id outside [0, v_valid) is
owned by no shard here (padding ids are never looked up) and gives a zero row.
"""
import numpy as np


def embed_sharded(ids, E, v_valid: int, t: int):
    """out[r] = sum over shards i of (E_i[ids[r] - i*v_pad/t] if shard i owns ids[r] else 0)."""
    E = np.asarray(E, dtype=np.float64)
    ids = np.asarray(ids, dtype=np.int64)
    v_pad = E.shape[0]
    if t < 1 or v_pad % t != 0:
        raise ValueError("t must divide the padded vocabulary")
    vs = v_pad // t
    out = np.zeros((ids.shape[0], E.shape[1]))
    for i in range(t):
        lo = i * vs
        E_i = E[lo:lo + vs]
        own = (ids >= lo) & (ids < lo + vs) & (ids < v_valid) & (ids >= 0)
        part = np.zeros_like(out)
        part[own] = E_i[ids[own] - lo]
        out += part          # the g all-reduce across shards
    return out
