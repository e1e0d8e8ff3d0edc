"""Pins of the oracle's vocab-parallel embedding (CPU only)."""
import numpy as np
import pytest

import oracle


@pytest.mark.parametrize("t", [1, 2, 4, 8])
def test_sharded_lookup_is_the_plain_lookup(t):
    # Exactly one shard owns each valid id, so the sum over shards is the row itself.
    rng = np.random.default_rng(t)
    E = rng.standard_normal((64, 5))
    ids = rng.integers(0, 60, 33)
    np.testing.assert_array_equal(oracle.embed_sharded(ids, E, 60, t), E[ids])


def test_invalid_ids_give_zero_rows():
    E = np.arange(32.0).reshape(8, 4)
    ids = np.array([0, 6, 7, -1, 3])          # 6, 7 are padding ids (v_valid = 6), -1 is invalid
    out = oracle.embed_sharded(ids, E, 6, 2)
    np.testing.assert_array_equal(out[[0, 4]], E[[0, 3]])
    assert np.all(out[1:4] == 0.0)


def test_rejects_planted_double_count():
    # Planted mistake: a shard that also claims the next shard's first id double-counts it.
    E = np.ones((8, 2))
    ids = np.array([4])
    good = oracle.embed_sharded(ids, E, 8, 2)
    vs = 4
    wrong = np.zeros((1, 2))
    for i in range(2):
        own = (ids >= i * vs) & (ids <= (i + 1) * vs)   # <= instead of <
        wrong[own] += E[ids[own]]
    assert not np.array_equal(wrong, good)
