"""The stabilised forward decides whether a tile's maximum occurs twice from
two partitions of the tile's 128 keys: the eight chains of keys with equal
c mod 8 (whose maxima the row max already computes) and the 16 blocks of 8
consecutive keys.  Two distinct keys differ in c mod 8 or, if not, in c div 8,
so the maximum repeats exactly when two chain maxima or two block maxima
equal it.  This checks that argument on every pair of key positions and on
random tiles, against a direct count (host-side model; the kernels' use of it
is checked by the statistics variant, whose shift follows the same decision
and whose unit-probability counts are compared with the oracle)."""
import itertools

import numpy as np


def _repeats_by_partitions(s):
    tm = s.max()
    chains = s.reshape(16, 8).max(axis=0)   # c mod 8: column e of the 16 x 8 view
    blocks = s.reshape(16, 8).max(axis=1)   # c div 8: row b
    return int((chains == tm).sum()) >= 2 or int((blocks == tm).sum()) >= 2


def test_every_pair_of_positions():
    rng = np.random.default_rng(1)
    base = rng.standard_normal(128).astype(np.float32)
    for i, j in itertools.combinations(range(128), 2):
        s = base.copy()
        s[i] = s[j] = np.float32(10.0)          # the maximum, exactly twice
        assert _repeats_by_partitions(s), (i, j)
        s[j] = np.float32(9.5)                  # now once
        assert not _repeats_by_partitions(s), (i, j)


def test_random_tiles_with_few_distinct_values():
    rng = np.random.default_rng(2)
    for _ in range(20000):
        s = rng.integers(-3, 4, 128).astype(np.float32)   # many exact repeats
        if rng.random() < 0.5:
            s[rng.integers(0, 128)] = np.float32(5.0)      # a unique maximum
        assert _repeats_by_partitions(s) == (int((s == s.max()).sum()) >= 2)
