"""Pin the oracle's Philox4x64-10 to numpy's independent implementation."""

import numpy as np

from oracle import philox


def _numpy_block(counter, key):
    # numpy's Philox bumps its 256-bit counter before producing each block of four
    # words, so start it one below the counter we want.
    c = sum(int(w) << (64 * i) for i, w in enumerate(counter)) - 1
    c %= 1 << 256
    words = np.array([(c >> (64 * i)) & philox.MASK64 for i in range(4)], dtype=np.uint64)
    bg = np.random.Philox(counter=words, key=np.array(key, dtype=np.uint64))
    return tuple(int(x) for x in bg.random_raw(4))


def test_philox_matches_numpy():
    rng = np.random.default_rng(2024)
    for _ in range(200):
        key = tuple(int(x) for x in rng.integers(0, 2**64, size=2, dtype=np.uint64))
        counter = tuple(int(x) for x in rng.integers(0, 2**64, size=4, dtype=np.uint64))
        assert philox.philox4x64_10(counter, key) == _numpy_block(counter, key)


def test_philox_small_counters_match_numpy():
    # the layout used by the method: (b, j, stream, 0) with key (seed, 0)
    for seed in (0, 1, 12345, 2**64 - 1):
        for b in (0, 1, 31):
            for j in (1, 7, 16):
                for stream in range(4):
                    ctr = (b, j, stream, 0)
                    if ctr == (0, 0, 0, 0):
                        continue
                    assert philox.philox4x64_10(ctr, (seed, 0)) == _numpy_block(ctr, (seed, 0))


def test_uniform_is_exact_24bit():
    seen = set()
    for seed in range(4):
        for j in range(1, 9):
            u = philox.uniform(seed, 3, j, 1)
            assert 0.0 <= u < 1.0
            assert float(np.float32(u)) == u          # exact in float32
            assert (u * 2**24) == int(u * 2**24)       # on the 2^-24 grid
            seen.add(u)
    assert len(seen) == 32                             # streams do not collide here
