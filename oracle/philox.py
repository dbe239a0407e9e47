"""Philox4x64-10 and the uniform draw used by the sampling steps (oracle side).

Test infrastructure only (see ``oracle/__init__.py``).

The pages fix no random number generator; the T=1 draft and verify steps only need
"a sample" and "accept with min(1, p/q)".  This oracle uses the counter-based
Philox4x64 generator with 10 rounds, written here from its published definition
(Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy as 1, 2, 3", SC'11,
section 3.2 and table 2), so that a replay of any (seed, request, position, stream)
gives the same draw on the CPU and on the GPU, each side with its own code.

Counter/key layout (a reading of the pages, which leave it open):

* key     = (seed_b, 0)
* counter = (b, j, stream, 0)   b = request index, j = 1-based position
* stream  = 0 draft sample, 1 accept test, 2 residual draw, 3 bonus draw
* u       = (word0 >> 40) * 2**-24, a 24-bit uniform in [0, 1) that is exact in
  both float32 and float64, so both sides compare against the same number.

Pin: ``tests/test_oracle_philox.py`` checks ``philox4x64_10`` against numpy's own,
independent Philox4x64-10 implementation on random keys and counters.
"""

MASK64 = (1 << 64) - 1

# Multipliers and Weyl key increments of Philox4x64 (Salmon et al. 2011, table 2).
PHILOX_M0 = 0xD2E7470EE14C6C93
PHILOX_M1 = 0xCA5A826395121157
PHILOX_W0 = 0x9E3779B97F4A7C15
PHILOX_W1 = 0xBB67AE8584CAA73B
ROUNDS = 10

STREAM_DRAFT = 0
STREAM_ACCEPT = 1
STREAM_RESIDUAL = 2
STREAM_BONUS = 3


def _mulhilo(a, b):
    prod = a * b
    return prod >> 64, prod & MASK64


def philox4x64_10(counter, key):
    """Return the four 64-bit output words for a 4-word counter and 2-word key.

    One round maps (c0, c1, c2, c3) with key (k0, k1) to
    (hi(M1*c2) ^ c1 ^ k0, lo(M1*c2), hi(M0*c0) ^ c3 ^ k1, lo(M0*c0));
    the key is bumped by the Weyl constants before every round but the first.
    """
    c0, c1, c2, c3 = (int(x) & MASK64 for x in counter)
    k0, k1 = (int(x) & MASK64 for x in key)
    for rnd in range(ROUNDS):
        if rnd:
            k0 = (k0 + PHILOX_W0) & MASK64
            k1 = (k1 + PHILOX_W1) & MASK64
        hi0, lo0 = _mulhilo(PHILOX_M0, c0)
        hi1, lo1 = _mulhilo(PHILOX_M1, c2)
        c0, c1, c2, c3 = hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0
    return c0, c1, c2, c3


def uniform(seed, b, j, stream):
    """The uniform in [0, 1) for request ``b``, position ``j`` and ``stream``."""
    w0 = philox4x64_10((b, j, stream, 0), (seed, 0))[0]
    return float(w0 >> 40) * 2.0 ** -24
