"""Row-level helpers shared by the oracle modules (float64 throughout).

Test infrastructure only (see ``oracle/__init__.py``).

Readings of the pages that these helpers encode (the pages are silent on them):

* ties in an argmax go to the lowest vocabulary index;
* sampling is a single-uniform inverse CDF in vocabulary-index order: the token is the
  smallest v with C_v > u * Z, where C_v is the running sum of the weights in index
  order and Z their total; if rounding leaves no such v, the last v of positive weight;
* a logit of -inf is a token of probability zero; a row holding NaN or +inf, or no
  finite entry at all, has no distribution and is reported invalid.
"""

import numpy as np

# Draws that land this close to a decision threshold (relative to the scale of the
# quantity compared) are "near-ties": float32 on the GPU may legitimately decide them
# the other way, so parity tests count them instead of failing on them.
NEAR_TIE = 1e-6


def as_f64(x):
    return np.asarray(x, dtype=np.float64)


def row_valid(z):
    """True when the row defines a distribution: no NaN, no +inf, some finite entry."""
    if np.isnan(z).any() or np.isposinf(z).any():
        return False
    return bool(np.isfinite(z).any())


def softmax(z):
    """Return (p, m, Z) with p = exp(z - m) / Z, m = max z, Z = sum exp(z - m)."""
    m = float(np.max(z))
    e = np.exp(z - m)
    Z = float(np.sum(e))
    return e / Z, m, Z


def argmax_lowest(z):
    """Index of the maximum; ties go to the lowest index (numpy's argmax does that)."""
    return int(np.argmax(z))


def top2_gap(z):
    """Difference between the largest entry and the largest entry at another index."""
    i = int(np.argmax(z))
    rest = np.delete(z, i)
    if rest.size == 0:
        return np.inf
    return float(z[i] - np.max(rest))


def inverse_cdf(w, u):
    """Inverse-CDF draw from non-negative weights ``w`` with uniform ``u`` in [0, 1).

    Returns (v, near): v is the smallest index with C_v > u * Z; ``near`` flags a
    draw whose threshold u * Z lies within NEAR_TIE * Z of a boundary C_{v-1} or C_v
    between two tokens that both have positive weight.
    """
    C = np.cumsum(w)
    Z = float(C[-1])
    t = u * Z
    v = int(np.searchsorted(C, t, side="right"))
    if v >= len(w):
        v = int(np.nonzero(w > 0)[0][-1])
    near = abs(C[v] - t) < NEAR_TIE * Z and v + 1 < len(w) and bool((w[v + 1:] > 0).any())
    if v > 0 and C[v - 1] > 0 and abs(C[v - 1] - t) < NEAR_TIE * Z:
        near = True
    return v, bool(near)
