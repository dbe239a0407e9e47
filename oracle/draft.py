"""DSpark block draft with the low-rank Markov logit bias (oracle side, float64).

Test infrastructure only (see ``oracle/__init__.py``).

Sources:

* "Speculative Decoding Part 2: the evolution of drafter architectures" (VESSL AI),
  section on DSpark, bias equation: B(x_{k-1}, .) = W_1[x_{k-1}] W_2 in R^V with
  W_1 in R^{V x r}, W_2 in R^{r x V}; the bias is added to every position's scores
  from the parallel backbone, so position k depends on the token chosen at k-1
  ("a light sequential step").
* Same page and section, confidence paragraph: a per-position pass probability.  The
  learned head is out of scope; the confidence here is c_j = max_v softmax(z_j)_v.
* "Solar Open2 DSpark" (sionic.ai), section 2: DSpark adds a low-rank Markov
  correction and per-position confidence to a DFlash parallel block.

Layout: U holds W_1 ([V, r], row x is the r-vector of token x) and Wt holds W_2
transposed ([V, r], row v is column v of W_2), so that
bias_v = sum_k U[x_{j-1}, k] * Wt[v, k].  Position 1 uses the anchor token as x_0.

Steps for each request b, positions j = 1..gamma, in order:

1. z_j = l_j + Wt @ U[x_{j-1}]                     (logits plus Markov bias)
2. m = max z_j,  Z = sum exp(z_j - m),  c_j = 1/Z   (softmax at temperature 1)
3. T=0: x_j = lowest index attaining m
   T=1: x_j = inverse-CDF draw from exp(z_j - m) with u = Philox(seed_b; b, j, 0)
4. q_j(x_j) = exp(z_{j, x_j} - m) / Z

Pins (``tests/test_oracle_draft.py``): W = 0 and r = 0 reduce to a plain argmax /
softmax sample; for tiny V the T=0 chain is the unique token path that satisfies the
recurrence (found by brute force over all V**gamma paths); the T=1 path distribution
equals prod_j q_j(x_j | x_{j-1}) (stratified uniforms over all paths); at V=2 the
confidence has the closed form sigmoid(|z_1 - z_0|).
"""

import numpy as np

from . import philox
from ._rows import NEAR_TIE, as_f64, row_valid, softmax, argmax_lowest, top2_gap, inverse_cdf


def draft_step(l_row, x_prev, U, Wt, temperature, u):
    """One position of the chain: returns dict(x, conf, qtok, near, z).

    ``l_row`` [V] logits, ``x_prev`` previous token (anchor at j=1), ``U``/``Wt``
    [V, r] or None for no bias, ``u`` the uniform for T=1 (ignored at T=0).
    """
    z = as_f64(l_row).copy()
    if not 0 <= x_prev < z.shape[0]:
        return dict(x=-1, conf=np.nan, qtok=np.nan, near=False, z=np.full_like(z, np.nan))
    has_bias = U is not None and Wt is not None and U.shape[1] > 0
    if has_bias:
        z = z + Wt @ U[x_prev]
    if not row_valid(z):
        return dict(x=-1, conf=np.nan, qtok=np.nan, near=False, z=z)
    p, m, Z = softmax(z)
    if temperature == 0:
        x = argmax_lowest(z)
        # float32 on the GPU decides the argmax the same way unless the top two
        # biased logits are closer than the rounding of z itself
        near = has_bias and top2_gap(z) < NEAR_TIE * max(1.0, abs(m))
    else:
        x, near = inverse_cdf(np.exp(z - m), u)
    return dict(x=x, conf=1.0 / Z, qtok=float(p[x]), near=bool(near), z=z)


def draft_block(logits, anchor, U, Wt, temperature, seeds, return_z=False, first_b=0):
    """Run the sequential chain for every request.

    logits [B, gamma, V]; anchor [B]; U, Wt [V, r] (or None); seeds [B] uint64.
    ``first_b`` is the index of request 0 in the whole batch (the Philox counter's
    request index), so that a slice of a batch can be replayed on its own.
    Returns dict with tokens [B, gamma] (int64), conf, qtok [B, gamma] (float64),
    near [B, gamma] (bool), valid [B] (bool) and, if ``return_z``, z [B, gamma, V].
    A request whose row j is invalid (see ``_rows``), or whose anchor lies outside
    [0, V), gets token -1 and NaN statistics from that position on.
    """
    L = as_f64(logits)
    B, gamma, V = L.shape
    if U is not None:
        U = as_f64(U)
        Wt = as_f64(Wt)
    tokens = np.full((B, gamma), -1, dtype=np.int64)
    conf = np.full((B, gamma), np.nan)
    qtok = np.full((B, gamma), np.nan)
    near = np.zeros((B, gamma), dtype=bool)
    valid = np.ones(B, dtype=bool)
    zs = np.full((B, gamma, V), np.nan) if return_z else None
    for b in range(B):
        x_prev = int(anchor[b])
        for j in range(1, gamma + 1):
            u = philox.uniform(int(seeds[b]), first_b + b, j, philox.STREAM_DRAFT) if temperature else 0.0
            step = draft_step(L[b, j - 1], x_prev, U, Wt, temperature, u)
            if return_z:
                zs[b, j - 1] = step["z"]
            if step["x"] < 0:
                valid[b] = False
                break
            tokens[b, j - 1] = step["x"]
            conf[b, j - 1] = step["conf"]
            qtok[b, j - 1] = step["qtok"]
            near[b, j - 1] = step["near"]
            x_prev = step["x"]
    out = dict(tokens=tokens, conf=conf, qtok=qtok, near=near, valid=valid)
    if return_z:
        out["z"] = zs
    return out
