"""Verify-budget scheduler (oracle side, float64).

Test infrastructure only (see ``oracle/__init__.py``).

Source: "Speculative Decoding Part 2: the evolution of drafter architectures" (VESSL
AI), DSpark section, the paragraphs after the bias equation.  A confidence head gives,
for each position, the probability that it passes given that every earlier position
passed.  A scheduler multiplies these into expected lengths (which is why the values
must be calibrated), gives the verification budget to the positions with the highest
pass probability across all requests of the batch, and maximises throughput against a
measured hardware curve, so gamma varies per request and with load.

The pages give no formula; this module takes the plainest reading:

  c[b, j] is clamped to [0, 1], NaN read as 0; P[b, j] = prod_{i <= j} c[b, i] is the
  probability that draft position j of request b is accepted (positions counted from 1).
  Candidates (b, j) are ordered by P descending, ties by the flat index b * gamma + j
  ascending.  P never grows with j, so the first k candidates hold a prefix of every
  request's positions.
  E(k) = B + (sum of the first k P): the expected committed tokens when k draft
  positions are verified in all (each request commits its accepted drafts and one more
  token).
  With a cost curve t[0..K] (time to verify k positions in all): k* = argmax over
  k = 0..K of E(k) / t[k], the smallest k on ties, a non-positive or NaN t[k] excluded.
  Without one: k* = K.
  gamma_b = number of request b's candidates among the first k*.

Pins (``tests/test_oracle_schedule.py``): brute force over every prefix-closed
allocation with at most K positions on small batches; the pages' compounding example
(10 % high per position is about 95 % high at gamma = 7); closed forms with all c = 1
or one request.
"""

import numpy as np


def pass_products(conf):
    """P[b, j] = prod_{i <= j} clamp(c[b, i]) in float64, in position order."""
    c = np.asarray(conf, dtype=np.float64)
    c = np.where(np.isnan(c), 0.0, np.clip(c, 0.0, 1.0))
    return np.cumprod(c, axis=1)


def candidate_order(P):
    """Flat candidate indices by P descending, ties by flat index ascending."""
    flat = P.reshape(-1)
    # lexsort sorts by the last key first: -P, then the index
    return np.lexsort((np.arange(flat.size), -flat))


def expected_committed(P, order):
    """E(k) for k = 0..N: B + sum of the first k candidates' P (plain running sum)."""
    B = P.shape[0]
    flat = P.reshape(-1)[order]
    E = np.empty(flat.size + 1, dtype=np.float64)
    E[0] = B
    run = float(B)
    for k, v in enumerate(flat):
        run += v
        E[k + 1] = run
    return E


def schedule(conf, budget, cost=None):
    """Returns dict(gamma=int array [B], k=k*, expected=E(k*), objective=array or None).

    conf: [B, gamma] confidences; budget: K (at most B * gamma positions in all);
    cost: optional [K + 1] times t[0..K]."""
    conf = np.asarray(conf, dtype=np.float64)
    B, G = conf.shape
    K = int(min(max(budget, 0), B * G))
    P = pass_products(conf)
    order = candidate_order(P)
    E = expected_committed(P, order)
    obj = None
    if cost is None:
        k_star = K
    else:
        t = np.asarray(cost, dtype=np.float64)[:K + 1]
        obj = np.full(K + 1, -np.inf)
        ok = np.isfinite(t) & (t > 0)
        obj[ok] = E[:K + 1][ok] / t[ok]
        k_star = int(np.argmax(obj)) if np.isfinite(obj).any() else 0   # first maximum
    gamma = np.zeros(B, dtype=np.int64)
    for idx in order[:k_star]:
        gamma[idx // G] += 1
    return dict(gamma=gamma, k=k_star, expected=float(E[k_star]), objective=obj)
