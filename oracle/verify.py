"""Target verification of a draft block (oracle side, float64).

Test infrastructure only (see ``oracle/__init__.py``).

Sources:

* "Solar Open2 DSpark" (sionic.ai), section 1: the target checks the drafted tokens in
  one forward pass; when the leading candidates agree with the target, several tokens
  are committed at once and drafting restarts at the first disagreement.
* Same page, section 6: the verify forward covers gamma + 1 positions.
* "Speculative Decoding Part 2" (VESSL AI), section on blockwise parallel decoding:
  one forward verifies and the longest matching prefix is accepted (T=0 rule, with
  the draft compared to the argmax of each target position).
* The T=1 rule is standard speculative rejection sampling (accept x with probability
  min(1, p(x)/q(x)), else draw from normalize(max(0, p - q))); the pages name it only
  through the overlap 1 - TV ("SpecOPD" summary (onedev.kr), section "how to use it";
  VESSL page, DSpark section: the pass label alpha = 1 - D_TV).
* "SpecOPD" summary, section "premises and limits": an acceptance length counts the
  bonus token, so the reported length is n + 1.

Row alignment: target row i (i = 0..gamma) is the distribution p_{i+1} of position
i+1; draft row j-1 is q_j; draft token j-1 is x_j.

T=0, per request:
  n = largest k with x_j == argmax p_j for every j <= k (ties: lowest index)
  y = argmax p_{n+1}
T=1, per request, for j = 1..gamma in order:
  u = Philox(seed_b; b, j, 1); accept iff u * q_j(x_j) < p_j(x_j)   (u < p/q, no division)
  first rejection at k: y = inverse-CDF draw from max(0, p_k - q_k) with
  u = Philox(seed_b; b, k, 2); if that residual sums to zero, from p_k
  all accepted: y = inverse-CDF draw from p_{gamma+1} with u = Philox(seed_b; b, gamma+1, 3)
Output: n, committed = (x_1..x_n, y) padded with -1, bonus = y.

A request with a draft token outside [0, V) or an invalid row (see ``_rows``) among
the rows it reads gets n = -1, committed all -1 and bonus -1.

Pins (``tests/test_oracle_verify.py``): constructed drafts with a known first
mismatch; committed tokens equal the greedy chain read off the target rows; at T=1,
by exhaustive enumeration of every draft path at V <= 8, gamma <= 3 with a
prefix-dependent Markov draft (each decision integrated exactly over its uniform),
the first committed token is distributed as p_1, the token after k accepted drafts as
p_{k+1}, and each acceptance has probability sum_v min(p, q) = 1 - TV; the same
marginals by Monte Carlo; with prefix-independent rows E[n] = sum_j prod_{i<=j} a_i,
tying this module to ``e2etv``'s survival products.
"""

import numpy as np

from . import philox
from ._rows import NEAR_TIE, as_f64, row_valid, softmax, argmax_lowest, inverse_cdf


def verify_request(target, draft, tokens, temperature, seed, b, uniform=None):
    """Verify one request.  target [gamma+1, V], draft [gamma, V] or None, tokens [gamma].

    ``uniform`` (optional) is a callable (j, stream) -> u in [0, 1) that replaces the
    Philox draw u = Philox(seed; b, j, stream); the exhaustive pin integrates the rule
    over it.  Returns dict(n, committed [gamma+1], bonus, near).
    """
    if uniform is None:
        def uniform(j, stream):
            return philox.uniform(seed, b, j, stream)
    P = as_f64(target)
    gamma = P.shape[0] - 1
    V = P.shape[1]
    committed = np.full(gamma + 1, -1, dtype=np.int64)
    bad = dict(n=-1, committed=committed, bonus=-1, near=False)
    x = [int(t) for t in tokens]
    if any(not 0 <= t < V for t in x):
        return bad

    if temperature == 0:
        rows_needed = P
        if not all(row_valid(r) for r in rows_needed):
            return bad
        am = [argmax_lowest(r) for r in P]
        n = 0
        while n < gamma and x[n] == am[n]:
            n += 1
        y = am[n]
        committed[:n] = x[:n]
        committed[n] = y
        return dict(n=n, committed=committed, bonus=y, near=False)

    Q = as_f64(draft)
    if not all(row_valid(r) for r in P) or not all(row_valid(r) for r in Q):
        return bad
    near = False
    for j in range(1, gamma + 1):
        p, _, _ = softmax(P[j - 1])
        q, _, _ = softmax(Q[j - 1])
        xj = x[j - 1]
        u = uniform(j, philox.STREAM_ACCEPT)
        if abs(u * q[xj] - p[xj]) < NEAR_TIE * q[xj]:
            near = True
        if u * q[xj] < p[xj]:
            continue
        resid = np.maximum(0.0, p - q)
        if not resid.sum() > 0:
            resid = p
        y, nr = inverse_cdf(resid, uniform(j, philox.STREAM_RESIDUAL))
        n = j - 1
        committed[:n] = x[:n]
        committed[n] = y
        return dict(n=n, committed=committed, bonus=y, near=near or nr)
    p_last, _, _ = softmax(P[gamma])
    y, nr = inverse_cdf(p_last, uniform(gamma + 1, philox.STREAM_BONUS))
    committed[:gamma] = x
    committed[gamma] = y
    return dict(n=gamma, committed=committed, bonus=y, near=near or nr)


def verify(target, draft, tokens, temperature, seeds):
    """Verify a batch.  target [B, gamma+1, V]; draft [B, gamma, V] (None at T=0);
    tokens [B, gamma]; seeds [B].  Returns dict(n [B], committed [B, gamma+1],
    bonus [B], near [B])."""
    B = target.shape[0]
    gamma = target.shape[1] - 1
    n = np.zeros(B, dtype=np.int64)
    committed = np.zeros((B, gamma + 1), dtype=np.int64)
    bonus = np.zeros(B, dtype=np.int64)
    near = np.zeros(B, dtype=bool)
    for b in range(B):
        r = verify_request(target[b], None if draft is None else draft[b], tokens[b],
                           temperature, int(seeds[b]) if seeds is not None else 0, b)
        n[b], committed[b], bonus[b], near[b] = r["n"], r["committed"], r["bonus"], r["near"]
    return dict(n=n, committed=committed, bonus=bonus, near=near)


def acceptance_length(n):
    """Acceptance length as the pages count it: accepted drafts plus the bonus token."""
    return np.asarray(n) + 1
