"""Exhaustive pin of the oracle's T=1 verification (no GPU).

Speculative sampling is exact: whatever the draft distribution q, the tokens that one
verification commits are distributed as the target's own autoregressive chain, and each
draft is accepted (given the earlier ones were) with probability sum_v min(p, q) =
1 - TV(p, q) ("SpecOPD" summary (onedev.kr), section "how to use it"; "Speculative
Decoding Part 2" (VESSL AI), DSpark section: alpha = 1 - D_TV).

The test enumerates every draft path of a tiny vocabulary (V <= 8, gamma <= 3) and, for
each, integrates the oracle's decisions over their uniforms exactly:

* the accept test of position j is a step function of its uniform u (accepted for u
  below some threshold); the threshold is found by bisecting the oracle's own decision to
  below 1e-15, and its measure is the acceptance probability;
* the residual and bonus draws are non-decreasing step functions of their uniform (an
  inverse CDF); the breakpoints are found the same way, and the lengths of the intervals
  are the probabilities of the tokens.

Nothing here restates the accept rule or the residual: the probabilities come from
calling ``verify_request`` with chosen uniforms.  The draft is a prefix-dependent Markov
draft (rank-2 bias large enough to change the rows), and the target rows depend on the
previous token too.  The assertions hold to 1e-12:

  (i)   P(t_1 = v) = p_1(v);
  (ii)  P(t_{k+1} = w | the first k committed tokens are the accepted drafts s) =
        p_{k+1}(w | s), for every accepted prefix s with 1 <= k <= gamma;
  (iii) P(accept_k | the first k-1 drafts accepted as s) = sum_v min(p_k, q_k)(. | s).
"""

from collections import defaultdict

import numpy as np
import pytest

from oracle import verify

TOL_BISECT = 1e-15


def _softmax(z):
    e = np.exp(z - z.max())
    return e / e.sum()


def _first_true(pred):
    """inf{u in [0, 1] : pred(u)} for a predicate that is false then true in u."""
    if pred(0.0):
        return 0.0
    hi_u = np.nextafter(1.0, 0.0)
    if not pred(hi_u):
        return 1.0
    lo, hi = 0.0, hi_u
    while hi - lo > TOL_BISECT:
        mid = 0.5 * (lo + hi)
        if pred(mid):
            hi = mid
        else:
            lo = mid
    return hi


def _draw_distribution(draw, V):
    """Token probabilities of a non-decreasing step function draw(r), r uniform in [0, 1)."""
    probs = np.zeros(V)
    prev = 0.0
    for v in range(V - 1):
        b = _first_true(lambda r: draw(r) > v)
        probs[v] = b - prev
        prev = b
    probs[V - 1] = 1.0 - prev
    return probs


class Problem:
    """A Markov target and a Markov draft with a rank-r bias, over V tokens."""

    def __init__(self, V, g, r, seed):
        rng = np.random.default_rng(seed)
        self.V, self.g = V, g
        self.A = rng.normal(0, 1.5, size=(g + 1, V, V))   # target logits of position j+1 given x_j
        self.L = rng.normal(0, 1.0, size=(g, V))          # drafter logits per position
        self.U = rng.normal(0, 1.2, size=(V, r))          # W_1
        self.W = rng.normal(0, 1.2, size=(r, V))          # W_2
        self.x0 = int(rng.integers(0, V))

    def p(self, j, prev):          # target distribution of position j (1-based)
        return _softmax(self.A[j - 1][prev])

    def qlogits(self, j, prev):    # draft logits of position j: l_j + W_1[x_{j-1}] W_2
        return self.L[j - 1] + self.U[prev] @ self.W

    def q(self, j, prev):
        return _softmax(self.qlogits(j, prev))

    def run(self, toks, us):
        ctx = [self.x0] + list(toks)
        P = np.stack([self.A[i][ctx[i]] for i in range(self.g + 1)])
        Q = np.stack([self.qlogits(i + 1, ctx[i]) for i in range(self.g)])
        return verify.verify_request(P, Q, list(toks), 1, 0, 0, uniform=lambda j, s: us.get((j, s), 0.0))


def exact_outcomes(pb):
    """Probability of every outcome (n, committed tokens) of one verification, with the
    draft path drawn from q and every uniform integrated out."""
    V, g = pb.V, pb.g
    out = defaultdict(float)

    def rec(prefix, w):
        k = len(prefix)
        if k == g:   # all accepted: the bonus draw (stream 3 at position g+1)
            toks = list(prefix)
            probs = _draw_distribution(lambda r: pb.run(toks, {(g + 1, 3): r})["bonus"], V)
            for y in range(V):
                if probs[y] > 0:
                    out[(g, tuple(prefix) + (y,))] += w * probs[y]
            return
        j = k + 1
        q = pb.q(j, pb.x0 if k == 0 else prefix[-1])
        for x in range(V):
            toks = list(prefix) + [x] + [0] * (g - j)
            # earlier uniforms are 0: accepted whenever p > 0, which holds for these rows
            t = _first_true(lambda u: pb.run(toks, {(j, 1): u})["n"] < j)
            if t > 0:
                rec(prefix + (x,), w * q[x] * t)
            if t < 1:
                ur = 0.5 * (t + 1.0)
                assert pb.run(toks, {(j, 1): ur})["n"] == k
                probs = _draw_distribution(lambda r: pb.run(toks, {(j, 1): ur, (j, 2): r})["bonus"], V)
                for y in range(V):
                    if probs[y] > 0:
                        out[(k, tuple(prefix) + (y,))] += w * q[x] * (1.0 - t) * probs[y]

    rec((), 1.0)
    return out


@pytest.mark.parametrize("V,g,r,seed", [(5, 3, 2, 11), (8, 2, 2, 12), (2, 3, 1, 20)])
def test_t1_exhaustive_marginals(V, g, r, seed):
    pb = Problem(V, g, r, seed)
    # the bias really changes the draft rows (the draft is prefix-dependent)
    spread = max(np.abs(pb.q(1, a) - pb.q(1, b)).max() for a in range(V) for b in range(V))
    assert spread > 0.2
    out = exact_outcomes(pb)
    assert abs(sum(out.values()) - 1.0) <= 1e-12

    # (i) the first committed token
    m1 = np.zeros(V)
    for (n, c), pr in out.items():
        m1[c[0]] += pr
    assert np.abs(m1 - pb.p(1, pb.x0)).max() <= 1e-12

    # accepted prefixes s (length k): mass of {n >= k, committed[:k] = s} and the
    # distribution of committed[k] on that event
    mass = defaultdict(float)
    nxt = defaultdict(lambda: np.zeros(V))
    for (n, c), pr in out.items():
        for k in range(0, n + 1):
            s = c[:k]
            mass[s] += pr
            nxt[s][c[k]] += pr
    assert abs(mass[()] - 1.0) <= 1e-12
    checked = 0
    for s, ms in mass.items():
        k = len(s)
        if k == 0:
            continue
        prev = s[-1]
        # (ii) the token after k accepted drafts follows p_{k+1}(. | s)
        assert np.abs(nxt[s] / ms - pb.p(k + 1, prev)).max() <= 1e-12 / ms, s
        # (iii) the k-th acceptance, given the first k-1 accepted as s[:-1]
        parent = s[:-1]
        pprev = pb.x0 if k == 1 else parent[-1]
        acc_mass = sum(mass[parent + (x,)] for x in range(V))
        overlap = np.minimum(pb.p(k, pprev), pb.q(k, pprev)).sum()
        assert abs(acc_mass / mass[parent] - overlap) <= 1e-12 / mass[parent], s
        checked += 1
    assert checked == sum(V ** k for k in range(1, g + 1))


def test_exhaustive_pin_catches_a_biased_residual():
    """The pin fails for a plausible mistake: a residual drawn from p instead of
    max(0, p - q) (planted in a copy of the rule, on the CPU)."""
    pb = Problem(4, 2, 2, 21)
    orig = verify.verify_request

    def wrong(P, Q, toks, T, seed, b, uniform=None):
        r = orig(P, Q, toks, T, seed, b, uniform=uniform)
        if 0 <= r["n"] < len(toks):   # a rejection: redraw y from p with the same uniform
            from oracle._rows import inverse_cdf
            p = _softmax(np.asarray(P[r["n"]], dtype=np.float64))
            y, _ = inverse_cdf(p, uniform(r["n"] + 1, 2))
            r = dict(r)
            r["bonus"] = y
        return r

    verify.verify_request = wrong
    try:
        out = exact_outcomes(pb)
    finally:
        verify.verify_request = orig
    m1 = np.zeros(4)
    for (n, c), pr in out.items():
        m1[c[0]] += pr
    assert np.abs(m1 - pb.p(1, pb.x0)).max() > 1e-3
