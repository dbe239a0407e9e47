"""Pins for the oracle's verification step (no GPU)."""

import numpy as np
import pytest

from oracle import verify, e2etv


def _softmax(z):
    e = np.exp(z - z.max())
    return e / e.sum()


def test_t0_known_first_mismatch():
    rng = np.random.default_rng(0)
    g, V = 6, 50
    P = rng.normal(0, 2, size=(g + 1, V))
    am = P.argmax(-1)
    for k in range(g + 1):
        toks = am[:g].copy()
        if k < g:
            toks[k] = (am[k] + 1 + rng.integers(0, V - 1)) % V   # any other token
        r = verify.verify_request(P, None, toks, 0, 0, 0)
        assert r["n"] == k
        assert r["committed"][:k].tolist() == am[:k].tolist()
        assert r["committed"][k] == am[k] == r["bonus"]
        assert (r["committed"][k + 1:] == -1).all()


def test_t0_ties_lowest_index():
    P = np.zeros((3, 5))
    P[0, [1, 3]] = 2.0
    P[1, 4] = 1.0
    r = verify.verify_request(P, None, [3, 4], 0, 0, 0)
    assert r["n"] == 0 and r["bonus"] == 1
    r = verify.verify_request(P, None, [1, 4], 0, 0, 0)
    assert r["n"] == 2 and r["committed"].tolist() == [1, 4, 0]


def test_t0_speculative_equals_autoregressive_greedy():
    """Greedy speculative decoding reproduces the target's own greedy chain: a toy
    target whose next-token logits depend on the previous token, any draft."""
    rng = np.random.default_rng(1)
    V, g, n_out = 12, 4, 40
    T = rng.normal(0, 2, size=(V, V))          # target logits given previous token
    D = T + rng.normal(0, 1.5, size=(V, V))    # an imperfect greedy drafter
    x0 = 5
    ar = [x0]
    for _ in range(n_out):
        ar.append(int(T[ar[-1]].argmax()))
    out = [x0]
    rounds = 0
    while len(out) < n_out + 1:
        drafts = []
        prev = out[-1]
        for _ in range(g):
            prev = int(D[prev].argmax())
            drafts.append(prev)
        ctx = [out[-1]] + drafts
        rows = np.stack([T[t] for t in ctx])    # target row i predicts position i+1
        r = verify.verify_request(rows, None, drafts, 0, 0, 0)
        out.extend(int(t) for t in r["committed"][: r["n"] + 1])
        rounds += 1
    assert out[: n_out + 1] == ar
    assert rounds < n_out                       # the draft got some tokens accepted


def _run_t1(T, Dq, x0, g, seed, rng):
    """One speculative round with a Markov target T and Markov draft Dq (logits),
    draft tokens sampled from q with numpy's generator."""
    drafts = []
    prev = x0
    for _ in range(g):
        prev = int(rng.choice(len(Dq), p=_softmax(Dq[prev])))
        drafts.append(prev)
    ctx = [x0] + drafts
    P = np.stack([T[t] for t in ctx])
    Q = np.stack([Dq[t] for t in ctx[:-1]])
    return verify.verify_request(P, Q, drafts, 1, seed, 0)


def test_t1_output_marginals_equal_target():
    """Speculative sampling is exact: the first committed token is distributed as p_1,
    and the second, given the first was an accepted draft, as p_2(. | t_1)."""
    rng = np.random.default_rng(2)
    V, g, trials = 4, 2, 20000
    T = rng.normal(0, 1, size=(V, V))
    Dq = T + rng.normal(0, 1.0, size=(V, V))
    x0 = 0
    c1 = np.zeros(V)
    c2 = np.zeros((V, V))
    for s in range(trials):
        r = _run_t1(T, Dq, x0, g, s, rng)
        c1[r["committed"][0]] += 1
        if r["n"] >= 1:
            c2[r["committed"][0], r["committed"][1]] += 1
    p1 = _softmax(T[x0])
    sig = np.sqrt(p1 * (1 - p1) / trials)
    assert (np.abs(c1 / trials - p1) <= 4 * sig + 1e-9).all()
    for v in range(V):
        n_v = c2[v].sum()
        if n_v < 500:
            continue
        p2 = _softmax(T[v])
        sig = np.sqrt(p2 * (1 - p2) / n_v)
        assert (np.abs(c2[v] / n_v - p2) <= 4 * sig + 1e-9).all()


def test_t1_expected_accepts_equal_survival_sum():
    """Rows that do not depend on the prefix: E[n] = sum_j prod_{i<=j} a_i with
    a_i = 1 - TV(p_i, q_i), the e2etv oracle's overlap and survival routines."""
    rng = np.random.default_rng(3)
    V, g, trials = 6, 3, 20000
    P = rng.normal(0, 1, size=(g + 1, V))
    Q = P[:g] + rng.normal(0, 0.7, size=(g, V))
    a = np.array([e2etv.overlap(_softmax(P[i]), _softmax(Q[i]))[0] for i in range(g)])
    expected = e2etv.survival(a).sum()
    ns = np.empty(trials)
    for s in range(trials):
        toks = [int(rng.choice(V, p=_softmax(Q[j]))) for j in range(g)]
        ns[s] = verify.verify_request(P, Q, toks, 1, s, 0)["n"]
    assert abs(ns.mean() - expected) <= 4 * ns.std() / np.sqrt(trials)


def test_t1_identical_distributions_accept_everything():
    rng = np.random.default_rng(4)
    P = rng.normal(0, 1, size=(4, 9))
    for s in range(50):
        toks = rng.integers(0, 9, size=3)
        r = verify.verify_request(P, P[:3], toks, 1, s, 0)
        assert r["n"] == 3 and r["committed"][:3].tolist() == toks.tolist()


@pytest.mark.filterwarnings("ignore:divide by zero")
def test_t1_zero_draft_probability():
    # q(x) = 0 while p(x) > 0: u * 0 < p(x) accepts; p(x) = 0 and q(x) > 0 rejects
    P = np.log(np.array([[0.5, 0.5, 1e-300], [0.2, 0.8, 0.0]]))
    Q = np.log(np.array([[1.0, 1e-300, 1e-300]]))
    Q[0, 1] = -np.inf
    r = verify.verify_request(P, Q, [1], 1, 0, 0)
    assert r["n"] == 1
    P2 = P.copy()
    P2[0] = np.log(np.array([0.0, 1.0, 0.0]) + 1e-320)
    P2[0, 0] = -np.inf
    r = verify.verify_request(P2, np.log(np.array([[1.0, 1e-9, 1e-9]])), [0], 1, 0, 0)
    assert r["n"] == 0 and r["bonus"] == 1     # residual max(0, p - q) sits on token 1


def test_invalid_requests():
    P = np.zeros((3, 4))
    r = verify.verify_request(P, None, [0, 4], 0, 0, 0)
    assert r["n"] == -1 and (r["committed"] == -1).all() and r["bonus"] == -1
    P[1, 2] = np.inf
    assert verify.verify_request(P, None, [0, 0], 0, 0, 0)["n"] == -1
    P[1, 2] = np.nan
    assert verify.verify_request(P, P[:2], [0, 0], 1, 0, 0)["n"] == -1


def test_acceptance_length_counts_bonus():
    assert verify.acceptance_length([0, 3, 7]).tolist() == [1, 4, 8]


def test_philox_stream_layout_read_off():
    """Rows built so each draw can be read off its uniform: the accept test uses
    stream 1 at position j, the residual stream 2 at the rejected position, the bonus
    stream 3 at position gamma + 1."""
    from oracle import philox
    lo = np.log
    for seed in range(20):
        # accept ratio p/q = 1/2 at j = 1: accept iff u_1 < 1/2
        P = lo(np.array([[0.5, 0.5], [0.5, 0.5]]))
        Q = lo(np.array([[1e-300, 1.0]]))
        Q[0, 0] = -np.inf
        r = verify.verify_request(P, Q, [1], 1, seed, 2)
        u1 = philox.uniform(seed, 2, 1, philox.STREAM_ACCEPT)
        assert (r["n"] == 1) == (u1 < 0.5)
        if r["n"] == 1:       # bonus from p_2 = (1/2, 1/2)
            assert r["bonus"] == int(philox.uniform(seed, 2, 2, philox.STREAM_BONUS) >= 0.5)
        else:                 # residual max(0, p - q) = (1/2, 0) -> token 0
            assert r["bonus"] == 0
        # certain rejection at j = 2 with an even residual over tokens 1 and 2
        P = np.log(np.array([[1.0, 1e-300, 1e-300], [1e-300, 0.5, 0.5], [1.0, 1e-300, 1e-300]]))
        P[0, 1:] = P[1, 0] = P[2, 1:] = -np.inf
        Q = P[:2].copy()
        Q[1] = np.array([0.0, -np.inf, -np.inf])
        r = verify.verify_request(P, Q, [0, 0], 1, seed, 5)
        u2 = philox.uniform(seed, 5, 2, philox.STREAM_RESIDUAL)
        assert r["n"] == 1 and r["bonus"] == 1 + int(u2 >= 0.5)


def test_inverse_cdf_strict_boundary():
    """The draw is the smallest v with C_v > u*Z: a threshold exactly on a boundary
    goes to the next token."""
    from oracle._rows import inverse_cdf
    assert inverse_cdf(np.array([1.0, 1.0]), 0.5)[0] == 1
    assert inverse_cdf(np.array([1.0, 0.0, 3.0]), 0.25)[0] == 2
    assert inverse_cdf(np.array([0.0, 2.0, 2.0]), 0.0)[0] == 1
