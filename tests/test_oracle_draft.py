"""Pins for the oracle's DSpark block draft (no GPU).

The bias is restated here in the page's own orientation, B(x, .) = W_1[x] W_2 with
W_2 of shape [r, V], while the oracle takes W_2 transposed; a transposed operand or
a wrong previous token in the oracle fails these tests.
"""

import itertools

import numpy as np
import pytest

from oracle import draft, philox


def _page_bias(W1, W2, x):
    return W1[x] @ W2          # row vector W_1[x] (1 x r) times W_2 (r x V)


def _softmax(z):
    e = np.exp(z - z.max())
    return e / e.sum()


def test_zero_bias_reduces_to_argmax():
    rng = np.random.default_rng(0)
    B, g, V, r = 3, 5, 97, 4
    L = rng.normal(0, 3, size=(B, g, V))
    W1 = rng.normal(0, 1, size=(V, r))
    W2 = np.zeros((r, V))
    anchor = rng.integers(0, V, size=B)
    out = draft.draft_block(L, anchor, W1, W2.T.copy(), 0, np.zeros(B, np.uint64))
    assert (out["tokens"] == L.argmax(-1)).all()
    out0 = draft.draft_block(L, anchor, None, None, 0, np.zeros(B, np.uint64))
    assert (out0["tokens"] == L.argmax(-1)).all()
    # confidence is the max probability of the softmax row
    for b in range(B):
        for j in range(g):
            assert out0["conf"][b, j] == pytest.approx(_softmax(L[b, j]).max(), rel=1e-12)


def test_argmax_ties_go_to_lowest_index():
    L = np.zeros((1, 2, 6))
    L[0, 0, [2, 4]] = 5.0
    L[0, 1, [1, 5]] = 3.0
    out = draft.draft_block(L, [0], None, None, 0, [0])
    assert out["tokens"].tolist() == [[2, 1]]


def test_t0_chain_is_unique_path_of_recurrence():
    """Brute force over all V**gamma token paths: exactly one satisfies
    x_j = argmax(l_j + W_1[x_{j-1}] W_2) for every j, and it is the oracle's chain."""
    rng = np.random.default_rng(1)
    V, g, r = 5, 4, 2
    for trial in range(20):
        L = rng.normal(0, 1, size=(g, V))
        W1 = rng.normal(0, 1.5, size=(V, r))
        W2 = rng.normal(0, 1.5, size=(r, V))    # large: the bias flips argmaxes
        x0 = int(rng.integers(0, V))
        good = []
        for path in itertools.product(range(V), repeat=g):
            prev = x0
            ok = True
            for j in range(g):
                z = L[j] + _page_bias(W1, W2, prev)
                if int(np.argmax(z)) != path[j]:
                    ok = False
                    break
                prev = path[j]
            if ok:
                good.append(path)
        assert len(good) == 1
        out = draft.draft_block(L[None], [x0], W1, W2.T.copy(), 0, [0])
        assert tuple(out["tokens"][0]) == good[0]


def test_bias_changes_the_chain():
    # guard that the pins above exercise the bias: it must flip some argmax
    rng = np.random.default_rng(1)
    V, g, r = 5, 4, 2
    flipped = 0
    for trial in range(20):
        L = rng.normal(0, 1, size=(g, V))
        W1 = rng.normal(0, 1.5, size=(V, r))
        W2 = rng.normal(0, 1.5, size=(r, V))
        x0 = int(rng.integers(0, V))
        out = draft.draft_block(L[None], [x0], W1, W2.T.copy(), 0, [0])
        flipped += int((out["tokens"][0] != L.argmax(-1)).any())
    assert flipped >= 5


def test_t1_step_distribution_stratified():
    """With stratified uniforms the sampled token frequencies equal softmax(z) to
    within one grid cell per CDF boundary."""
    rng = np.random.default_rng(2)
    V, r, M = 7, 3, 20000
    l = rng.normal(0, 1.5, size=V)
    W1 = rng.normal(0, 1, size=(V, r))
    W2 = rng.normal(0, 1, size=(r, V))
    x_prev = 3
    q = _softmax(l + _page_bias(W1, W2, x_prev))
    counts = np.zeros(V)
    for i in range(M):
        s = draft.draft_step(l, x_prev, W1, W2.T.copy(), 1, (i + 0.5) / M)
        counts[s["x"]] += 1
        if i == 0:
            assert s["conf"] == pytest.approx(q.max(), rel=1e-12)
    assert np.abs(counts / M - q).max() <= 2.0 / M


def test_t1_path_distribution_conditional():
    """P(x_1, x_2) = q_1(x_1 | x_0) q_2(x_2 | x_1): each position's sampler, fed the
    previous token, reproduces the conditional computed from the page's bias."""
    rng = np.random.default_rng(3)
    V, r, M = 4, 2, 8000
    L = rng.normal(0, 1, size=(2, V))
    W1 = rng.normal(0, 1, size=(V, r))
    W2 = rng.normal(0, 1, size=(r, V))
    x0 = 1
    Wt = W2.T.copy()
    # marginal of x_1
    c1 = np.zeros(V)
    for i in range(M):
        c1[draft.draft_step(L[0], x0, W1, Wt, 1, (i + 0.5) / M)["x"]] += 1
    q1 = _softmax(L[0] + _page_bias(W1, W2, x0))
    assert np.abs(c1 / M - q1).max() <= 2.0 / M
    # conditional of x_2 for every x_1
    for x1 in range(V):
        c2 = np.zeros(V)
        for i in range(M):
            c2[draft.draft_step(L[1], x1, W1, Wt, 1, (i + 0.5) / M)["x"]] += 1
        q2 = _softmax(L[1] + _page_bias(W1, W2, x1))
        assert np.abs(c2 / M - q2).max() <= 2.0 / M


def test_t1_block_monte_carlo_matches_product():
    """The whole block with Philox draws: path frequencies over seeds match
    prod_j q_j(x_j | x_{j-1}) within 4 sigma."""
    rng = np.random.default_rng(4)
    V, r, g, trials = 3, 2, 2, 6000
    L = rng.normal(0, 1, size=(1, g, V))
    W1 = rng.normal(0, 1, size=(V, r))
    W2 = rng.normal(0, 1, size=(r, V))
    x0 = 2
    counts = {}
    for s in range(trials):
        t = tuple(draft.draft_block(L, [x0], W1, W2.T.copy(), 1, [s])["tokens"][0])
        counts[t] = counts.get(t, 0) + 1
    for path in itertools.product(range(V), repeat=g):
        prob = 1.0
        prev = x0
        for j in range(g):
            prob *= _softmax(L[0, j] + _page_bias(W1, W2, prev))[path[j]]
            prev = path[j]
        f = counts.get(path, 0) / trials
        sigma = np.sqrt(prob * (1 - prob) / trials)
        assert abs(f - prob) <= 4 * sigma + 1e-9


def test_confidence_closed_form_v2():
    """V = 2: max prob = 1 / (1 + exp(-|z_1 - z_0|)) = sigmoid(|delta|)."""
    rng = np.random.default_rng(5)
    for _ in range(20):
        l = rng.normal(0, 2, size=2)
        s = draft.draft_step(l, 0, None, None, 0, 0.0)
        d = abs(l[1] - l[0])
        assert s["conf"] == pytest.approx(1.0 / (1.0 + np.exp(-d)), rel=1e-14)
        assert s["x"] == int(l[1] > l[0])


def test_invalid_rows_and_anchor():
    L = np.zeros((2, 3, 4))
    L[0, 1, 2] = np.nan
    out = draft.draft_block(L, [0, 9], None, None, 0, [0, 0])
    assert out["tokens"][0].tolist() == [0, -1, -1]
    assert out["tokens"][1].tolist() == [-1, -1, -1]
    assert not out["valid"].any()
    L = np.full((1, 1, 4), -np.inf)
    L[0, 0, 3] = 0.0                       # -inf entries are zero-probability tokens
    out = draft.draft_block(L, [0], None, None, 1, [7])
    assert out["tokens"].tolist() == [[3]] and out["conf"][0, 0] == 1.0
    L = np.full((1, 1, 4), -np.inf)        # no finite entry: no distribution
    assert draft.draft_block(L, [0], None, None, 0, [0])["tokens"].tolist() == [[-1]]


def test_uniform_drawn_per_position_stream0():
    """T=1 draws use Philox(seed_b; b, j, stream 0): a V=2 row of equal weights maps
    u < 1/2 to token 0, so the chain reads off the uniforms directly."""
    L = np.zeros((2, 4, 2))
    out = draft.draft_block(L, [0, 1], None, None, 1, [11, 11])
    for b in range(2):
        for j in range(1, 5):
            u = philox.uniform(11, b, j, philox.STREAM_DRAFT)
            assert out["tokens"][b, j - 1] == int(u >= 0.5)
