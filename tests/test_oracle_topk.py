"""Pins of the top-k / top-p oracle (oracle/topk.py), on the CPU.

The filter is tied to a worked example with exact values and to its defining
properties (shortest prefix reaching top_p, at most k entries, lowest index on boundary
ties); the filtered chain and verification reduce to the pinned unfiltered oracles when
nothing is filtered; and the rejection rule on filtered rows still commits tokens
distributed as the filtered target row.
"""

import os

import numpy as np
import pytest

from oracle import draft as od, philox, topk as ot, verify as ov

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _setting():
    vals = {}
    for line in open(os.path.join(GOLDEN, "dspine_sampling_setting.txt")):
        if "=" in line and not line.startswith("#"):
            k, v = line.strip().split("=")
            vals[k] = float(v)
    return int(vals["top_k"]), vals["top_p"], int(vals["temperature"])


def test_worked_example():
    # probabilities 0.5, 0.3, 0.15, 0.05 placed at indices 2, 0, 3, 1
    probs = np.array([0.3, 0.05, 0.5, 0.15])
    z = np.log(probs)
    pf, kept = ot.filtered(z, 4, 0.8)          # 0.5 + 0.3 reaches 0.8
    assert kept.tolist() == [0, 2]
    assert np.allclose(pf, [0.375, 0.0, 0.625, 0.0], atol=1e-15)
    pf, kept = ot.filtered(z, 4, 0.81)         # needs the 0.15 as well
    assert kept.tolist() == [0, 2, 3]
    assert np.allclose(pf[[0, 2, 3]], np.array([0.3, 0.5, 0.15]) / 0.95, atol=1e-15)
    pf, kept = ot.filtered(z, 2, 1.0)          # top-k alone
    assert kept.tolist() == [0, 2]
    # top-p over the top-k set renormalised: 0.5/0.8 = 0.625 < 0.7 <= 1
    pf, kept = ot.filtered(z, 2, 0.7)
    assert kept.tolist() == [0, 2]
    pf, kept = ot.filtered(z, 2, 0.6)
    assert kept.tolist() == [2]


@pytest.mark.parametrize("seed", range(6))
def test_shortest_prefix_and_at_most_k(seed):
    rng = np.random.default_rng(seed)
    z = rng.normal(0, 2, size=300)
    k, top_p, _ = _setting()
    pf, kept = ot.filtered(z, k, top_p)
    p = np.exp(z - z.max())
    p /= p.sum()
    top = np.argsort(-z, kind="stable")[:k]
    pt = np.sort(p[top])[::-1] / p[top].sum()
    n = len(kept)
    assert 1 <= n <= k
    assert pt[:n].sum() >= top_p - 1e-15
    assert n == 1 or pt[:n - 1].sum() < top_p
    # the kept entries are the n largest, and pf is p renormalised on them
    assert set(kept.tolist()) == set(top[:n].tolist())
    assert abs(pf.sum() - 1.0) < 1e-12 and (pf[kept] > 0).all()
    assert np.allclose(pf[kept], p[kept] / p[kept].sum(), rtol=1e-12)


def test_argmax_limits_and_boundary_ties():
    z = np.array([1.0, 3.0, 3.0, -2.0, 3.0])
    pf, kept = ot.filtered(z, 1, 1.0)
    assert kept.tolist() == [1]                 # three-way tie: lowest index
    pf, kept = ot.filtered(z, 2, 1.0)
    assert kept.tolist() == [1, 2]
    pf, kept = ot.filtered(z, 5, 1e-9)          # a tiny top_p keeps the top entry
    assert kept.tolist() == [1]


def test_nothing_filtered_reduces_to_the_plain_oracles():
    rng = np.random.default_rng(9)
    B, G, V, r = 3, 4, 40, 3
    L = rng.normal(0, 2, size=(B, G, V))
    U = rng.normal(0, 0.5, size=(V, r))
    Wt = rng.normal(0, 0.5, size=(V, r))
    anchor = rng.integers(0, V, size=B)
    seeds = np.arange(5, 5 + B, dtype=np.uint64)
    plain = od.draft_block(L, anchor, U, Wt, 1, seeds)
    filt = ot.draft_block_filtered(L, anchor, U, Wt, seeds, V, 1.0)
    assert (plain["tokens"] == filt["tokens"]).all()
    assert np.allclose(plain["qtok"], filt["qtok"], rtol=1e-12)
    assert np.allclose(plain["conf"], filt["conf"], rtol=0, atol=0)
    P = rng.normal(0, 2, size=(B, G + 1, V))
    v_plain = ov.verify(P, L, plain["tokens"], 1, seeds)
    v_filt = ot.verify_filtered(P, L, plain["tokens"], seeds, V, 1.0)
    for key in ("n", "committed", "bonus"):
        assert (v_plain[key] == v_filt[key]).all(), key


def test_filtering_changes_the_draws():
    rng = np.random.default_rng(3)
    L = rng.normal(0, 1, size=(4, 3, 500))
    anchor = rng.integers(0, 500, size=4)
    seeds = np.arange(4, dtype=np.uint64)
    k, top_p, _ = _setting()
    f = ot.draft_block_filtered(L, anchor, None, None, seeds, k, top_p)
    # every filtered draw is among its row's top k
    for b in range(4):
        for j in range(3):
            top = np.argsort(-L[b, j], kind="stable")[:k]
            assert f["tokens"][b, j] in top
    plain = od.draft_block(L, anchor, None, None, 1, seeds)
    assert (plain["tokens"] != f["tokens"]).any()


def test_committed_token_follows_the_filtered_target():
    """gamma = 1: the committed token (accepted draft or residual draw) is distributed
    as the filtered p_1, whatever the filtered q_1 the draft was drawn from."""
    rng = np.random.default_rng(17)
    V, k, top_p = 8, 5, 0.9
    P = rng.normal(0, 1.2, size=(1, 2, V))
    Q = P[:, :1] + rng.normal(0, 0.8, size=(1, 1, V))
    pf, _ = ot.filtered(P[0, 0], k, top_p)
    qf, _ = ot.filtered(Q[0, 0], k, top_p)
    n_trials = 20000
    counts = np.zeros(V)
    for s in range(n_trials):
        x, _ = ot.inverse_cdf(qf, philox.uniform(s + 1000, 0, 1, philox.STREAM_DRAFT))
        r = ot.verify_request_filtered(P[0], Q[0], [x], s, 0, k, top_p)
        counts[r["committed"][0]] += 1
    sd = np.sqrt(n_trials * pf * (1 - pf))
    assert (np.abs(counts - n_trials * pf) <= 4 * sd + 1e-9).all(), (counts / n_trials, pf)
    assert counts[pf == 0].sum() == 0
