"""Pins of the verify-budget scheduler oracle (oracle/schedule.py), on the CPU.

The expected committed tokens are recomputed here from the distribution of the number
of accepted drafts n (P(n) = (prod_{i<=n} c_i) (1 - c_{n+1}), P(g) = prod_{i<=g} c_i),
not from the oracle's running sum of cumulative products, and every prefix-closed
allocation is enumerated on small batches.
"""

import itertools
import os

import numpy as np
import pytest

from oracle import schedule as osch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def committed_by_distribution(c_row, g):
    """E[n + 1] for one request verifying its first g positions."""
    c = [0.0 if np.isnan(x) else min(1.0, max(0.0, float(x))) for x in c_row[:g]]
    e = 0.0
    run = 1.0
    for n in range(g + 1):
        p_n = run * (1.0 - c[n]) if n < g else run
        e += (n + 1) * p_n
        if n < g:
            run *= c[n]
    return e


def brute_force(conf, K, cost=None):
    """Best objective over all allocations (g_b in 0..gamma) with sum g_b <= K (== K
    without a cost curve)."""
    B, G = conf.shape
    best = -np.inf
    for alloc in itertools.product(range(G + 1), repeat=B):
        k = sum(alloc)
        if k > K or (cost is None and k != K):
            continue
        E = sum(committed_by_distribution(conf[b], alloc[b]) for b in range(B))
        if cost is None:
            val = E
        else:
            if not (np.isfinite(cost[k]) and cost[k] > 0):
                continue
            val = E / cost[k]
        best = max(best, val)
    return best


def alloc_value(conf, gamma, cost):
    B = conf.shape[0]
    E = sum(committed_by_distribution(conf[b], int(gamma[b])) for b in range(B))
    k = int(np.sum(gamma))
    return E if cost is None else E / cost[k]


@pytest.mark.parametrize("seed", range(12))
def test_brute_force_small_batches(seed):
    rng = np.random.default_rng(seed)
    B = int(rng.integers(1, 4))
    G = int(rng.integers(1, 4))
    conf = rng.uniform(0.0, 1.0, size=(B, G))
    K = int(rng.integers(0, B * G + 1))
    # without a cost curve: exactly K positions, the largest expected length
    r = osch.schedule(conf, K)
    assert int(r["gamma"].sum()) == K and r["k"] == K
    assert abs(alloc_value(conf, r["gamma"], None) - brute_force(conf, K)) <= 1e-12
    assert abs(r["expected"] - alloc_value(conf, r["gamma"], None)) <= 1e-12
    # with a cost curve: the best throughput over all allocations of at most K
    cost = np.cumsum(rng.uniform(0.1, 1.0, size=K + 1)) + rng.uniform(0.0, 3.0)
    r = osch.schedule(conf, K, cost)
    assert abs(alloc_value(conf, r["gamma"], cost) - brute_force(conf, K, cost)) <= 1e-12
    assert int(r["gamma"].sum()) == r["k"] <= K


def test_prefix_closed_and_order():
    rng = np.random.default_rng(5)
    conf = rng.uniform(0.2, 1.0, size=(6, 9))
    conf[2, 3] = 1.0   # ties inside a request keep position order
    P = osch.pass_products(conf)
    order = osch.candidate_order(P)
    flat = P.reshape(-1)[order]
    assert (np.diff(flat) <= 0).all()
    for K in range(0, 55, 7):
        g = osch.schedule(conf, K)["gamma"]
        chosen = set(order[:K].tolist())
        for b in range(6):   # request b's chosen positions are exactly its first g[b]
            assert {i - 9 * b for i in chosen if i // 9 == b} == set(range(g[b]))


def test_pages_compounding_example():
    """10 % high at every position makes the product about 95 % high at gamma = 7
    (tests/golden/calibration_compounding.txt)."""
    vals = {}
    for line in open(os.path.join(GOLDEN, "calibration_compounding.txt")):
        if "=" in line and not line.startswith("#"):
            k, v = line.strip().split("=")
            vals[k] = float(v)
    G = int(vals["gamma"])
    over = vals["per_position_overestimate"]
    rng = np.random.default_rng(3)
    c = rng.uniform(0.3, 0.8, size=(4, G))   # stays below 1 after the overestimate
    ratio = osch.pass_products(c * (1.0 + over))[:, G - 1] / osch.pass_products(c)[:, G - 1]
    assert np.allclose(ratio, (1.0 + over) ** G, rtol=1e-12)
    assert round((ratio[0] - 1.0) * 100) == vals["printed_total_overestimate_pct"]


@pytest.mark.parametrize("a,B,K,k_star", [(10.0, 4, 12, 12), (2.0, 4, 12, 0), (4.0, 4, 12, 0)])
def test_certain_passes_closed_form(a, B, K, k_star):
    """All c = 1: E(k) = B + k; with t(k) = a + k the ratio rises with k when a > B,
    falls when a < B, and is flat when a = B (the smallest k is kept)."""
    conf = np.ones((B, 3))
    r = osch.schedule(conf, K, a + np.arange(K + 1, dtype=np.float64))
    assert r["k"] == k_star
    assert r["expected"] == B + k_star


def test_one_request_and_clamping():
    conf = np.array([[0.9, np.nan, 1.7, 0.5]])
    P = osch.pass_products(conf)
    assert P.tolist() == [[0.9, 0.0, 0.0, 0.0]]   # NaN reads as 0, 1.7 as 1
    r = osch.schedule(conf, 4)
    assert r["gamma"].tolist() == [4] and abs(r["expected"] - 1.9) < 1e-15
    # a strictly rising cost stops before the positions that cannot pass
    r = osch.schedule(conf, 4, np.array([1.0, 1.1, 1.2, 1.3, 1.4]))
    assert r["k"] == 1 and r["gamma"].tolist() == [1]


def test_unusable_cost_entries():
    conf = np.full((2, 2), 0.8)
    cost = np.array([np.nan, -1.0, 0.0, 5.0, 6.0])
    r = osch.schedule(conf, 4, cost)
    assert r["k"] == 3   # (2 + 0.8 + 0.8 + 0.64) / 5 > (2 + 2.88) / 6
