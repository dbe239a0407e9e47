"""Pins for the oracle's E2E-TV surrogate (no GPU)."""

import os

import numpy as np
import pytest

from oracle import e2etv

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _softmax(z):
    e = np.exp(z - z.max())
    return e / e.sum()


def _rows(rng, n_rows, V, sigma):
    T = rng.normal(0, 3, size=(n_rows, V))
    D = T + rng.normal(0, sigma, size=(n_rows, V))
    return T, D


def test_overlap_is_one_minus_tv():
    rng = np.random.default_rng(0)
    for _ in range(50):
        p = _softmax(rng.normal(0, 2, size=33))
        q = _softmax(rng.normal(0, 2, size=33))
        a, s = e2etv.overlap(p, q)
        assert a == pytest.approx(1.0 - 0.5 * np.abs(p - q).sum(), abs=1e-15)
        assert 0.0 <= a <= 1.0
        assert s <= a + 1e-15


def test_identical_rows_full_overlap_zero_grad():
    rng = np.random.default_rng(1)
    T = rng.normal(0, 3, size=(8, 40))
    r = e2etv.e2etv(T, T.copy(), 2, 4)
    assert np.allclose(r["a"], 1.0, atol=1e-15)
    assert r["loss"] == pytest.approx(0.0, abs=1e-15)
    assert np.abs(r["grad"]).max() == 0.0


def test_survival_non_increasing_and_bounded():
    rng = np.random.default_rng(2)
    T, D = _rows(rng, 7 * 6, 64, 1.0)
    r = e2etv.e2etv(T, D, 6, 7)
    S = r["surv"].reshape(6, 7)
    assert (np.diff(S, axis=1) <= 1e-15).all()
    assert ((S >= 0) & (S <= 1)).all()
    assert r["loss"] == pytest.approx(1.0 - S.mean(), abs=1e-15)


def test_gradient_matches_finite_differences():
    rng = np.random.default_rng(3)
    N, Wb, V = 2, 4, 16
    T, D = _rows(rng, N * Wb, V, 1.0)
    g = e2etv.e2etv(T, D, N, Wb)["grad"]
    h = 1e-6
    num = np.zeros_like(D)
    for i in range(N * Wb):
        for v in range(V):
            Dp = D.copy()
            Dm = D.copy()
            Dp[i, v] += h
            Dm[i, v] -= h
            num[i, v] = (e2etv.loss_only(T, Dp, N, Wb) - e2etv.loss_only(T, Dm, N, Wb)) / (2 * h)
    # skip entries where p and q are within the step of crossing (kinks of min)
    rel = np.linalg.norm(num - g) / np.linalg.norm(g)
    assert rel <= 1e-6


def test_gradient_rows_sum_to_zero():
    rng = np.random.default_rng(4)
    T, D = _rows(rng, 14, 200, 1.0)
    g = e2etv.e2etv(T, D, 2, 7)["grad"]
    scale = np.abs(g).sum(axis=1)
    assert (np.abs(g.sum(axis=1)) <= 1e-14 * np.maximum(scale, 1e-300) + 1e-300).all()


def test_kappa_is_derivative_of_mean_survival():
    rng = np.random.default_rng(5)
    a = rng.uniform(0.2, 1.0, size=7)
    n_total = 21

    def M(av):
        return np.cumprod(av).sum() / n_total

    k = e2etv.kappa(a, n_total)
    h = 1e-7
    for i in range(7):
        ap = a.copy()
        am = a.copy()
        ap[i] += h
        am[i] -= h
        assert k[i] == pytest.approx((M(ap) - M(am)) / (2 * h), rel=1e-7)


def test_calibration_compounding_golden():
    """VESSL page, DSpark section: at gamma = 7, a +10% error per position inflates the
    product-based estimate by about 95%."""
    with open(os.path.join(GOLDEN, "calibration_compounding.txt")) as f:
        fields = dict(line.split("=", 1) for line in f if "=" in line and not line.startswith("#"))
    gamma = int(fields["gamma"])
    per_pos = float(fields["per_position_overestimate"])
    printed_pct = float(fields["printed_total_overestimate_pct"])
    a = np.full(gamma, 0.5)
    ratio = e2etv.survival(a * (1 + per_pos))[-1] / e2etv.survival(a)[-1]
    assert ratio == pytest.approx((1 + per_pos) ** gamma, rel=1e-13)
    assert abs((ratio - 1) * 100 - printed_pct) < 1.0     # the page rounds to "about 95%"


def test_invalid_branch():
    T = np.zeros((4, 5))
    D = np.zeros((4, 5))
    D[2, 1] = np.nan
    r = e2etv.e2etv(T, D, 2, 2)
    assert np.isnan(r["a"][2:]).all() and np.isfinite(r["a"][:2]).all()
    assert np.isnan(r["loss"])
