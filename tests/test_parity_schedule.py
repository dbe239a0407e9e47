"""spec_verify_budget on the GPU against the oracle (oracle/schedule.py).

Both sides read the same float32 confidences and costs (the oracle widens them
exactly) and form the pass products in float64 in position order, so the candidate
order is the same.  The positions per request must be identical.  Only where the
oracle's best objective values lie within 1e-12 of each other may the GPU's blocked
prefix sums pick another of them; its allocation must then be the oracle's for that
k.  E(k*) comes back as float32: within 1e-6 relative.
"""

import numpy as np
import pytest
import torch

import verify_spec_draft_gb300 as vsd
from oracle import schedule as osch

pytestmark = pytest.mark.gpu


def _run(conf32, budget, cost32=None):
    dev = torch.device("cuda")
    out = vsd.verify_budget(torch.from_numpy(conf32).to(dev), budget,
                            None if cost32 is None else torch.from_numpy(cost32).to(dev))
    torch.cuda.synchronize()
    return out["gamma"].cpu().numpy().astype(np.int64), float(out["expected"].cpu()[0])


def _check(conf32, budget, cost32=None):
    g, e = _run(conf32, budget, cost32)
    conf64 = conf32.astype(np.float64)
    ref = osch.schedule(conf64, budget, None if cost32 is None else cost32.astype(np.float64))
    k_gpu = int(g.sum())
    if cost32 is not None and k_gpu != ref["k"]:
        obj = ref["objective"]
        best = obj[ref["k"]]
        assert np.isfinite(obj[k_gpu]) and abs(obj[k_gpu] - best) <= 1e-12 * abs(best), (k_gpu, ref["k"])
        ref = osch.schedule(conf64, k_gpu)
    assert (g == ref["gamma"]).all()
    assert abs(e - ref["expected"]) <= 1e-6 * ref["expected"]
    return g


def _conf(rng, B, G, lo=0.05, hi=1.0):
    return rng.uniform(lo, hi, size=(B, G)).astype(np.float32)


@pytest.mark.parametrize("B,G", [(1, 1), (1, 15), (4, 7), (32, 7), (32, 16), (100, 40), (128, 64), (8192, 1)])
def test_random_batches(spec, B, G):
    rng = np.random.default_rng(B * 131 + G)
    conf = _conf(rng, B, G)
    N = B * G
    for budget in sorted({0, 1, N // 3, N // 2, N}):
        _check(conf, budget)
        cost = (rng.uniform(2.0, 6.0) + np.arange(budget + 1) * rng.uniform(0.05, 0.5)
                + rng.uniform(0.0, 0.05, size=budget + 1)).astype(np.float32)
        _check(conf, budget, cost)


def test_ties_and_certain_passes(spec):
    """Equal confidences make many equal products: the index order decides."""
    conf = np.full((16, 8), 0.5, dtype=np.float32)
    for budget in (0, 5, 17, 64, 128):
        g = _check(conf, budget)
        assert g.sum() == budget
    ones = np.ones((6, 5), dtype=np.float32)
    g = _check(ones, 13)
    assert g.tolist() == [5, 5, 3, 0, 0, 0]   # all P = 1: flat index order


def test_invalid_confidences_and_costs(spec):
    rng = np.random.default_rng(7)
    conf = _conf(rng, 8, 6)
    conf[1, 2] = np.nan
    conf[3, 0] = -0.5
    conf[4, 4] = 3.0
    conf[5, 1] = -0.0   # the same as +0
    _check(conf, 30)
    cost = np.linspace(3.0, 9.0, 31).astype(np.float32)
    cost[[0, 5, 11]] = [np.nan, -1.0, 0.0]
    cost[20] = np.inf
    _check(conf, 30, cost)
    # no usable entry: nothing verified
    g, e = _run(conf, 4, np.array([np.nan, 0.0, -1.0, np.nan, 0.0], dtype=np.float32))
    assert g.sum() == 0 and e == 8.0


def test_largest_batch_with_curve(spec):
    rng = np.random.default_rng(11)
    conf = _conf(rng, 128, 64, 0.5, 1.0)
    budget = 128 * 64
    cost = (20.0 + 0.01 * np.arange(budget + 1)).astype(np.float32)
    _check(conf, budget, cost)
