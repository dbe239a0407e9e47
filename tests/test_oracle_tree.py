"""Pins of the draft-tree oracle (oracle/tree.py), on the CPU.

The T=0 tree walk is tied to the block verification it generalises (a chain is a block)
and to brute force over every root-to-node path; the selection is tied to its defining
properties (the m largest path products, prefix-closed)."""

import numpy as np
import pytest

from oracle import tree as otr
from oracle import verify as ov


def _random_tree(rng, n, V):
    """Topologically ordered tree with distinct tokens among siblings."""
    parent = np.empty(n, dtype=np.int64)
    token = np.empty(n, dtype=np.int64)
    used = {}
    for i in range(n):
        par = int(rng.integers(-1, i)) if i > 0 else -1
        free = [v for v in range(V) if v not in used.get(par, set())]
        if not free:
            par = -1 if i == 0 else i - 1
            free = [v for v in range(V) if v not in used.get(par, set())]
        t = int(rng.choice(free))
        used.setdefault(par, set()).add(t)
        parent[i], token[i] = par, t
    return parent, token


def test_chain_is_block_verification():
    rng = np.random.default_rng(0)
    for trial in range(20):
        G, V = int(rng.integers(1, 6)), int(rng.integers(2, 6))
        target = rng.normal(0, 1, size=(G + 1, V))
        am = target.argmax(-1)
        x = am[:G].copy()
        k = int(rng.integers(0, G + 1))
        if k < G:
            x[k] = (x[k] + 1) % V
        parent = np.arange(-1, G - 1)
        r = otr.verify_t0(parent, x, target)
        ref = ov.verify_request(target, None, x, 0, 0, 0)
        assert r["n"] == ref["n"]
        assert r["committed"] == ref["committed"][:ref["n"] + 1].tolist()
        assert r["bonus"] == ref["bonus"]


def _brute_force(parent, token, rows):
    """The longest root-to-node path along which every node's token is the argmax of
    its parent's row (unique when siblings hold distinct tokens)."""
    n = len(parent)
    best = []
    for end in range(-1, n):
        path = []
        cur = end
        while cur >= 0:
            path.append(cur)
            cur = int(parent[cur])
        path.reverse()
        ok = all(int(token[c]) == int(np.argmax(rows[0] if parent[c] < 0 else rows[1 + parent[c]])) for c in path)
        if ok and len(path) > len(best):
            best = path
    return best


@pytest.mark.parametrize("seed", range(15))
def test_walk_is_the_longest_matching_path(seed):
    rng = np.random.default_rng(seed)
    n, V = int(rng.integers(1, 13)), 3
    parent, token = _random_tree(rng, n, V)
    rows = rng.normal(0, 1, size=(1 + n, V))
    # make matches likely: rows favour their children's tokens
    for i in range(-1, n):
        kids = [c for c in range(n) if parent[c] == i]
        if kids and rng.random() < 0.8:
            rows[0 if i < 0 else 1 + i, token[kids[int(rng.integers(0, len(kids)))]]] += 5.0
    r = otr.verify_t0(parent, token, rows)
    best = _brute_force(parent, token, rows)
    assert r["path"] == best
    last = rows[0] if not best else rows[1 + best[-1]]
    assert r["committed"] == [int(token[c]) for c in best] + [int(np.argmax(last))]


@pytest.mark.parametrize("seed", range(10))
def test_selection_is_prefix_closed_and_keeps_the_largest(seed):
    rng = np.random.default_rng(100 + seed)
    n = int(rng.integers(1, 30))
    parent, _ = _random_tree(rng, n, 50)
    conf = rng.uniform(0.0, 1.0, size=n)
    conf[rng.random(n) < 0.1] = 1.0     # ties between parent and child
    s = otr.scores(parent, conf)
    for i in range(n):
        if parent[i] >= 0:
            assert s[i] <= s[parent[i]]
    for m in range(0, n + 1):
        sel = set(otr.select(parent, conf, m).tolist())
        assert len(sel) == m
        for i in sel:
            assert parent[i] < 0 or int(parent[i]) in sel
        if 0 < m < n:
            assert min(s[list(sel)]) >= max(s[[i for i in range(n) if i not in sel]])


def test_pruned_walk_and_degenerate_trees():
    rows = np.array([[0.0, 3.0, 1.0], [5.0, 0.0, 0.0], [0.0, 0.0, 4.0]])
    parent = np.array([-1, 0])
    token = np.array([1, 0])
    assert otr.verify_t0(parent, token, rows)["committed"] == [1, 0, 2]
    assert otr.verify_t0(parent, token, rows, keep=[0])["committed"] == [1, 0]   # node 1 pruned
    empty = otr.verify_t0(np.array([], dtype=np.int64), np.array([], dtype=np.int64), rows[:1])
    assert empty["n"] == 0 and empty["committed"] == [1]
    bad = rows.copy()
    bad[1, 2] = np.nan
    assert otr.verify_t0(parent, token, bad)["n"] == -1


def test_scores_are_path_products():
    """Each score is the product of the confidences from the root to the node, found
    here by walking up the parent map (independent of the oracle's forward recurrence,
    up to the order of the float64 products)."""
    rng = np.random.default_rng(7)
    parent, _ = _random_tree(rng, 40, 100)
    conf = rng.uniform(0, 1, size=40)
    conf[3] = np.nan     # read as 0: it and its subtree score 0
    conf[5] = 1.7        # clamped to 1
    s = otr.scores(parent, conf)
    c = np.clip(np.nan_to_num(conf, nan=0.0), 0, 1)
    for i in range(40):
        prod, cur = 1.0, i
        while cur >= 0:
            prod *= c[cur]
            cur = int(parent[cur])
        assert abs(s[i] - prod) <= 1e-15


def test_parents_out_of_order_make_the_tree_invalid():
    rows = np.zeros((4, 3))
    token = np.array([0, 0, 0])
    for parent in (np.array([-1, 1, 0]), np.array([-1, 0, 5]), np.array([-2, 0, 1]), np.array([0, 0, 1])):
        assert not otr.valid_parents(parent)
        assert np.isnan(otr.scores(parent, [0.5, 0.5, 0.5])).all()
        assert otr.select(parent, [0.5, 0.5, 0.5], 2).size == 0
        assert otr.verify_t0(parent, token, rows)["n"] == -1
    assert otr.valid_parents(np.array([-1, 0, 0, 2, -1]))
