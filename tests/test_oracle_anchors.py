"""Pins of the anchor-branch plan oracle (oracle/anchors.py), on the CPU.

The anchor choice is tied to what "n anchors at random" means (every n-subset equally
likely, each position with probability n/L), not to the oracle's own key sort; the
packing metadata is tied to the tree it must describe (the depth found by walking the
parent map is the semantic position; the ancestors are the reference prefix and the
branch's own history)."""

import itertools

import numpy as np
import pytest

from oracle import anchors as oa
from oracle import draft as od


def test_every_subset_equally_likely():
    L, n, seeds = 6, 2, 3000
    subsets = {s: 0 for s in itertools.combinations(range(L), n)}
    incl = np.zeros(L)
    for seed in range(seeds):
        a = oa.choose_anchors(seed, 0, L, n)
        subsets[tuple(int(x) for x in a)] += 1
        incl[a] += 1
    counts = np.array(list(subsets.values()), dtype=np.float64)
    expect = seeds / len(subsets)
    chi2 = ((counts - expect) ** 2 / expect).sum()
    assert chi2 < 45.0, chi2   # 14 degrees of freedom: P(chi2 > 45) is about 4e-5
    # each position is an anchor with probability n / L (binomial, 5 sigma)
    p = n / L
    sd = np.sqrt(seeds * p * (1 - p))
    assert (np.abs(incl - seeds * p) < 5 * sd).all(), incl


@pytest.mark.parametrize("L,n", [(1, 1), (5, 5), (40, 7), (300, 64)])
def test_counts_distinct_sorted(L, n):
    for ref in range(3):
        a = oa.choose_anchors(11, ref, L, n)
        assert len(a) == n and len(set(a.tolist())) == n
        assert (np.diff(a) > 0).all() and a[0] >= 0 and a[-1] < L
    if n == L:
        assert oa.choose_anchors(11, 0, L, n).tolist() == list(range(L))
    assert oa.choose_anchors(11, 0, n - 1, n) is None


def test_references_draw_independently():
    a0 = oa.choose_anchors(5, 0, 200, 20)
    a1 = oa.choose_anchors(5, 1, 200, 20)
    b0 = oa.choose_anchors(6, 0, 200, 20)
    assert a0.tolist() != a1.tolist() and a0.tolist() != b0.tolist()


def _walk(parent_of, node):
    """Ancestors of `node` (nearest first) by following the parent map."""
    out = []
    while parent_of(node) >= 0:
        node = parent_of(node)
        out.append(node)
    return out


@pytest.mark.parametrize("L,n,W", [(30, 4, 3), (12, 12, 1), (50, 5, 7)])
def test_tree_depth_and_ancestors(L, n, W):
    a = oa.choose_anchors(3, 0, L, n)
    parent, position = oa.branch_tree(a, L, W)

    def parent_of(node):
        return node - 1 if node < L else int(parent[node - L])

    for k in range(n):
        for t in range(1, W + 1):
            node = L + k * W + t - 1
            anc = _walk(parent_of, node)
            # the depth below the trunk's first token is the semantic position
            assert len(anc) == position[node - L] == a[k] + t
            # ancestors: the branch's earlier steps, then the reference prefix 0..a_k
            own = [L + k * W + s - 1 for s in range(t - 1, 0, -1)]
            assert anc == own + list(range(int(a[k]), -1, -1))
            # parents come before children in packing order
            assert parent_of(node) < node
    # every node id of the packing is used once
    assert sorted(range(L, L + n * W)) == list(range(L, L + n * W))


def test_plan_gathers_anchor_tokens_and_flags_short_references():
    rng = np.random.default_rng(0)
    trunk = rng.integers(0, 1000, size=(3, 40))
    lengths = np.array([40, 6, 25])
    out = oa.plan(trunk, lengths, 8, 2, seed=9)
    for r in (0, 2):
        a = out["anchors"][r]
        assert (out["anchor_tok"][r] == trunk[r, a]).all()
        assert a.max() < lengths[r]
    assert (out["anchors"][1] == -1).all() and (out["parent"][1] == -1).all()


def test_draft_first_b_replays_a_slice():
    """The request index of the Philox counter is the index in the whole batch."""
    rng = np.random.default_rng(4)
    B, G, V = 5, 3, 16
    logits = rng.normal(0, 2, size=(B, G, V))
    anchor = rng.integers(0, V, size=B)
    seeds = np.arange(100, 100 + B, dtype=np.uint64)
    full = od.draft_block(logits, anchor, None, None, 1, seeds)
    part = od.draft_block(logits[2:4], anchor[2:4], None, None, 1, seeds[2:4], first_b=2)
    assert (part["tokens"] == full["tokens"][2:4]).all()
    moved = od.draft_block(logits[2:4], anchor[2:4], None, None, 1, seeds[2:4])
    assert (moved["tokens"] != full["tokens"][2:4]).any()
