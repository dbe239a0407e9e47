"""Draft-tree selection and T=0 tree verification (oracle side, float64).

Test infrastructure only (see ``oracle/__init__.py``).

Source: "Speculative Decoding Part 2: the evolution of drafter architectures" (VESSL AI),
EAGLE section: EAGLE-2 does not fix the draft tree's shape.  Each branch is scored by
the product of the confidences from the root to it, an estimate of the probability that
it will be used; because the score multiplies along the path, a parent scores at least
as high as its children, so keeping the few highest-scored nodes keeps their parents
too.  Verification of a tree follows the same longest-matching-prefix rule as a block
("Solar Open2 DSpark" (sionic.ai), sections 1 and 6), along the tree's paths.

The pages give no formula; the readings taken here:

  A tree has nodes 0..n-1 in topological order: parent[i] is -1 (the root, the last
  committed token) or a node before i; token[i] is node i's drafted token and conf[i] its
  confidence (the probability that it passes given that its parent passed).  A tree
  with a parent outside [-1, i) is not a tree in this order: it has no scores (NaN), no
  selection, and its verification is invalid (n = -1).
  score[i] = conf[i] * score[parent[i]], the root's score being 1.
  select(m): the m nodes with the largest scores, ties to the lower index, listed in
  index order.  Scores never grow along a path and a parent has the lower index, so the
  selection holds every selected node's parent (prefix-closed).
  verify T=0: the target row of the root is rows[0] and that of node i is rows[1 + i]
  (the distribution of the position after the node's token).  From the root, move to
  the selected child whose token is the argmax of the current node's row (the lowest
  index of such children; argmax ties to the lowest vocabulary index); stop when there
  is none.  n is the number of nodes passed; the committed tokens are theirs, in path
  order, then the bonus y = argmax of the last node's row.

Pins (``tests/test_oracle_tree.py``): a chain reduces to the block verification of
``verify`` at T=0; the accepted path is the longest one found by enumerating every
root-to-node path; the selection is prefix-closed and keeps the m largest scores; the
scores never grow along a path; the scores are products of the confidences along the
path, found by walking up from each node; parents out of order make the tree invalid.
"""

import numpy as np

from ._rows import as_f64, argmax_lowest, row_valid


def valid_parents(parent):
    """True when every parent[i] is -1 or an earlier node (topological order)."""
    return all(-1 <= int(par) < i for i, par in enumerate(parent))


def scores(parent, conf):
    """Path products score[i] = conf[i] * score[parent[i]] (root 1); NaN for every node
    of a tree whose parents are not in topological order."""
    if not valid_parents(parent):
        return np.full(len(parent), np.nan)
    conf = np.clip(np.nan_to_num(as_f64(conf), nan=0.0), 0.0, 1.0)
    s = np.empty(len(parent))
    for i, par in enumerate(parent):
        s[i] = conf[i] * (1.0 if par < 0 else s[par])
    return s


def select(parent, conf, m):
    """Indices (ascending) of the m nodes with the largest scores, ties to the lower index
    (none for a tree whose parents are not in topological order)."""
    if not valid_parents(parent):
        return np.array([], dtype=np.int64)
    s = scores(parent, conf)
    order = np.lexsort((np.arange(len(s)), -s))
    return np.sort(order[:int(m)])


def verify_t0(parent, token, rows, keep=None):
    """T=0 verification of a tree.  parent, token [n]; rows [1 + n, V] (root first);
    keep: the selected node indices (all nodes by default).  Returns dict(n, path
    [node indices], committed [tokens of the path, then the bonus], bonus); n = -1 and
    empty outputs when a row on the walk has no distribution."""
    rows = as_f64(rows)
    n_nodes = len(parent)
    if not valid_parents(parent):
        return dict(n=-1, path=[], committed=[], bonus=-1)
    keep = set(range(n_nodes)) if keep is None else set(int(i) for i in keep)
    children = {}
    for i in range(n_nodes):
        if i in keep:
            children.setdefault(int(parent[i]), []).append(i)
    cur, path = -1, []
    while True:
        row = rows[0] if cur < 0 else rows[1 + cur]
        if not row_valid(row):
            return dict(n=-1, path=[], committed=[], bonus=-1)
        a = argmax_lowest(row)
        nxt = [c for c in children.get(cur, []) if int(token[c]) == a]
        if not nxt:
            return dict(n=len(path), path=path, committed=[int(token[c]) for c in path] + [a], bonus=a)
        cur = min(nxt)
        path.append(cur)
