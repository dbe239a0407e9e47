"""SpecOPD anchor-branch plan (oracle side): anchors on each reference response and
the tree-packing metadata of the branches drafted from them.

Test infrastructure only (see ``oracle/__init__.py``).

Source: "SpecOPD" paper summary (onedev.kr), section "how it works": the reference
response is a shared trunk; B anchors are picked at random on it, and from each the
current drafter samples a branch of W tokens, the branches independent of one another
with causal order kept inside each.  Section "how it differs": the branches are packed
into one proposal tree; the trunk is prefilled once and every branch node sees only
its own reference prefix and its own sampled history, through a parent map and its
semantic position (an ancestors-and-self mask for full attention; rotary position from
the semantic position, not the packing order).

The pages give no formula; the readings taken here:

  Anchors of reference r (length L_r): n distinct positions of 0..L_r-1, uniformly at
  random.  Position i gets the key k_i = word0 >> 40 of Philox4x64-10 with
  key (seed, 0) and counter (r, i, 4, 0) (stream 4 = anchor choice, next to the
  draft's 0..3); the n positions with the smallest (k_i, i) are the anchors, listed in
  ascending position.  (Sorting independent keys and keeping a prefix gives every
  n-subset the same probability.)  A reference shorter than n gets no anchors (-1).
  The anchor token (x_0 of the branch's draft block) is the trunk token at the anchor.
  Packing of reference r: trunk tokens are nodes 0..L_r-1 (node i's parent is i-1,
  its position i); branch k (k-th anchor a_k), step t = 1..W, is node
  L_r + k*W + t-1 with parent a_k for t = 1 and the node before otherwise, and
  semantic position a_k + t.  Only the branch nodes' metadata is returned; the trunk's
  is implicit.

Pins (``tests/test_oracle_anchors.py``): every 2-subset of 6 positions is drawn equally
often over many seeds (chi-square), each position with probability n/L; counts,
distinctness and order; the semantic position of every node equals its depth found by
walking the parent map, and its ancestors are exactly its reference prefix and its own
branch's earlier steps; parents precede children in packing order.
"""

import numpy as np

from . import philox

STREAM_ANCHOR = 4


def anchor_keys(seed, ref, L):
    """The 24-bit key of each position 0..L-1 of reference ``ref``."""
    return np.array([philox.philox4x64_10((ref, i, STREAM_ANCHOR, 0), (seed, 0))[0] >> 40 for i in range(L)],
                    dtype=np.int64)


def choose_anchors(seed, ref, L, n):
    """The n positions with the smallest (key, position), ascending; None if L < n."""
    if L < n:
        return None
    keys = anchor_keys(seed, ref, L)
    order = np.lexsort((np.arange(L), keys))   # by key, then by position
    return np.sort(order[:n])


def branch_tree(anchors, L, W):
    """parent and semantic position of every branch node, [n*W] each (node ids as in
    the packing described above)."""
    n = len(anchors)
    parent = np.empty(n * W, dtype=np.int64)
    position = np.empty(n * W, dtype=np.int64)
    for k in range(n):
        a = int(anchors[k])
        for t in range(1, W + 1):
            node = L + k * W + (t - 1)
            parent[k * W + t - 1] = a if t == 1 else node - 1
            position[k * W + t - 1] = a + t
    return parent, position


def plan(trunk, lengths, n, W, seed):
    """The plan of every reference.

    trunk [R, Lmax] token ids; lengths [R].  Returns dict of int64 arrays:
    anchors [R, n], anchor_tok [R, n], parent [R, n*W], position [R, n*W]; all -1 for a
    reference with fewer than n positions (or more than Lmax)."""
    trunk = np.asarray(trunk)
    R, Lmax = trunk.shape
    out = dict(anchors=np.full((R, n), -1, np.int64), anchor_tok=np.full((R, n), -1, np.int64),
               parent=np.full((R, n * W), -1, np.int64), position=np.full((R, n * W), -1, np.int64))
    for r in range(R):
        L = int(lengths[r])
        if L > Lmax:
            continue
        a = choose_anchors(seed, r, L, n)
        if a is None:
            continue
        out["anchors"][r] = a
        out["anchor_tok"][r] = trunk[r, a]
        out["parent"][r], out["position"][r] = branch_tree(a, L, W)
    return out
