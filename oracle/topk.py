"""Top-k / top-p filtered sampling at T=1 (oracle side, float64): the sampling setting of
the DSpine card applied to the draft's draws and to the target's verification.

Test infrastructure only (see ``oracle/__init__.py``).

Source: "DSpine card numbers and public file headers" (aiwithghost.com), section "How
much does the gain shrink when the temperature is raised?": the card's general benchmark
table reports greedy decoding (T=0) beside sampling at T=1 with top_p 0.95 and top_k 20
(``tests/golden/dspine_sampling_setting.txt``).

The page names only the setting; the readings taken here:

  filtered(z; k, top_p): p = softmax(z) at T=1.  The top-k set holds the k entries of
  largest z, ties at the boundary going to the lowest index (as for an argmax).  Those
  entries, in order of z descending (ties: lowest index first), are renormalised over
  the set; the kept set is the shortest prefix of that order whose running sum reaches
  top_p, and holds at least one entry.  The filtered distribution is p on the kept set,
  renormalised to sum 1, and 0 elsewhere.  k >= V with top_p >= 1 leaves p unchanged.

  A draw from a filtered row is the inverse CDF in vocabulary-index order, as for an
  unfiltered row (``_rows.inverse_cdf``).  The draft chain is the DSpark chain of
  ``draft`` with that draw; its confidence stays c_j = 1/Z of the unfiltered row, and
  q_j(x_j) is the filtered probability.  Verification applies the rejection rule of
  ``verify`` to the filtered target and draft rows: accept iff u q_f(x) < p_f(x); on the
  first rejection draw from max(0, p_f - q_f) (from p_f if that sums to 0); if all are
  accepted draw the bonus from the filtered last target row.

Pins (``tests/test_oracle_topk.py``): a worked example of the two cut-offs, with exact
values; k >= V and top_p = 1 reduce the chain and verification to ``draft`` and
``verify`` at T=1; k = 1 or a tiny top_p is the argmax; boundary ties keep the lowest
index; the kept set is the shortest prefix reaching top_p; the committed token's
distribution equals the filtered target row (Monte Carlo over seeds, 4 sigma).
"""

import numpy as np

from . import draft as _draft
from . import philox
from ._rows import NEAR_TIE, as_f64, row_valid, softmax, inverse_cdf


def filtered(z, k, top_p):
    """Filtered distribution of one row: returns (pf [V], kept indices ascending)."""
    z = as_f64(z)
    V = z.shape[0]
    p, _, _ = softmax(z)
    order = np.lexsort((np.arange(V), -z))   # z descending, then index ascending
    top = order[:min(int(k), V)]
    pt = p[top] / p[top].sum()
    run = 0.0
    n_keep = 0
    for w in pt:
        run += w
        n_keep += 1
        if run >= top_p:
            break
    kept = np.sort(top[:n_keep])
    pf = np.zeros(V)
    pf[kept] = p[kept] / p[kept].sum()
    return pf, kept


def draft_step_filtered(l_row, x_prev, U, Wt, u, k, top_p):
    """One position of the chain with a filtered draw: dict(x, conf, qtok, near, z)."""
    base = _draft.draft_step(l_row, x_prev, U, Wt, 1, u)
    if base["x"] < 0:
        return base
    z = base["z"]
    pf, _ = filtered(z, k, top_p)
    x, near = inverse_cdf(pf, u)
    return dict(x=x, conf=base["conf"], qtok=float(pf[x]), near=bool(near), z=z)


def draft_block_filtered(logits, anchor, U, Wt, seeds, k, top_p, first_b=0):
    """The DSpark chain of every request with filtered draws (T=1).  Same layout and
    outputs as ``draft.draft_block``."""
    L = as_f64(logits)
    B, gamma, V = L.shape
    if U is not None:
        U = as_f64(U)
        Wt = as_f64(Wt)
    tokens = np.full((B, gamma), -1, dtype=np.int64)
    conf = np.full((B, gamma), np.nan)
    qtok = np.full((B, gamma), np.nan)
    near = np.zeros((B, gamma), dtype=bool)
    for b in range(B):
        x_prev = int(anchor[b])
        for j in range(1, gamma + 1):
            u = philox.uniform(int(seeds[b]), first_b + b, j, philox.STREAM_DRAFT)
            st = draft_step_filtered(L[b, j - 1], x_prev, U, Wt, u, k, top_p)
            if st["x"] < 0:
                break
            tokens[b, j - 1] = st["x"]
            conf[b, j - 1] = st["conf"]
            qtok[b, j - 1] = st["qtok"]
            near[b, j - 1] = st["near"]
            x_prev = st["x"]
    return dict(tokens=tokens, conf=conf, qtok=qtok, near=near)


def verify_request_filtered(target, draft, tokens, seed, b, k, top_p):
    """Verify one request at T=1 against filtered rows.  target [gamma+1, V], draft
    [gamma, V], tokens [gamma].  Returns dict(n, committed [gamma+1], bonus, near)."""
    P = as_f64(target)
    Q = as_f64(draft)
    gamma = P.shape[0] - 1
    V = P.shape[1]
    committed = np.full(gamma + 1, -1, dtype=np.int64)
    x = [int(t) for t in tokens]
    if any(not 0 <= t < V for t in x) or not all(row_valid(r) for r in P) or not all(row_valid(r) for r in Q):
        return dict(n=-1, committed=committed, bonus=-1, near=False)
    near = False
    for j in range(1, gamma + 1):
        p, _ = filtered(P[j - 1], k, top_p)
        q, _ = filtered(Q[j - 1], k, top_p)
        xj = x[j - 1]
        u = philox.uniform(seed, b, j, philox.STREAM_ACCEPT)
        if abs(u * q[xj] - p[xj]) < NEAR_TIE * q[xj]:
            near = True
        if u * q[xj] < p[xj]:   # q = 0 accepts iff p > 0
            continue
        resid = np.maximum(0.0, p - q)
        if not resid.sum() > 0:
            resid = p
        y, nr = inverse_cdf(resid, philox.uniform(seed, b, j, philox.STREAM_RESIDUAL))
        n = j - 1
        committed[:n] = x[:n]
        committed[n] = y
        return dict(n=n, committed=committed, bonus=y, near=near or nr)
    p_last, _ = filtered(P[gamma], k, top_p)
    y, nr = inverse_cdf(p_last, philox.uniform(seed, b, gamma + 1, philox.STREAM_BONUS))
    committed[:gamma] = x
    committed[gamma] = y
    return dict(n=gamma, committed=committed, bonus=y, near=near or nr)


def verify_filtered(target, draft, tokens, seeds, k, top_p):
    """Verify a batch at T=1 against filtered rows; same outputs as ``verify.verify``."""
    B = target.shape[0]
    gamma = target.shape[1] - 1
    n = np.zeros(B, dtype=np.int64)
    committed = np.zeros((B, gamma + 1), dtype=np.int64)
    bonus = np.zeros(B, dtype=np.int64)
    near = np.zeros(B, dtype=bool)
    for b in range(B):
        r = verify_request_filtered(target[b], draft[b], tokens[b], int(seeds[b]), b, k, top_p)
        n[b], committed[b], bonus[b], near[b] = r["n"], r["committed"], r["bonus"], r["near"]
    return dict(n=n, committed=committed, bonus=bonus, near=near)
