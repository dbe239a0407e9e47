"""SpecOPD E2E-TV surrogate over anchor branches (oracle side, float64).

Test infrastructure only (see ``oracle/__init__.py``).

Sources:

* "SpecOPD" paper summary (onedev.kr), section "how does it work": B anchors on a
  shared reference; from each anchor the drafter samples a W-token branch; branches
  are independent, positions inside a branch are causal.
* Same summary, section "how to use it": at each position the overlap of the draft
  distribution q and the target distribution p is one minus their total variation;
  the loss maximises the mean, over branches and positions j, of the prefix survival
  probability (the product of the acceptance probabilities of the positions up to j).
  Sampled tokens and the target distribution are held fixed; the draft
  probabilities and the prefix products are differentiated.
* "Speculative Decoding Part 2" (VESSL AI), DSpark section: the pass label is
  alpha = 1 - D_TV.

Notation: rows are branch-major, row n*Wb + i is position i of branch n.  For each
row, p = softmax(target row), q = softmax(draft row) (temperature 1).

  a_{n,i} = sum_v min(p_v, q_v)                       (= 1 - TV(p, q))
  s_{n,i} = sum_{v: q_v < p_v} q_v
  S_{n,j} = prod_{i<=j} a_{n,i}
  M = mean over all (n, j) of S_{n,j},   L = 1 - M   (minimised)
  kappa_{n,i} = dM/da_{n,i} = (1/(N*Wb)) * sum_{j>=i} prod_{k<=j, k!=i} a_{n,k}
  dL/dz_{n,i,v} = -kappa_{n,i} * q_v * (1[q_v < p_v] - s_{n,i})

The last line is the chain rule through q = softmax(z) with the subgradient
d min(p, q)/dq = 1[q < p] (strict); at p = q both conventions give zero gradient.

Pins (``tests/test_oracle_e2etv.py``): a equals 1 - (1/2) sum |p - q|; a = 1 when
p = q; 0 <= a <= 1; S is non-increasing along a branch; central finite differences
of L agree with the analytic gradient; each gradient row sums to zero; the gradient
vanishes when p = q; a per-position calibration error of +10% compounds to 1.1**7
over seven positions (VESSL page, DSpark section: "about 95%").
"""

import numpy as np

from ._rows import as_f64, row_valid, softmax


def overlap(p, q):
    """(a, s) for one position: a = sum min(p, q), s = sum over q < p of q."""
    lt = q < p
    return float(np.minimum(p, q).sum()), float(q[lt].sum())


def survival(a):
    """Prefix survival products S_j = prod_{i<=j} a_i along one branch."""
    return np.cumprod(as_f64(a))


def kappa(a, n_total):
    """dM/da_i for one branch, M = (1/n_total) * sum over the branch's S_j (plus other
    branches, which do not depend on these a's).  kappa_i = P_{i-1} * T_i / n_total with
    P the prefix product before i and T_i = 1 + a_{i+1} * T_{i+1}, T_last = 1, i.e.
    sum_{j>=i} prod_{i<k<=j} a_k; no division by a_i."""
    a = as_f64(a)
    W = a.shape[0]
    prefix = np.ones(W)
    for i in range(1, W):
        prefix[i] = prefix[i - 1] * a[i - 1]
    T = np.ones(W)
    for i in range(W - 2, -1, -1):
        T[i] = 1.0 + a[i + 1] * T[i + 1]
    return prefix * T / n_total


def branch(target_rows, draft_rows, n_total, with_grad=True):
    """E2E-TV quantities for one branch of Wb positions.

    Returns dict(a [Wb], s [Wb], surv [Wb], sum_surv, grad [Wb, V] or None, valid).
    A branch with an invalid row has no distribution: NaN a, s and surv, a zero
    gradient (nothing to descend), and it makes the loss NaN.
    ``n_total`` is N*Wb over the whole batch (the mean's denominator).
    """
    P = as_f64(target_rows)
    Q = as_f64(draft_rows)
    Wb, V = P.shape
    if not all(row_valid(r) for r in P) or not all(row_valid(r) for r in Q):
        nan = np.full(Wb, np.nan)
        return dict(a=nan, s=nan, surv=nan, sum_surv=np.nan,
                    grad=np.zeros((Wb, V)) if with_grad else None, valid=False)
    a = np.zeros(Wb)
    s = np.zeros(Wb)
    ps, qs = [], []
    for i in range(Wb):
        p, _, _ = softmax(P[i])
        q, _, _ = softmax(Q[i])
        a[i], s[i] = overlap(p, q)
        ps.append(p)
        qs.append(q)
    S = survival(a)
    grad = None
    if with_grad:
        k = kappa(a, n_total)
        grad = np.empty((Wb, V))
        for i in range(Wb):
            ind = (qs[i] < ps[i]).astype(np.float64)
            grad[i] = -k[i] * qs[i] * (ind - s[i])
    return dict(a=a, s=s, surv=S, sum_surv=float(S.sum()), grad=grad, valid=True)


def e2etv(target, draft, n_branches, Wb, with_grad=True):
    """Whole batch: target, draft [N*Wb, V] branch-major.

    Returns dict(a [R], surv [R], loss, grad [R, V] or None).
    """
    R = n_branches * Wb
    V = target.shape[1]
    a = np.empty(R)
    S = np.empty(R)
    grad = np.empty((R, V)) if with_grad else None
    total = 0.0
    for n in range(n_branches):
        sl = slice(n * Wb, (n + 1) * Wb)
        r = branch(target[sl], draft[sl], R, with_grad)
        a[sl], S[sl] = r["a"], r["surv"]
        total += r["sum_surv"]
        if with_grad:
            grad[sl] = r["grad"]
    return dict(a=a, surv=S, loss=1.0 - total / R, grad=grad)


def loss_only(target, draft, n_branches, Wb):
    """L = 1 - mean S, used by the finite-difference pin."""
    return e2etv(target, draft, n_branches, Wb, with_grad=False)["loss"]
