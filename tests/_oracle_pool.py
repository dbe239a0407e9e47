"""Oracle work spread over host processes, for the full-size parity tests.

The pool is started with the "spawn" method: the tests that use it have already
initialised CUDA, and a process forked after that hangs.  Workers receive raw bf16
words (uint16) and widen them to float64 exactly before calling the oracle.
"""

import multiprocessing as mp
import os
from concurrent.futures import ProcessPoolExecutor

import numpy as np


def bf16_bits_to_f64(u16):
    return (np.asarray(u16, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _e2etv_branches(args):
    t_bits, d_bits, Wb, n_total = args
    from oracle import e2etv as oe
    t = bf16_bits_to_f64(t_bits)
    d = bf16_bits_to_f64(d_bits)
    nb = t.shape[0] // Wb
    a = np.empty(nb * Wb)
    S = np.empty(nb * Wb)
    sums = np.empty(nb)
    for n in range(nb):
        sl = slice(n * Wb, (n + 1) * Wb)
        r = oe.branch(t[sl], d[sl], n_total, with_grad=False)
        a[sl], S[sl], sums[n] = r["a"], r["surv"], r["sum_surv"]
    return a, S, sums


def workers():
    return max(1, min(16, os.cpu_count() or 1))


def e2etv_no_grad(t_bits, d_bits, n_branches, Wb, chunk_branches=16):
    """The oracle's a, S and loss of a whole batch (no gradient), rows as uint16 bf16
    words [N*Wb, V]; branches in chunks over a spawn pool."""
    n_total = n_branches * Wb
    jobs = []
    for b0 in range(0, n_branches, chunk_branches):
        b1 = min(n_branches, b0 + chunk_branches)
        jobs.append((t_bits[b0 * Wb:b1 * Wb], d_bits[b0 * Wb:b1 * Wb], Wb, n_total))
    ctx = mp.get_context("spawn")
    with ProcessPoolExecutor(max_workers=workers(), mp_context=ctx) as ex:
        parts = list(ex.map(_e2etv_branches, jobs))
    a = np.concatenate([p[0] for p in parts])
    S = np.concatenate([p[1] for p in parts])
    total = sum(float(x) for p in parts for x in p[2])   # branch sums in branch order
    return dict(a=a, surv=S, loss=1.0 - total / n_total)
