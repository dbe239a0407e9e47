"""spec_e2etv on the GPU against the float64 oracle.

Bars: |delta a|, |delta S|, |delta loss| <= 1e-5; gradient relative error
||g_gpu - bf16(g_ref)|| / ||bf16(g_ref)|| <= 1e-3, globally and per row (the GPU
rounds its float32 gradient once to bf16; comparing to the unrounded reference would
charge bf16's own rounding, about 2^-9, to the kernel).
"""

import numpy as np
import pytest
import torch

import verify_spec_draft_gb300 as vsd
from verify_spec_draft_gb300 import synth
from oracle import e2etv as oe

pytestmark = pytest.mark.gpu


def _bf16(x):
    return torch.from_numpy(np.asarray(x, dtype=np.float64)).to(torch.bfloat16).double().numpy()


def _grad_relerr(g_gpu, g_ref):
    ref = _bf16(g_ref)
    num = np.linalg.norm(g_gpu - ref)
    den = np.linalg.norm(ref)
    return num / den if den > 0 else num


def _check_rows(out, t, d, N, Wb, rows_of_branches, total_branches):
    R_total = total_branches * Wb
    a = out["a"].cpu().double().numpy()
    S = out["surv"].cpu().double().numpy()
    for n in rows_of_branches:
        sl = slice(n * Wb, (n + 1) * Wb)
        ref = oe.branch(t[sl].double().cpu().numpy(), d[sl].double().cpu().numpy(), R_total)
        assert np.abs(a[sl] - ref["a"]).max() <= 1e-5, n
        assert np.abs(S[sl] - ref["surv"]).max() <= 1e-5, n
        g = out["grad"][sl].double().cpu().numpy()
        assert _grad_relerr(g, ref["grad"]) <= 1e-3, n
        for i in range(Wb):
            assert _grad_relerr(g[i], ref["grad"][i]) <= 1e-3, (n, i)


@pytest.mark.parametrize("N,Wb,V", [(3, 4, 1000), (2, 7, 999), (5, 1, 64), (1, 64, 300), (4, 7, 33000), (9, 3, 20000)])
def test_small(spec, N, Wb, V):
    t, d = synth.e2etv_rows(N, Wb, V, 1.0, seed=N * 100 + V)
    out = vsd.e2etv(t.cuda(), d.cuda(), N, Wb)
    torch.cuda.synchronize()
    ref = oe.e2etv(t.double().numpy(), d.double().numpy(), N, Wb)
    assert abs(float(out["loss"].item()) - ref["loss"]) <= 1e-5
    _check_rows(out, t, d, N, Wb, range(N), N)
    assert vsd.device_status(out["ws"]) == 0


def test_identical_rows(spec):
    t, _ = synth.e2etv_rows(3, 5, 4096, seed=1)
    out = vsd.e2etv(t.cuda(), t.cuda().clone(), 3, 5)
    torch.cuda.synchronize()
    assert torch.allclose(out["a"].cpu(), torch.ones(15), atol=1e-6)
    assert abs(float(out["loss"].item())) <= 1e-5
    assert out["grad"].float().abs().max().item() == 0.0


def test_invalid_branch(spec):
    N, Wb, V = 4, 3, 2048
    t, d = synth.e2etv_rows(N, Wb, V, seed=2)
    d[4, 100] = float("nan")          # branch 1
    t[9, :] = float("-inf")           # branch 3
    out = vsd.e2etv(t.cuda(), d.cuda(), N, Wb)
    torch.cuda.synchronize()
    a = out["a"].cpu()
    assert torch.isnan(a[3:6]).all() and torch.isnan(a[9:12]).all()
    assert torch.isfinite(a[0:3]).all() and torch.isfinite(a[6:9]).all()
    assert torch.isnan(out["loss"].cpu()).all()
    assert out["grad"][3:6].float().abs().max().item() == 0.0
    assert vsd.device_status(out["ws"]) & vsd.DEV_NONFINITE
    _check_rows(out, t, d, N, Wb, [0, 2], N)


def test_deterministic(spec):
    N, Wb, V = 64, 7, 50000
    t, d = synth.e2etv_rows(N, Wb, V, seed=3, device="cuda")
    ws = vsd.workspace(vsd.OP_E2ETV, N, Wb, V)
    outs = [vsd.e2etv(t, d, N, Wb, ws=ws) for _ in range(3)]
    torch.cuda.synchronize()
    for o in outs[1:]:
        for k in ("a", "surv", "loss", "grad"):
            assert torch.equal(o[k], outs[0][k])


@pytest.mark.slow
def test_config5_full_size(spec):
    """16 x 64 x 7 rows, V = 248320, as timed by the benchmark: a, S and the loss of all
    7168 rows against the oracle (computed on the host in chunks, without the
    gradient); the gradient of sampled branches against the oracle's; gradient rows
    summing to zero."""
    import _oracle_pool
    inp = synth.config_inputs(5, device="cuda")
    c = inp["cfg"]
    N, Wb = c.B, c.gamma
    out = vsd.e2etv(inp["target"], inp["draft"], N, Wb)
    torch.cuda.synchronize()
    t_bits = inp["target"].view(torch.int16).cpu().numpy().view(np.uint16)
    d_bits = inp["draft"].view(torch.int16).cpu().numpy().view(np.uint16)
    ref = _oracle_pool.e2etv_no_grad(t_bits, d_bits, N, Wb)
    del t_bits, d_bits
    a = out["a"].double().cpu().numpy()
    S = out["surv"].double().cpu().numpy()
    assert np.abs(a - ref["a"]).max() <= 1e-5
    assert np.abs(S - ref["surv"]).max() <= 1e-5
    assert abs(float(out["loss"].item()) - ref["loss"]) <= 1e-5
    sample = [0, 1, 137, 511, 512, 777, 1022, 1023]
    _check_rows(out, inp["target"], inp["draft"], N, Wb, sample, N)
    g = out["grad"][: 8 * Wb].double()
    scale = g.abs().sum(dim=1)
    assert (g.sum(dim=1).abs() <= 1e-2 * scale + 1e-30).all()
    assert vsd.device_status(out["ws"]) == 0


def test_shards_match_one_call(spec):
    """spec_e2etv_shard on two halves of a batch (as two ranks would run it) equals one
    spec_e2etv call over the whole batch: the same a, S and gradient, and shares that add
    up to 1 - loss."""
    from verify_spec_draft_gb300 import shard
    N, Wb, V = 6, 4, 5000
    t, d = synth.e2etv_rows(N, Wb, V, 1.0, seed=12, device="cuda")
    whole = vsd.e2etv(t, d, N, Wb)
    shares = 0.0
    for rank in range(2):
        b0, n = shard.shard_range(N, rank, 2)
        rows = slice(b0 * Wb, (b0 + n) * Wb)
        part = vsd.e2etv_shard(t[rows].contiguous(), d[rows].contiguous(), n, Wb, N)
        torch.cuda.synchronize()
        assert torch.allclose(part["a"], whole["a"][rows], atol=1e-6, rtol=0)
        assert torch.allclose(part["surv"], whole["surv"][rows], atol=1e-6, rtol=0)
        g0 = whole["grad"][rows].double()
        assert ((part["grad"].double() - g0).norm() / g0.norm()).item() <= 1e-3
        shares += float(part["msum"].item())
        assert vsd.device_status(part["ws"]) == 0
    assert abs((1.0 - shares) - float(whole["loss"].item())) <= 1e-6


def test_shard_with_an_invalid_branch(spec):
    """A NaN in one branch of a shard makes that shard's share NaN (so the all-reduced
    loss is NaN) and flags NONFINITE; the other branches are unaffected."""
    N, Wb, V = 4, 3, 2048
    t, d = synth.e2etv_rows(N, Wb, V, seed=31)
    d[4, 7] = float("nan")   # branch 1
    out = vsd.e2etv_shard(t.cuda(), d.cuda(), N, Wb, 10)
    torch.cuda.synchronize()
    assert torch.isnan(out["msum"].cpu()).all()
    a = out["a"].cpu()
    assert torch.isnan(a[3:6]).all() and torch.isfinite(a[:3]).all() and torch.isfinite(a[6:]).all()
    assert out["grad"][3:6].float().abs().max().item() == 0.0
    assert vsd.device_status(out["ws"]) & vsd.DEV_NONFINITE
    # the valid branches, normalised by the batch of 10 branches
    _check_rows(out, t, d, N, Wb, [0, 2, 3], 10)
