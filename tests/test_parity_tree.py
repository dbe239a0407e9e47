"""spec_tree_select and spec_tree_verify on the GPU against the float64 oracle
(oracle/tree.py).

Selection: the scores are float64 products along each path, taken in the same order
on both sides, so they must be identical bit for bit, and so must the kept set and
the selected indices.  Verification (T=0) is integer work: n, the accepted path, the
committed tokens and the bonus must be identical.
"""

import numpy as np
import pytest
import torch

import verify_spec_draft_gb300 as vsd
from verify_spec_draft_gb300 import synth
from oracle import tree as otr

pytestmark = pytest.mark.gpu


def _oracle_verify(target, parent, token, keep=None):
    """Per tree: (n, path, committed, bonus) of the oracle, padded with -1 as the ABI."""
    T, R, V = target.shape
    n = R - 1
    rows = target.double().cpu().numpy()
    par = parent.cpu().numpy() if n > 0 else np.zeros((T, 0), dtype=np.int64)
    tok = token.cpu().numpy() if n > 0 else np.zeros((T, 0), dtype=np.int64)
    kp = None if keep is None else keep.cpu().numpy()
    res = []
    for t in range(T):
        sel = None if kp is None else np.nonzero(kp[t])[0]
        r = otr.verify_t0(par[t], tok[t], rows[t], keep=sel)
        path = r["path"] + [-1] * (n - len(r["path"]))
        com = r["committed"] + [-1] * (n + 1 - len(r["committed"]))
        res.append((r["n"], path, com, r["bonus"]))
    return res


def _compare_verify(out, ref):
    n = out["n"].cpu().tolist()
    path = out["path"].cpu().tolist()
    com = out["committed"].cpu().tolist()
    bonus = out["bonus"].cpu().tolist()
    for t, (rn, rp, rc, rb) in enumerate(ref):
        assert n[t] == rn, (t, n[t], rn)
        assert path[t] == rp, t
        assert com[t] == rc, t
        assert bonus[t] == rb, t


@pytest.mark.parametrize("T,n,V,dtype,shape", [
    (4, 12, 1000, torch.float32, "bushy"),
    (6, 40, 20001, torch.bfloat16, "bushy"),     # V % 8 != 0: scalar loads, ragged chunk
    (4, 12, 1000, torch.bfloat16, "bushy"),      # rows of 16-byte words but not 32-byte ones
    (3, 30, 9000, torch.float32, "chain"),
    (2, 1024, 64, torch.bfloat16, "bushy"),      # the most nodes per tree
    (5, 1, 8192, torch.bfloat16, "chain"),       # one node, exactly one chunk
])
def test_verify_small(spec, T, n, V, dtype, shape):
    x = synth.tree_inputs(T, n, V, dtype, seed=T * 1000 + n, device="cuda", shape=shape, p_match=0.8)
    out = vsd.tree_verify(x["target"], x["parent"], x["token"])
    torch.cuda.synchronize()
    _compare_verify(out, _oracle_verify(x["target"], x["parent"], x["token"]))
    assert vsd.device_status(out["ws"]) == 0
    assert (out["n"] > 0).any()   # the trees accept something


def test_chain_equals_block_verify(spec):
    """A chain is a block: spec_tree_verify equals spec_verify at T=0."""
    T, G, V = 8, 7, 30000
    x = synth.tree_inputs(T, G, V, torch.bfloat16, seed=5, device="cuda", shape="chain", p_match=0.85)
    tv = vsd.tree_verify(x["target"], x["parent"], x["token"])
    bv = vsd.verify(x["target"], None, x["token"], 0, None)
    torch.cuda.synchronize()
    assert torch.equal(tv["n"], bv["n"])
    assert torch.equal(tv["committed"], bv["committed"])
    assert torch.equal(tv["bonus"], bv["bonus"])


def test_select_matches_oracle(spec):
    T, n = 6, 300
    x = synth.tree_inputs(T, n, 16, torch.float32, seed=9, device="cuda")
    conf = x["conf"].clone()
    conf[0, 5] = float("nan")      # read as 0
    conf[1, 7] = 1.5               # clamped to 1
    conf[2, :40] = 1.0             # ties between parents and children
    conf[3, 10:20] = 0.5           # ties between siblings and cousins
    conf[4, 3] = -0.25             # clamped to 0
    for m in (0, 1, 17, 60, n, n + 5):
        out = vsd.tree_select(x["parent"], conf, m)
        torch.cuda.synchronize()
        par = x["parent"].cpu().numpy()
        cf = conf.cpu().numpy()
        for t in range(T):
            s_ref = otr.scores(par[t], cf[t])
            assert np.array_equal(out["score"][t].cpu().numpy(), s_ref), t   # bit for bit
            sel = otr.select(par[t], cf[t], m)
            keep = np.zeros(n, dtype=np.int32)
            keep[sel] = 1
            assert np.array_equal(out["keep"][t].cpu().numpy(), keep), (t, m)
            if m > 0:
                want = sel.tolist() + [-1] * (m - len(sel))
                assert out["selected"][t].cpu().tolist() == want, (t, m)


def test_select_then_verify_pruned(spec):
    """The EAGLE-2 step: keep the top-m nodes, verify only those (rows of dropped
    nodes are never read: they hold NaN here)."""
    T, n, V, m = 8, 64, 40000, 20
    x = synth.tree_inputs(T, n, V, torch.bfloat16, seed=21, device="cuda", p_match=0.8)
    sel = vsd.tree_select(x["parent"], x["conf"], m)
    torch.cuda.synchronize()
    target = x["target"].clone()
    dropped = (sel["keep"] == 0).nonzero()
    target[dropped[:, 0], dropped[:, 1] + 1, 3] = float("nan")
    out = vsd.tree_verify(target, x["parent"], x["token"], keep=sel["keep"])
    torch.cuda.synchronize()
    _compare_verify(out, _oracle_verify(x["target"], x["parent"], x["token"], keep=sel["keep"]))
    assert vsd.device_status(out["ws"]) == 0


def test_invalid_trees(spec):
    T, n, V = 5, 10, 3000
    x = synth.tree_inputs(T, n, V, torch.float32, seed=33, device="cuda", shape="chain", p_match=1.0)
    parent, target = x["parent"].clone(), x["target"].clone()
    parent[1, 4] = 4                 # tree 1: a node that is its own parent
    parent[2, 6] = 8                 # tree 2: a parent after its child
    target[3, 3, 11] = float("nan")  # tree 3: the walk reaches node 2's row (all drafts match)
    target[4, 0, :] = float("-inf")  # tree 4: the root row has no finite entry
    out = vsd.tree_verify(target, parent, x["token"])
    torch.cuda.synchronize()
    _compare_verify(out, _oracle_verify(target, parent, x["token"]))
    n_out = out["n"].cpu().tolist()
    assert n_out[0] == n and n_out[1:] == [-1, -1, -1, -1]
    flags = vsd.device_status(out["ws"])
    assert flags & vsd.DEV_TOKEN and flags & vsd.DEV_NONFINITE
    sel = vsd.tree_select(parent, x["conf"], 4)
    torch.cuda.synchronize()
    assert torch.isnan(sel["score"][1]).all() and (sel["keep"][1] == 0).all()
    assert (sel["selected"][2] == -1).all()
    assert (sel["keep"][0].sum() == 4).item()


def test_nan_row_off_the_walk_is_not_read(spec):
    T, n, V = 1, 6, 500
    x = synth.tree_inputs(T, n, V, torch.float32, seed=34, device="cuda", shape="chain", p_match=1.0)
    token = x["token"].clone()
    token[0, 1] = (token[0, 1] + 1) % V    # the walk stops after node 0
    target = x["target"].clone()
    target[0, 4, 0] = float("nan")          # node 3's row, never reached
    out = vsd.tree_verify(target, x["parent"], token)
    torch.cuda.synchronize()
    assert int(out["n"][0]) == 1
    _compare_verify(out, _oracle_verify(target, x["parent"], token))
    assert vsd.device_status(out["ws"]) == 0


def test_empty_trees(spec):
    """No draft nodes: the committed token is the root row's argmax."""
    g = torch.Generator(device="cuda").manual_seed(3)
    target = torch.randn((4, 1, 7000), generator=g, device="cuda").to(torch.bfloat16)
    out = vsd.tree_verify(target, None, None)
    torch.cuda.synchronize()
    assert (out["n"] == 0).all()
    assert torch.equal(out["committed"][:, 0].long(), target.float().argmax(-1)[:, 0])
    assert torch.equal(out["bonus"], out["committed"][:, 0])


def test_workspace_reuse(spec):
    T, n, V = 6, 50, 12000
    x = synth.tree_inputs(T, n, V, torch.bfloat16, seed=40, device="cuda")
    ws = vsd.workspace(vsd.OP_TREE_VERIFY, T, n, V)
    outs = [vsd.tree_verify(x["target"], x["parent"], x["token"], ws=ws) for _ in range(3)]
    torch.cuda.synchronize()
    for o in outs[1:]:
        for k in ("n", "path", "committed", "bonus"):
            assert torch.equal(o[k], outs[0][k])
    _compare_verify(outs[-1], _oracle_verify(x["target"], x["parent"], x["token"]))


def test_full_size(spec):
    """32 trees x 64 nodes over V = 248,320 bf16 rows (2080 rows, 1.03 GB), as the
    benchmark times it: every tree against the oracle, then the top-24 selection and
    the pruned verification."""
    c = synth.TREE_CONFIG
    x = synth.tree_inputs(c.B, c.gamma, c.V, c.dtype, seed=c.seed, device="cuda", p_match=0.75)
    out = vsd.tree_verify(x["target"], x["parent"], x["token"])
    torch.cuda.synchronize()
    _compare_verify(out, _oracle_verify(x["target"], x["parent"], x["token"]))
    assert vsd.device_status(out["ws"]) == 0
    sel = vsd.tree_select(x["parent"], x["conf"], 24)
    out2 = vsd.tree_verify(x["target"], x["parent"], x["token"], keep=sel["keep"])
    torch.cuda.synchronize()
    _compare_verify(out2, _oracle_verify(x["target"], x["parent"], x["token"], keep=sel["keep"]))
