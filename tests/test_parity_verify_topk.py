"""spec_verify_topk on the GPU against the float64 oracle (oracle/topk.py).

Both sides take the filtered rows' cut-offs in float64 and draw the same 24-bit
uniforms, so n, the committed tokens and the bonus are identical except for requests
the oracle flags as near-ties (a draw within 1e-6 of its threshold).
"""

import numpy as np
import pytest
import torch

import verify_spec_draft_gb300 as vsd
from verify_spec_draft_gb300 import synth
from oracle import topk as ot

pytestmark = pytest.mark.gpu


def _compare(out, ref, max_near=1):
    n = out["n"].cpu().numpy()
    com = out["committed"].cpu().numpy()
    bonus = out["bonus"].cpu().numpy()
    near = ref["near"]
    same = (n == ref["n"]) & (bonus == ref["bonus"]) & (com == ref["committed"]).all(axis=1)
    assert (same | near).all(), np.nonzero(~(same | near))
    assert near.sum() <= max_near
    return int(same.sum())


def _filtered_tokens(d, k, top_p, seed):
    """Tokens a top-k / top-p drafter draws from its own rows (no Markov bias)."""
    B, G, V = d.shape
    seeds = np.arange(seed, seed + B, dtype=np.uint64)
    anchor = np.zeros(B, dtype=np.int64)
    return ot.draft_block_filtered(d.double().numpy(), anchor, None, None, seeds, k, top_p)["tokens"]


@pytest.mark.parametrize("B,G,V,k,top_p,tdt,ddt,dist", [
    (4, 3, 1000, 20, 0.95, torch.bfloat16, torch.bfloat16, "zipf"),
    (3, 5, 777, 1, 1.0, torch.float32, torch.float32, "gaussian"),     # V not a multiple of 8: scalar loads
    (2, 2, 40, 32, 1.0, torch.float32, torch.float32, "gaussian"),     # the largest k, top_p 1
    (5, 4, 5000, 7, 0.5, torch.bfloat16, torch.float32, "zipf"),
    (3, 3, 20, 32, 0.9, torch.float32, torch.bfloat16, "gaussian"),    # V < k: every entry is a candidate
])
@pytest.mark.parametrize("own_tokens", [True, False])
def test_small(spec, B, G, V, k, top_p, tdt, ddt, dist, own_tokens):
    t, d = synth.target_and_draft(B, G, V, dist, 0.7, torch.float32, seed=V + k)
    t, d = t.to(tdt), d.to(ddt)
    if own_tokens:
        tok = torch.from_numpy(_filtered_tokens(d.float(), k, top_p, 40)).to(torch.int32)
    else:
        tok = synth.draft_tokens(d.float(), 1, seed=V)
    seeds = synth.seeds_for(B, 7)
    dev = torch.device("cuda")
    out = vsd.verify_topk(t.to(dev), d.to(dev), tok.to(dev).contiguous(), k, top_p, seeds.to(dev))
    torch.cuda.synchronize()
    ref = ot.verify_filtered(t.double().numpy(), d.double().numpy(), tok.numpy(), seeds.numpy(), k, top_p)
    _compare(out, ref)
    assert vsd.device_status(out["ws"]) == 0


def test_invalid_requests(spec):
    B, G, V, k, top_p = 4, 3, 600, 20, 0.95
    t, d = synth.target_and_draft(B, G, V, "gaussian", 0.5, torch.float32, seed=5)
    tok = synth.draft_tokens(d, 1, seed=5)
    d[1, 2, 40] = float("nan")        # request 1: a draft row without a distribution
    tok[2, 0] = V + 3                  # request 2: a token outside the vocabulary
    t[3, 1, :] = float("-inf")         # request 3: a target row with no finite entry
    seeds = synth.seeds_for(B, 3)
    dev = torch.device("cuda")
    out = vsd.verify_topk(t.to(dev), d.to(dev), tok.to(dev).contiguous(), k, top_p, seeds.to(dev))
    torch.cuda.synchronize()
    ref = ot.verify_filtered(t.double().numpy(), d.double().numpy(), tok.numpy(), seeds.numpy(), k, top_p)
    _compare(out, ref)
    n = out["n"].cpu().tolist()
    assert n[1] == n[2] == n[3] == -1 and n[0] >= 0
    assert vsd.device_status(out["ws"]) & vsd.DEV_TOKEN


def test_config4_full_size(spec):
    """B=32, gamma=7, V=248320 bf16 rows with the DSpine setting (top_k 20, top_p 0.95),
    draft tokens sampled from the unfiltered draft rows (so some fall outside the
    filtered set and must be rejected): every request against the oracle.  Requests the
    oracle flags as near-ties may differ; they are counted and must stay rare (at most
    B*gamma/64, as in the other full-size T=1 comparisons)."""
    inp = synth.config_inputs(4, device="cuda")
    c = inp["cfg"]
    k, top_p = 20, 0.95
    d = inp["draft"]
    tok = synth.draft_tokens(d, 1, seed=c.seed)
    out = vsd.verify_topk(inp["target"], d, tok, k, top_p, inp["seeds"])
    torch.cuda.synchronize()
    ref = ot.verify_filtered(inp["target"].double().cpu().numpy(), d.double().cpu().numpy(), tok.cpu().numpy(),
                             inp["seeds"].cpu().numpy(), k, top_p)
    B, G = c.B, c.gamma
    same = _compare(out, ref, max_near=B * G // 64)
    assert same >= B - B * G // 64
    assert vsd.device_status(out["ws"]) == 0


def test_workspace_reuse_rows_in_pieces(spec):
    """Rows long enough to be split over several CTAs, whose pieces share a bound through
    the workspace.  A second call with the same workspace, on rows whose logits all lie
    lower, must start from no bound: a bound left from the first call would lie above
    every key of the second and empty its lists.  Both calls against the oracle, and the
    second against a call with a fresh workspace."""
    B, G, V, k, top_p = 4, 3, 200_000, 20, 0.95
    dev = torch.device("cuda")
    seeds = synth.seeds_for(B, 9)
    ws = None
    for shift in (0.0, -5.0):
        t, d = synth.target_and_draft(B, G, V, "zipf", 0.7, torch.float32, seed=321)
        t, d = (t + shift).to(torch.bfloat16), (d + shift).to(torch.bfloat16)
        tok = synth.draft_tokens(d.float(), 1, seed=17)
        args = (t.to(dev), d.to(dev), tok.to(dev).contiguous(), k, top_p, seeds.to(dev))
        out = vsd.verify_topk(*args, ws=ws)
        torch.cuda.synchronize()
        ref = ot.verify_filtered(t.double().numpy(), d.double().numpy(), tok.numpy(), seeds.numpy(), k, top_p)
        _compare(out, ref)
        assert vsd.device_status(out["ws"]) == 0
        if ws is not None:
            fresh = vsd.verify_topk(*args)
            torch.cuda.synchronize()
            for key in ("n", "committed", "bonus"):
                assert torch.equal(out[key], fresh[key])
        ws = out["ws"]
