"""spec_draft_block_topk on the GPU against the float64 oracle (oracle/topk.py,
draft_block_filtered).

The chain is compared position by position: tokens must be identical until the first
position the oracle flags as a near-tie (a draw within 1e-6 of a boundary, where float32
may decide the other way; the chain can then legitimately diverge, so the rest of that
request is not compared).  Near-ties are counted and must stay rare.  Where tokens agree,
the confidence (1/Z of the unfiltered row) and q_j(x_j) (the filtered probability) agree
to 1e-5.
"""

import numpy as np
import pytest
import torch

import verify_spec_draft_gb300 as vsd
from verify_spec_draft_gb300 import synth
from oracle import topk as ot

pytestmark = pytest.mark.gpu


def _inputs(B, G, V, r, ldtype, scale, seed, dist="zipf"):
    _, d = synth.target_and_draft(B, G, V, dist, 0.5, torch.float32, seed=seed)
    d = d.to(ldtype)
    U = Wt = None
    if r > 0:
        U, Wt = synth.markov_weights(V, r, torch.bfloat16, seed=seed, scale=scale)
    anchor = synth.anchors(B, V, seed=seed)
    seeds = synth.seeds_for(B, seed)
    return d, U, Wt, anchor, seeds


def _run(d, U, Wt, anchor, seeds, k, top_p):
    dev = torch.device("cuda")
    out = vsd.draft_block_topk(d.to(dev), anchor.to(dev), None if U is None else U.to(dev),
                               None if Wt is None else Wt.to(dev), k, top_p, seeds.to(dev))
    torch.cuda.synchronize()
    return out


def _oracle(d, U, Wt, anchor, seeds, k, top_p):
    return ot.draft_block_filtered(d.double().numpy(), anchor.numpy(), None if U is None else U.double().numpy(),
                                   None if Wt is None else Wt.double().numpy(), seeds.numpy(), k, top_p)


def _compare(out, ref):
    tok = out["tokens"].cpu().numpy()
    conf = out["conf"].cpu().numpy()
    qtok = out["qtok"].cpu().numpy()
    B, G = tok.shape
    near = 0
    compared = 0
    for b in range(B):
        for j in range(G):
            assert tok[b, j] == ref["tokens"][b, j], (b, j, tok[b], ref["tokens"][b])
            if ref["tokens"][b, j] < 0:
                assert np.isnan(conf[b, j])
                continue
            assert abs(conf[b, j] - ref["conf"][b, j]) <= 1e-5, (b, j)
            assert abs(qtok[b, j] - ref["qtok"][b, j]) <= 1e-5, (b, j)
            compared += 1
            if ref["near"][b, j]:   # the chain may diverge from here on
                near += 1
                break
    return near, compared


@pytest.mark.parametrize("B,G,V,r,k,top_p,ldtype,scale", [
    (3, 4, 1000, 16, 20, 0.95, torch.bfloat16, 0.3),
    (2, 5, 5000, 64, 1, 1.0, torch.float32, 0.3),      # k = 1: the argmax
    (4, 3, 300, 0, 32, 0.9, torch.float32, 0.0),       # no bias
    (2, 6, 33000, 256, 20, 0.95, torch.bfloat16, 0.1),  # many tiles, ragged last tile
    (1, 7, 20, 32, 32, 1.0, torch.float32, 0.5),       # V < k: every entry a candidate
    (40, 2, 3000, 32, 20, 0.95, torch.bfloat16, 0.3),  # more than one chunk of 32 requests
    (3, 3, 7001, 48, 7, 0.5, torch.float32, 0.4),      # V % 8 != 0, small top_p
    # tensor-core tiles kernel (r a multiple of 64, rows a multiple of 16 bytes):
    (40, 2, 3000, 64, 20, 0.95, torch.bfloat16, 0.3),  # two chunks of requests
    (70, 2, 2048, 128, 16, 0.9, torch.bfloat16, 0.3),  # three chunks: the U buffers are reused
    (2, 3, 40, 64, 32, 1.0, torch.bfloat16, 0.5),      # one ragged tile, V < k
])
def test_small(spec, B, G, V, r, k, top_p, ldtype, scale):
    d, U, Wt, anchor, seeds = _inputs(B, G, V, r, ldtype, scale, seed=V + k + r)
    out = _run(d, U, Wt, anchor, seeds, k, top_p)
    ref = _oracle(d, U, Wt, anchor, seeds, k, top_p)
    near, compared = _compare(out, ref)
    assert near <= 1 and compared >= B
    assert vsd.device_status(out["ws"]) == 0


def test_the_bias_changes_the_chain(spec):
    """With a strong bias the filtered chain differs from the one drawn without it."""
    B, G, V, r = 4, 6, 4000, 32
    d, U, Wt, anchor, seeds = _inputs(B, G, V, r, torch.bfloat16, 1.0, seed=3)
    with_bias = _run(d, U, Wt, anchor, seeds, 20, 0.95)
    without = _run(d, None, None, anchor, seeds, 20, 0.95)
    assert not torch.equal(with_bias["tokens"], without["tokens"])
    _compare(with_bias, _oracle(d, U, Wt, anchor, seeds, 20, 0.95))


def test_draws_lie_in_the_kept_set(spec):
    """Every drawn token is among the row's top_k largest biased logits."""
    B, G, V, r, k = 8, 4, 2000, 16, 5
    d, U, Wt, anchor, seeds = _inputs(B, G, V, r, torch.float32, 0.5, seed=9, dist="gaussian")
    out = _run(d, U, Wt, anchor, seeds, k, 0.95)
    ref = _oracle(d, U, Wt, anchor, seeds, k, 0.95)
    _compare(out, ref)
    tok = out["tokens"].cpu().numpy()
    assert (tok >= 0).all()
    assert (out["qtok"].cpu().numpy() > 0).all()


def test_invalid_requests(spec):
    B, G, V, r = 4, 4, 1500, 16
    d, U, Wt, anchor, seeds = _inputs(B, G, V, r, torch.float32, 0.3, seed=17)
    anchor[1] = V + 5                 # request 1: anchor out of range
    d[2, 2, 100] = float("nan")       # request 2: no distribution at position 3
    d[3, 0, :] = float("-inf")        # request 3: no finite entry at position 1
    out = _run(d, U, Wt, anchor, seeds, 20, 0.95)
    ref = _oracle(d, U, Wt, anchor, seeds, 20, 0.95)
    _compare(out, ref)
    tok = out["tokens"].cpu().numpy()
    assert (tok[1] == -1).all() and (tok[3] == -1).all()
    assert (tok[2, :2] >= 0).all() and (tok[2, 2:] == -1).all()
    assert (tok[0] >= 0).all()
    flags = vsd.device_status(out["ws"])
    assert flags & vsd.DEV_TOKEN and flags & vsd.DEV_NONFINITE


def test_config4_full_size(spec):
    """B=32, gamma=7, V=248320, rank-256 bf16 weights, the DSpine setting (top_k 20,
    top_p 0.95): every request against the oracle."""
    inp = synth.config_inputs(4, device="cpu")
    c = inp["cfg"]
    out = _run(inp["draft"], inp["U"], inp["Wt"], inp["anchor"], inp["seeds"], 20, 0.95)
    ref = _oracle(inp["draft"], inp["U"], inp["Wt"], inp["anchor"], inp["seeds"], 20, 0.95)
    near, compared = _compare(out, ref)
    assert near <= c.B * c.gamma // 64
    assert compared >= c.B
    assert vsd.device_status(out["ws"]) == 0
