"""spec_draft_verify (one greedy block step in one call) on the GPU.

The call must give exactly what spec_draft_block followed by spec_verify give, bit for
bit, with its one workspace, on the tensor-core and CUDA-core draft paths.  Its
verification results are also checked against the float64 oracle run on the draft's
own tokens.
"""

import pytest
import torch

import verify_spec_draft_gb300 as vsd
from verify_spec_draft_gb300 import synth
from oracle import verify as ov

pytestmark = pytest.mark.gpu


def _inputs(B, gamma, V, r, dtype, wdtype=None, tdtype=None, seed=0):
    dev = torch.device("cuda")
    t, d = synth.target_and_draft(B, gamma, V, "zipf", 0.6, dtype, seed=seed, device=dev)
    if tdtype is not None:
        t = t.to(tdtype).contiguous()
    wdtype = wdtype or dtype
    U, Wt = (None, None) if r == 0 else synth.markov_weights(V, r, wdtype, seed=seed, device=dev, scale=0.3)
    anchor = synth.anchors(B, V, seed=seed, device=dev)
    return d, t, U, Wt, anchor


def _separate(d, t, U, Wt, anchor):
    dr = vsd.draft_block(d, anchor, U, Wt, 0, None)
    vr = vsd.verify(t, None, dr["tokens"], 0, None)
    torch.cuda.synchronize()
    return dr, vr


def _compare(fused, dr, vr):
    for k in ("tokens", "conf", "qtok", "passes"):
        assert torch.equal(fused[k], dr[k]) or (k in ("conf", "qtok") and torch.equal(
            torch.nan_to_num(fused[k], nan=-7.0), torch.nan_to_num(dr[k], nan=-7.0))), k
    for k in ("n", "committed", "bonus"):
        assert torch.equal(fused[k], vr[k]), k
    assert vsd.device_status(fused["ws"]) == (vsd.device_status(dr["ws"]) | vsd.device_status(vr["ws"]))


CASES = [  # (B, gamma, V, r, dtype, weight dtype, target dtype)
    (1, 15, 4104, 64, torch.bfloat16, None, None),            # tensor cores, ragged last tile
    (2, 7, 30000, 128, torch.bfloat16, None, None),           # tensor cores
    (3, 5, 20000, 256, torch.bfloat16, None, torch.float32),  # tensor cores, float32 target rows
    (20, 7, 2048, 64, torch.bfloat16, None, None),            # tensor cores, two M tiles
    (2, 6, 5000, 16, torch.bfloat16, None, None),             # CUDA cores (r not a multiple of 64)
    (2, 5, 3000, 8, torch.float32, None, None),               # CUDA cores (float32 weights)
    (1, 7, 999, 64, torch.bfloat16, None, None),              # rows not 16-byte aligned
    (1, 7, 200000, 64, torch.float32, torch.bfloat16, None),  # float32 logits, large V
]


@pytest.mark.parametrize("B,gamma,V,r,dtype,wdtype,tdtype", CASES)
def test_fused_equals_separate_calls(spec, B, gamma, V, r, dtype, wdtype, tdtype):
    d, t, U, Wt, anchor = _inputs(B, gamma, V, r, dtype, wdtype, tdtype, seed=B * 7 + V)
    fused = vsd.draft_verify(d, t, anchor, U, Wt)
    torch.cuda.synchronize()
    dr, vr = _separate(d, t, U, Wt, anchor)
    _compare(fused, dr, vr)
    # and the verification half against the oracle, on the draft's tokens
    ref = ov.verify(t.double().cpu().numpy(), None, fused["tokens"].cpu().numpy(), 0, None)
    assert (fused["n"].cpu().numpy() == ref["n"]).all()
    assert (fused["committed"].cpu().numpy() == ref["committed"]).all()
    assert (fused["bonus"].cpu().numpy() == ref["bonus"]).all()


def test_drafts_that_match_the_target_are_all_accepted(spec):
    """Draft rows equal to the target rows and no bias: every draft token is the
    target argmax, so n = gamma and the bonus is the argmax of the last target row."""
    B, gamma, V = 2, 7, 8192
    dev = torch.device("cuda")
    t, _ = synth.target_and_draft(B, gamma, V, "zipf", 0.0, torch.bfloat16, seed=3, device=dev)
    d = t[:, :gamma].contiguous()
    U, Wt = synth.markov_weights(V, 64, torch.bfloat16, seed=3, device=dev)
    U = torch.zeros_like(U)
    anchor = synth.anchors(B, V, seed=3, device=dev)
    out = vsd.draft_verify(d, t, anchor, U, Wt)
    torch.cuda.synchronize()
    assert (out["n"] == gamma).all()
    assert torch.equal(out["bonus"], t[:, gamma].float().argmax(-1).to(torch.int32))


def test_invalid_rows_and_anchor(spec):
    B, gamma, V, r = 3, 5, 4096, 64
    d, t, U, Wt, anchor = _inputs(B, gamma, V, r, torch.bfloat16, seed=11)
    d[1, 2, 17] = float("nan")       # a draft row without a distribution
    t[0, 3, 5] = float("inf")        # a target row without a distribution
    anchor[2] = V + 3                # an anchor outside the vocabulary
    fused = vsd.draft_verify(d, t, anchor, U, Wt)
    torch.cuda.synchronize()
    dr, vr = _separate(d, t, U, Wt, anchor)
    _compare(fused, dr, vr)
    assert (fused["n"].cpu() == -1).all()
    flags = vsd.device_status(fused["ws"])
    assert flags & vsd.DEV_NONFINITE and flags & vsd.DEV_TOKEN


def test_latency_workload_full_size(spec):
    """B=1, gamma=15, V=248,320, r=256 (the bench's headline step)."""
    inp = synth.config_inputs(3, device="cuda")
    d, t, U, Wt, anchor = inp["draft"], inp["target"], inp["U"], inp["Wt"], inp["anchor"]
    ws = vsd.workspace(vsd.OP_DRAFT_VERIFY, 1, 15, 248320, 256)
    outs = [vsd.draft_verify(d, t, anchor, U, Wt, ws=ws) for _ in range(2)]
    torch.cuda.synchronize()
    dr, vr = _separate(d, t, U, Wt, anchor)
    for o in outs:
        _compare(o, dr, vr)
