"""Failure detection on the GPU: every device wait is bounded.

A kernel's grid barrier is made to wait on an arrival count that can never reach its
target: the test writes a large value into the barrier counter of a fresh workspace,
so the barrier's condition never holds, whatever the CTAs do.  Each CTA must give up
after the wait limit (one second), set SPEC_DEV_TIMEOUT in the workspace status word
and return, so that the host reads the status and the CUDA context stays usable.
Nothing here faults or traps the GPU; the kernels only spin, bounded, and exit.
"""

import numpy as np
import pytest
import torch

import verify_spec_draft_gb300 as vsd
from verify_spec_draft_gb300 import synth
from oracle import draft as od

pytestmark = pytest.mark.gpu

# Workspace header: a status word and its padding (128 B), 32 last-CTA counters
# (128 B), then 64 barrier slots of 64 words; slot 0's arrival count is at byte 256.
BARRIER0_COUNT = 256
# Half the counter range away from any count a launch reaches: the draft barrier
# (which waits until the count has caught up with its target, compared as a signed
# difference) sees it forever behind, and the verify barrier's arrival count never
# equals the number of CTAs.
POISON = 0x80000000


def _poison(ws):
    ws[BARRIER0_COUNT:BARRIER0_COUNT + 4] = torch.tensor(
        list(POISON.to_bytes(4, "little")), dtype=torch.uint8, device=ws.device)


@pytest.mark.parametrize("r,dtype", [(64, torch.bfloat16), (8, torch.float32)])
def test_draft_barrier_wait_times_out(spec, r, dtype):
    """tcgen05 kernel (bf16, r = 64) and CUDA-core kernel (float32, r = 8)."""
    B, gamma, V = 2, 5, 4104
    L, _ = synth.target_and_draft(B, gamma - 1, V, "gaussian", 0.0, dtype, seed=3, device="cuda")
    L = L[:, :gamma].contiguous()
    U, Wt = synth.markov_weights(V, r, dtype, seed=3, device="cuda", scale=0.3)
    anchor = synth.anchors(B, V, seed=3, device="cuda")
    ws = vsd.workspace(vsd.OP_DRAFT, B, gamma, V, r)
    _poison(ws)
    out = vsd.draft_block(L, anchor, U, Wt, 0, None, ws=ws)
    flags = vsd.device_status(out["ws"])
    assert flags & vsd.DEV_TIMEOUT
    # the context still works: a fresh workspace gives the oracle's tokens
    good = vsd.draft_block(L, anchor, U, Wt, 0, None)
    torch.cuda.synchronize()
    ref = od.draft_block(L.double().cpu().numpy(), anchor.cpu().numpy(), U.double().cpu().numpy(),
                         Wt.double().cpu().numpy(), 0, np.zeros(B, dtype=np.int64))
    assert (good["tokens"].cpu().numpy() == ref["tokens"]).all()
    assert vsd.device_status(good["ws"]) == 0


def test_verify_t1_barrier_wait_times_out(spec):
    B, gamma, V = 3, 4, 20000
    t, d = synth.target_and_draft(B, gamma, V, "gaussian", 0.7, torch.bfloat16, seed=4, device="cuda")
    tok = synth.draft_tokens(d, 1, seed=4)
    seeds = synth.seeds_for(B, 4, "cuda")
    ws = vsd.workspace(vsd.OP_VERIFY, B, gamma, V, 0)
    _poison(ws)
    out = vsd.verify(t, d, tok, 1, seeds, ws=ws)
    assert vsd.device_status(out["ws"]) & vsd.DEV_TIMEOUT
    again = vsd.verify(t, d, tok, 1, seeds)
    ref = vsd.verify(t, d, tok, 1, seeds)
    torch.cuda.synchronize()
    assert torch.equal(again["n"], ref["n"]) and torch.equal(again["committed"], ref["committed"])
    assert vsd.device_status(again["ws"]) == 0
