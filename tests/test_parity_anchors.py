"""spec_branch_plan and spec_draft_block over many branches, on the GPU, against the
oracle (oracle/anchors.py, oracle/draft.py).

The plan is integer work: anchors, anchor tokens, parents and positions must be
identical.  A draft batch larger than one launch runs as several launches; its tokens
must be the oracle's for the whole batch (the Philox request index is the index in the
batch), bit for bit except at a flagged near-tie, after which that request is not
compared further; confidences agree to 1e-5.
"""

import numpy as np
import pytest
import torch

import verify_spec_draft_gb300 as vsd
from verify_spec_draft_gb300 import synth
from oracle import anchors as oa, draft as od

pytestmark = pytest.mark.gpu


def _plan_check(trunk, lengths, n, W, seed):
    dev = torch.device("cuda")
    out = vsd.branch_plan(trunk.to(dev), lengths.to(dev), n, W, seed)
    torch.cuda.synchronize()
    ref = oa.plan(trunk.numpy(), lengths.numpy(), n, W, seed)
    for k in ("anchors", "anchor_tok", "parent", "position"):
        assert (out[k].cpu().numpy() == ref[k]).all(), k
    return out


@pytest.mark.parametrize("R,Lmax,n,W", [(1, 1, 1, 1), (3, 1000, 1000, 2), (4, 300, 17, 7), (2, 16384, 64, 7),
                                        (5, 777, 64, 64)])
def test_plan_matches_oracle(spec, R, Lmax, n, W):
    g = torch.Generator().manual_seed(R * 7 + n)
    trunk = torch.randint(0, 248320, (R, Lmax), generator=g, dtype=torch.int32)
    lengths = torch.full((R,), Lmax, dtype=torch.int32)
    out = _plan_check(trunk, lengths, n, W, seed=R + Lmax)
    assert vsd.device_status(out["ws"]) == 0


def test_plan_ragged_and_short_references(spec):
    g = torch.Generator().manual_seed(3)
    trunk = torch.randint(0, 1000, (5, 500), generator=g, dtype=torch.int32)
    lengths = torch.tensor([500, 40, 12, 501, 233], dtype=torch.int32)   # 12 < n; 501 > Lmax
    out = _plan_check(trunk, lengths, 16, 3, seed=11)
    a = out["anchors"].cpu()
    assert (a[2] == -1).all() and (a[3] == -1).all()
    assert (a[1] < 40).all() and (a[4] < 233).all()
    assert vsd.device_status(out["ws"]) & vsd.DEV_TOKEN


def _draft_check(out, L, anchor, U, Wt, T, seeds, rows, first=None):
    """Compare the requests `rows` (indices in the batch) with the oracle."""
    tok = out["tokens"].cpu().numpy()
    conf = out["conf"].cpu().numpy()
    Un = None if U is None else U.double().cpu().numpy()
    Wn = None if Wt is None else Wt.double().cpu().numpy()
    compared = 0
    for b in rows:
        ref = od.draft_block(L[b:b + 1].double().cpu().numpy(), anchor[b:b + 1].cpu().numpy(), Un, Wn, T,
                             seeds[b:b + 1].cpu().numpy(), first_b=b)
        for j in range(tok.shape[1]):
            if ref["tokens"][0, j] < 0:   # invalid from here on: -1 and NaN on both sides
                assert tok[b, j] == -1 and np.isnan(conf[b, j]), (b, j)
                compared += 1
                continue
            if tok[b, j] != ref["tokens"][0, j]:
                assert ref["near"][0, j], (b, j, tok[b, j], ref["tokens"][0, j])
                break   # the chain diverges legitimately from here
            assert abs(conf[b, j] - ref["conf"][0, j]) <= 1e-5, (b, j)
            compared += 1
    return compared


@pytest.mark.parametrize("T", [0, 1])
def test_batched_draft_tensor_cores(spec, T):
    """40 requests x 7 = 280 rows: two launches of the tcgen05 kernel (36 + 4 requests)."""
    B, G, V, r = 40, 7, 2000, 64
    L, _ = synth.target_and_draft(B, G - 1, V, "zipf", 0.0, torch.bfloat16, seed=21)
    L = L[:, :G].contiguous()
    U, Wt = synth.markov_weights(V, r, torch.bfloat16, seed=21, scale=0.5)
    anchor = synth.anchors(B, V, seed=21)
    seeds = synth.seeds_for(B, 5)
    dev = torch.device("cuda")
    out = vsd.draft_block(L.to(dev), anchor.to(dev), U.to(dev), Wt.to(dev), T, seeds.to(dev))
    torch.cuda.synchronize()
    assert _draft_check(out, L, anchor, U, Wt, T, seeds, range(B)) >= B * G - 2 * G
    assert 1 <= int(out["passes"].item()) <= G
    assert vsd.device_status(out["ws"]) == 0


def test_batched_draft_cuda_cores(spec):
    """float32 weights, 600 requests x 7 = 4200 rows: two launches of the CUDA-core
    kernel (585 + 15 requests); sampled requests on both sides of the cut."""
    B, G, V, r = 600, 7, 300, 4
    L, _ = synth.target_and_draft(B, G - 1, V, "gaussian", 0.0, torch.float32, seed=22)
    L = L[:, :G].contiguous()
    U, Wt = synth.markov_weights(V, r, torch.float32, seed=22, scale=0.5)
    anchor = synth.anchors(B, V, seed=22)
    seeds = synth.seeds_for(B, 9)
    dev = torch.device("cuda")
    out = vsd.draft_block(L.to(dev), anchor.to(dev), U.to(dev), Wt.to(dev), 1, seeds.to(dev))
    torch.cuda.synchronize()
    rows = [0, 1, 300, 583, 584, 585, 586, 599]
    assert _draft_check(out, L, anchor, U, Wt, 1, seeds, rows) >= len(rows) * G - 2 * G


def test_sampler_full_size_sampled(spec):
    """16 references x 64 anchors, W = 7, V = 248320, r = 256, T = 1, as the benchmark
    times it: the plan in full, sampled branches of the draft against the oracle."""
    c = synth.BRANCH_CONFIG
    x = c.extra
    dev = torch.device("cuda")
    inp = synth.branch_inputs(x["n_refs"], x["n_anchors"], c.gamma, c.V, c.r, x["Lmax"], c.dtype, c.seed, dev)
    plan = _plan_check(inp["trunk"].cpu(), inp["lengths"].cpu(), x["n_anchors"], c.gamma, c.seed)
    anchor = plan["anchor_tok"].reshape(-1)
    out = vsd.draft_block(inp["logits"], anchor, inp["U"], inp["Wt"], 1, inp["seeds"])
    torch.cuda.synchronize()
    assert vsd.device_status(out["ws"]) == 0
    tok = out["tokens"]
    assert bool(((tok >= 0) & (tok < c.V)).all())
    rows = [0, 35, 36, 511, 1000, 1023]   # both sides of a launch boundary
    assert _draft_check(out, inp["logits"], anchor.cpu(), inp["U"], inp["Wt"], 1, inp["seeds"], rows) >= 30


def test_plan_every_position_at_the_largest_reference(spec):
    """n = L = 16384 (SPEC_MAX_TRUNK): every position is an anchor, in order."""
    L = 16384
    trunk = torch.arange(L, dtype=torch.int32).view(1, L) % 1000
    out = _plan_check(trunk, torch.tensor([L], dtype=torch.int32), L, 1, seed=5)
    assert out["anchors"].cpu().view(-1).tolist() == list(range(L))


def test_batched_draft_invalid_requests_across_slices(spec):
    """A NaN row in the first launch's slice and an invalid anchor in the second: those
    requests get -1 from the bad position on, the flags of both launches are kept, and
    every other request matches the oracle."""
    B, G, V, r = 40, 7, 2000, 64
    L, _ = synth.target_and_draft(B, G - 1, V, "zipf", 0.0, torch.bfloat16, seed=23)
    L = L[:, :G].contiguous()
    L[3, 4, 17] = float("nan")
    U, Wt = synth.markov_weights(V, r, torch.bfloat16, seed=23, scale=0.5)
    anchor = synth.anchors(B, V, seed=23)
    anchor[38] = -2
    seeds = synth.seeds_for(B, 2)
    dev = torch.device("cuda")
    for T in (0, 1):
        out = vsd.draft_block(L.to(dev), anchor.to(dev), U.to(dev), Wt.to(dev), T, seeds.to(dev))
        torch.cuda.synchronize()
        tok = out["tokens"].cpu()
        assert tok[3, 4:].tolist() == [-1, -1, -1] and (tok[3, :4] >= 0).all()
        assert (tok[38] == -1).all()
        flags = vsd.device_status(out["ws"])
        assert flags & vsd.DEV_NONFINITE and flags & vsd.DEV_TOKEN
        rows = [0, 3, 35, 36, 38, 39]
        assert _draft_check(out, L, anchor, U, Wt, T, seeds, rows) >= 4 * G - 2 * G


@pytest.mark.parametrize("T", [0, 1])
def test_batched_draft_position_path_two_slices(spec, T):
    """1100 requests x 3 = 3300 rows with bf16 logits and weights, r = 64: the
    position-by-position path in two slices of requests (1024 + 76); sampled requests on
    both sides of the cut against the oracle, and the Philox request index of the second
    slice is the request's index in the whole batch."""
    B, G, V, r = 1100, 3, 1000, 64
    L, _ = synth.target_and_draft(B, G - 1, V, "zipf", 0.0, torch.bfloat16, seed=24)
    L = L[:, :G].contiguous()
    U, Wt = synth.markov_weights(V, r, torch.bfloat16, seed=24, scale=0.5)
    anchor = synth.anchors(B, V, seed=24)
    seeds = synth.seeds_for(B, 9)
    dev = torch.device("cuda")
    out = vsd.draft_block(L.to(dev), anchor.to(dev), U.to(dev), Wt.to(dev), T, seeds.to(dev))
    torch.cuda.synchronize()
    assert vsd.device_status(out["ws"]) == 0
    assert int(out["passes"].item()) == G   # the weights are read once per position
    rows = [0, 127, 128, 511, 1023, 1024, 1025, 1099]
    assert _draft_check(out, L, anchor, U, Wt, T, seeds, rows) >= len(rows) * G - 2 * G


@pytest.mark.parametrize("B,G,V,r,T", [
    (300, 3, 40000, 192, 0),    # r = 192 (three k blocks), a ragged last M tile (300 = 2 x 128 + 44)
    (130, 2, 7000, 128, 1),     # just over 256 rows; an odd count of 128-entry tiles
    (600, 5, 3000, 256, 1),     # five M tiles: both epilogue groups hold several
])
def test_batched_draft_position_path_shapes(spec, B, G, V, r, T):
    """The position-by-position path on other ranks, M tiles and vocabularies."""
    L, _ = synth.target_and_draft(B, G - 1, V, "zipf", 0.0, torch.bfloat16, seed=B + V)
    L = L[:, :G].contiguous()
    U, Wt = synth.markov_weights(V, r, torch.bfloat16, seed=B + V, scale=0.3)
    anchor = synth.anchors(B, V, seed=B + V)
    seeds = synth.seeds_for(B, 3)
    dev = torch.device("cuda")
    out = vsd.draft_block(L.to(dev), anchor.to(dev), U.to(dev), Wt.to(dev), T, seeds.to(dev))
    torch.cuda.synchronize()
    assert vsd.device_status(out["ws"]) == 0
    assert int(out["passes"].item()) == G
    rows = [0, 1, 127, 128, B // 2, B - 2, B - 1]
    assert _draft_check(out, L, anchor, U, Wt, T, seeds, rows) >= len(rows) * G - 2 * G


@pytest.mark.parametrize("T", [0, 1])
def test_batched_draft_position_path_offset_rows(spec, T):
    """Drafter rows that start 16 bytes past a 32-byte boundary (a view into a larger
    buffer), with a vocabulary of whole 32-byte rows: the position path takes its
    16-byte loads there, and the results are the chain's."""
    B, G, V, r = 260, 2, 4096, 64
    L, _ = synth.target_and_draft(B, G - 1, V, "zipf", 0.0, torch.bfloat16, seed=31)
    L = L[:, :G].contiguous()
    U, Wt = synth.markov_weights(V, r, torch.bfloat16, seed=31, scale=0.3)
    anchor = synth.anchors(B, V, seed=31)
    seeds = synth.seeds_for(B, 5)
    dev = torch.device("cuda")
    big = torch.empty(L.numel() + 8, dtype=torch.bfloat16, device=dev)
    Ld = big[8:].view(B, G, V)
    Ld.copy_(L.to(dev))
    assert Ld.data_ptr() % 32 == 16
    out = vsd.draft_block(Ld, anchor.to(dev), U.to(dev), Wt.to(dev), T, seeds.to(dev))
    torch.cuda.synchronize()
    assert vsd.device_status(out["ws"]) == 0
    assert int(out["passes"].item()) == G
    rows = [0, 1, 127, 128, 255, 258, 259]
    assert _draft_check(out, L, anchor, U, Wt, T, seeds, rows) >= len(rows) * G - 2 * G
