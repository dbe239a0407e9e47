"""spec_verify_noalloc: verification for callers that cannot allocate device memory.

Such callers (a plugin inside a host program whose allocator owns the GPU's memory
and lends none out; a server whose caching pool holds nearly all of it) cannot hand
spec_verify a workspace.  spec_verify_noalloc runs the same kernels with their
workspace in a fixed 4 MiB static device array of the library.  These tests call it
through the C ABI and require the very outputs of spec_verify (integers: bit for bit)
on two calls in a row, so that what the first call leaves in the shared array cannot
change the second.  The file is named so that pytest collects it last.
"""

import ctypes

import pytest
import torch

import verify_spec_draft_gb300 as vsd
from verify_spec_draft_gb300 import synth

A = 0x10000   # a 16-byte aligned fake device address, never dereferenced


def _outputs(B, gamma, dev):
    return dict(
        n=torch.full((B,), -7, dtype=torch.int32, device=dev),
        committed=torch.full((B, gamma + 1), -7, dtype=torch.int32, device=dev),
        bonus=torch.full((B,), -7, dtype=torch.int32, device=dev),
        near=torch.full((B,), -7, dtype=torch.int32, device=dev),
    )


def _noalloc(lib, target, draft, tokens, T, seeds, out):
    B, g1, V = target.shape
    p = lambda t: ctypes.c_void_p(0 if t is None else t.data_ptr())
    dt = lambda t: vsd.BF16 if t.dtype == torch.bfloat16 else vsd.F32
    code = lib.spec_verify_noalloc(
        p(target), dt(target), p(draft if T == 1 else None), dt(draft) if T == 1 else vsd.F32, p(tokens),
        B, g1 - 1, V, T, p(seeds if T == 1 else None), p(out["n"]), p(out["committed"]), p(out["bonus"]),
        p(out["near"]), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert code == vsd.OK, vsd.status_string(code)


def _case(kind):
    dev = torch.device("cuda")
    if kind == "latency":          # B=1, gamma=15, V=248,320, bf16, T=0
        inp = synth.config_inputs(3, device=dev)
        T = 0
    elif kind == "throughput":     # B=32, gamma=7, V=248,320, bf16, T=1
        inp = synth.config_inputs(4, device=dev)
        T = 1
    else:                          # ragged: V not a multiple of 8, float32 draft rows
        t, d = synth.target_and_draft(3, 5, 20001, "gaussian", 0.7, torch.float32, seed=77, device=dev)
        inp = dict(target=t, draft=d, seeds=synth.seeds_for(3, 5, dev))
        T = 1 if kind == "ragged_t1" else 0
    tokens = synth.draft_tokens(inp["draft"], T, seed=11)
    return inp["target"], inp["draft"], tokens, T, inp["seeds"]


@pytest.mark.gpu
@pytest.mark.parametrize("kind", ["latency", "throughput", "ragged_t0", "ragged_t1"])
def test_noalloc_matches_spec_verify_twice(spec, kind):
    lib = spec.load()
    target, draft, tokens, T, seeds = _case(kind)
    B, g1, V = target.shape
    ref = vsd.verify(target, draft if T == 1 else None, tokens, T, seeds if T == 1 else None)
    first, second = _outputs(B, g1 - 1, target.device), _outputs(B, g1 - 1, target.device)
    _noalloc(lib, target, draft, tokens, T, seeds, first)
    _noalloc(lib, target, draft, tokens, T, seeds, second)
    torch.cuda.synchronize()
    for out in (first, second):
        for k in ("n", "committed", "bonus", "near"):
            assert torch.equal(out[k], ref[k]), (kind, k)


@pytest.mark.gpu
def test_noalloc_alternating_problems(spec):
    """Calls of different sizes and temperatures back to back on one stream: each one
    clears the scratch it uses, so none sees what the one before left there."""
    lib = spec.load()
    cases = [_case("throughput"), _case("latency"), _case("ragged_t1"), _case("throughput")]
    refs = [vsd.verify(t, d if T == 1 else None, x, T, s if T == 1 else None) for t, d, x, T, s in cases]
    outs = []
    for t, d, x, T, s in cases:
        outs.append(_outputs(t.shape[0], t.shape[1] - 1, t.device))
        _noalloc(lib, t, d, x, T, s, outs[-1])
    torch.cuda.synchronize()
    for ref, out in zip(refs, outs):
        for k in ("n", "committed", "bonus", "near"):
            assert torch.equal(out[k], ref[k]), k


def test_noalloc_rejects_problems_beyond_the_scratch():
    """A problem whose verify workspace exceeds the static array is refused with
    SPEC_ERR_SHAPE before any CUDA call (the addresses here are never touched)."""
    from verify_spec_draft_gb300 import build
    if build.needs_build():
        build.build()
    lib = vsd.load()
    B, gamma, V = 1000, 7, 248320
    assert lib.spec_workspace_bytes(vsd.OP_VERIFY, B, gamma, V, 0) > (4 << 20)
    a = ctypes.c_void_p(A)
    code = lib.spec_verify_noalloc(a, vsd.BF16, a, vsd.BF16, a, B, gamma, V, 1, a, a, a, a, None, None)
    assert code == 2   # SPEC_ERR_SHAPE


@pytest.mark.gpu
def test_noalloc_reports_an_invalid_request(spec):
    """The status word lives in the shared array, so this entry point reports a device
    condition only through the outputs: a request whose draft row holds a NaN comes back
    with n = -1 and bonus -1, the others as spec_verify gives them, and the next call
    (on clean rows) is not affected by what the first left in the array."""
    lib = spec.load()
    dev = torch.device("cuda")
    B, gamma, V = 4, 5, 3000
    t, d = synth.target_and_draft(B, gamma, V, "zipf", 0.7, torch.float32, seed=91, device=dev)
    tokens = synth.draft_tokens(d, 1, seed=91)
    seeds = synth.seeds_for(B, 9, dev)
    bad = d.clone()
    bad[2, 1, 17] = float("nan")          # request 2 has no distribution at position 2
    ref = vsd.verify(t, d, tokens, 1, seeds)
    first, second = _outputs(B, gamma, dev), _outputs(B, gamma, dev)
    _noalloc(lib, t, bad, tokens, 1, seeds, first)
    _noalloc(lib, t, d, tokens, 1, seeds, second)
    torch.cuda.synchronize()
    assert int(first["n"][2]) == -1 and int(first["bonus"][2]) == -1
    assert (first["committed"][2] == -1).all()
    keep = [0, 1, 3]
    for k in ("n", "committed", "bonus", "near"):
        assert torch.equal(first[k][keep], ref[k][keep]), k
        assert torch.equal(second[k], ref[k]), k
