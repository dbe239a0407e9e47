"""C ABI checks that need no GPU: the library loads, exports every function that
include/spec.h declares, and rejects bad arguments before enqueuing anything.

Every call below carries at least one invalid argument, so it returns before its
first CUDA call; fake device addresses are never dereferenced.
"""

import os
import re

import pytest

import verify_spec_draft_gb300 as vsd
from verify_spec_draft_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "spec.h")

A = 0x10000          # a 16-byte aligned fake device address
MIS = 0x10008        # misaligned


@pytest.fixture(scope="module")
def lib():
    if build.needs_build():
        build.build()
    return vsd.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(spec_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_boundary():
    fns = declared_functions()
    for name in ("spec_draft_block", "spec_verify", "spec_e2etv", "spec_workspace_bytes",
                 "spec_workspace_init", "spec_get_device_status", "spec_status_string"):
        assert name in fns


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    assert set(declared_functions()) >= set(vsd.SIGNATURES)


def test_status_strings(lib):
    for code in range(10):
        s = lib.spec_status_string(code).decode()
        assert s and s != "unknown status"
    assert lib.spec_status_string(99).decode() == "unknown status"


def test_workspace_bytes_ranges(lib):
    wb = lib.spec_workspace_bytes
    assert wb(vsd.OP_VERIFY, 32, 7, 248320, 0) > 0
    assert wb(vsd.OP_DRAFT, 1, 15, 248320, 256) > 0
    assert wb(vsd.OP_E2ETV, 1024, 7, 248320, 0) > 0
    assert wb(vsd.OP_VERIFY, 0, 7, 100, 0) == 0
    assert wb(vsd.OP_VERIFY, 1, 65, 100, 0) == 0
    assert wb(vsd.OP_VERIFY, 1, 7, 0, 0) == 0
    assert wb(vsd.OP_DRAFT, 1, 7, 100, 257) == 0
    assert wb(vsd.OP_DRAFT, (1 << 20) + 1, 1, 100, 8) == 0
    # a batch beyond one launch needs one slice's workspace (4096 rows at most)
    assert wb(vsd.OP_DRAFT, 1024, 7, 248320, 256) == wb(vsd.OP_DRAFT, 4096 // 7, 7, 248320, 256)
    assert wb(vsd.OP_BRANCH_PLAN, 16, 7, 4096, 0) > 0
    assert wb(vsd.OP_E2ETV, 1 << 20, 64, 8, 0) == 0
    assert wb(8, 1, 1, 1, 0) == 0
    # bigger problems never need less workspace
    assert wb(vsd.OP_VERIFY, 64, 7, 248320, 0) >= wb(vsd.OP_VERIFY, 32, 7, 248320, 0)


def _draft(lib, **kw):
    a = dict(logits=A, ldt=vsd.BF16, anchor=A, U=A, Wt=A, wdt=vsd.BF16, r=8, B=2, gamma=3, V=100, T=0,
             seeds=A, tokens=A, conf=A, qtok=0, qlogits=0, passes=0, ws=A, wsb=1 << 30)
    a.update(kw)
    return lib.spec_draft_block(a["logits"], a["ldt"], a["anchor"], a["U"], a["Wt"], a["wdt"], a["r"], a["B"],
                                a["gamma"], a["V"], a["T"], a["seeds"], a["tokens"], a["conf"], a["qtok"],
                                a["qlogits"], a["passes"], a["ws"], a["wsb"], None)


def test_draft_argument_errors(lib):
    assert _draft(lib, logits=0) == 1
    assert _draft(lib, T=2) == 1
    assert _draft(lib, T=1, seeds=0) == 1
    assert _draft(lib, U=0) == 1
    assert _draft(lib, ldt=5) == 3
    assert _draft(lib, wdt=9) == 3
    assert _draft(lib, gamma=0) == 2
    assert _draft(lib, gamma=65) == 2
    assert _draft(lib, r=257) == 2
    assert _draft(lib, B=(1 << 20) + 1, gamma=1) == 2
    assert _draft(lib, V=0) == 2
    assert _draft(lib, logits=MIS) == 4
    assert _draft(lib, Wt=MIS) == 4
    assert _draft(lib, qlogits=MIS) == 4
    assert _draft(lib, ws=0) == 9
    assert _draft(lib, wsb=100) == 9


def _verify(lib, **kw):
    a = dict(target=A, tdt=vsd.BF16, draft=A, ddt=vsd.BF16, tokens=A, B=2, gamma=3, V=100, T=0, seeds=A,
             n=A, com=A, bonus=A, near=0, ws=A, wsb=1 << 30)
    a.update(kw)
    return lib.spec_verify(a["target"], a["tdt"], a["draft"], a["ddt"], a["tokens"], a["B"], a["gamma"], a["V"],
                           a["T"], a["seeds"], a["n"], a["com"], a["bonus"], a["near"], a["ws"], a["wsb"], None)


def test_verify_argument_errors(lib):
    assert _verify(lib, target=0) == 1
    assert _verify(lib, tokens=0) == 1
    assert _verify(lib, n=0) == 1
    assert _verify(lib, T=1, draft=0) == 1
    assert _verify(lib, T=1, seeds=0) == 1
    assert _verify(lib, T=3) == 1
    assert _verify(lib, tdt=2) == 3
    assert _verify(lib, T=1, ddt=2) == 3
    assert _verify(lib, B=0) == 2
    assert _verify(lib, B=65536) == 2
    assert _verify(lib, gamma=65) == 2
    assert _verify(lib, V=(1 << 26) + 1) == 2
    assert _verify(lib, target=MIS) == 4
    assert _verify(lib, T=1, draft=MIS) == 4
    assert _verify(lib, ws=0) == 9
    assert _verify(lib, wsb=10) == 9


def _e2etv(lib, **kw):
    a = dict(target=A, draft=A, N=4, Wb=7, V=64, a=A, s=A, loss=A, grad=A, ws=A, wsb=1 << 30)
    a.update(kw)
    return lib.spec_e2etv(a["target"], a["draft"], a["N"], a["Wb"], a["V"], a["a"], a["s"], a["loss"], a["grad"],
                          a["ws"], a["wsb"], None)


def test_e2etv_argument_errors(lib):
    assert _e2etv(lib, target=0) == 1
    assert _e2etv(lib, grad=0) == 1
    assert _e2etv(lib, loss=0) == 1
    assert _e2etv(lib, N=0) == 2
    assert _e2etv(lib, Wb=65) == 2
    assert _e2etv(lib, V=0) == 2
    assert _e2etv(lib, draft=MIS) == 4
    assert _e2etv(lib, grad=MIS) == 4
    assert _e2etv(lib, ws=0) == 9
    assert _e2etv(lib, wsb=100) == 9


def test_verify_topk_argument_errors(lib):
    def call(target=A, tdt=vsd.BF16, draft=A, ddt=vsd.BF16, tokens=A, B=2, G=3, V=100, k=20, top_p=0.95, seeds=A,
             n=A, com=A, bonus=A, near=0, ws=A, wsb=1 << 30):
        return lib.spec_verify_topk(target, tdt, draft, ddt, tokens, B, G, V, k, top_p, seeds, n, com, bonus, near,
                                    ws, wsb, None)
    assert call(tdt=7) == 3
    assert call(ddt=7) == 3
    assert call(k=0) == 2
    assert call(k=33) == 2                 # more than SPEC_MAX_TOP_K
    assert call(G=65) == 2
    assert call(B=0) == 2
    assert call(top_p=0.0) == 1
    assert call(top_p=1.5) == 1
    assert call(top_p=float("nan")) == 1
    assert call(seeds=0) == 1
    assert call(draft=0) == 1
    assert call(target=MIS) == 4
    assert call(wsb=100) == 9
    assert lib.spec_workspace_bytes(vsd.OP_VERIFY_TOPK, 32, 7, 248320, 0) > 0


def test_e2etv_shard_argument_errors(lib):
    def call(target=A, draft=A, N=2, Wb=3, V=100, total=4, a=A, surv=A, msum=A, grad=A, ws=A, wsb=1 << 30):
        return lib.spec_e2etv_shard(target, draft, N, Wb, V, total, a, surv, msum, grad, ws, wsb, None)
    assert call(msum=0) == 1
    assert call(target=0) == 1
    assert call(total=1) == 2              # fewer branches in the batch than in the shard
    assert call(N=0) == 2
    assert call(Wb=65) == 2
    assert call(grad=MIS) == 4
    assert call(wsb=100) == 9


def test_verify_budget_argument_errors(lib):
    def call(conf=A, B=4, gamma=7, budget=10, cost=A, gamma_out=A, expected=A):
        return lib.spec_verify_budget(conf, B, gamma, budget, cost, gamma_out, expected, None)
    assert call(conf=0) == 1
    assert call(gamma_out=0) == 1
    assert call(B=0) == 2
    assert call(gamma=0) == 2
    assert call(gamma=65) == 2
    assert call(B=8193, gamma=1) == 2      # more than SPEC_MAX_BUDGET_CANDIDATES
    assert call(budget=-1) == 2
    assert call(budget=29) == 2            # more than B * gamma


def test_branch_plan_argument_errors(lib):
    def call(trunk=A, lengths=A, R=4, Lmax=100, n=8, W=7, anchors=A, tok=A, parent=A, pos=A, ws=A, wsb=1 << 20):
        return lib.spec_branch_plan(trunk, lengths, R, Lmax, n, W, 5, anchors, tok, parent, pos, ws, wsb, None)
    assert call(trunk=0) == 1
    assert call(parent=0) == 1
    assert call(R=0) == 2
    assert call(Lmax=16385) == 2           # more than SPEC_MAX_TRUNK
    assert call(n=0) == 2
    assert call(n=101) == 2                # more anchors than positions
    assert call(W=0) == 2
    assert call(W=65) == 2
    assert call(ws=0) == 9
    assert call(wsb=16) == 9


def test_workspace_init_rejects_missing(lib):
    assert lib.spec_workspace_init(None, 1 << 20, None) == 9
    assert lib.spec_workspace_init(A, 16, None) == 9
    assert lib.spec_get_device_status(None, None, None) == 9


def test_binding_refuses_cpu_tensors(lib):
    torch = pytest.importorskip("torch")
    x = torch.zeros((1, 2, 8))
    with pytest.raises(ValueError, match="CUDA tensor"):
        vsd.verify(x, None, torch.zeros((1, 1), dtype=torch.int32))


def test_tree_calls_reject_bad_arguments(lib):
    wb = lib.spec_workspace_bytes
    assert wb(vsd.OP_TREE_VERIFY, 32, 64, 248320, 0) > 0
    assert wb(vsd.OP_TREE_VERIFY, 32, 0, 100, 0) > 0            # trees without draft nodes
    assert wb(vsd.OP_TREE_VERIFY, 32, 1025, 100, 0) == 0
    assert wb(vsd.OP_TREE_VERIFY, 0, 8, 100, 0) == 0
    assert wb(vsd.OP_TREE_VERIFY, 4, 1000, 100, 0) > wb(vsd.OP_TREE_VERIFY, 4, 64, 100, 0)
    a = A
    sel = lib.spec_tree_select
    assert sel(a, a, 4, 0, 2, a, a, a, None) == 2                  # no nodes
    assert sel(a, a, 4, 1025, 2, a, a, a, None) == 2               # too many nodes
    assert sel(a, a, 4, 8, -1, a, a, a, None) == 2                 # m < 0
    assert sel(a, a, 0, 8, 2, a, a, a, None) == 2
    assert sel(None, a, 4, 8, 2, a, a, a, None) == 1
    assert sel(a, a, 4, 8, 2, a, None, a, None) == 1               # keep_out required
    tv = lib.spec_tree_verify
    big = 1 << 30
    assert tv(a, 7, a, a, a, 4, 8, 100, a, a, a, a, a, big, None) == 3        # dtype
    assert tv(a, vsd.BF16, a, a, a, 4, 1025, 100, a, a, a, a, a, big, None) == 2
    assert tv(a, vsd.BF16, a, a, a, 4, 8, 0, a, a, a, a, a, big, None) == 2
    assert tv(a, vsd.BF16, None, a, a, 4, 8, 100, a, a, a, a, a, big, None) == 1   # parent needed (n > 0)
    assert tv(a, vsd.BF16, a, a, a, 4, 8, 100, a, None, a, a, a, big, None) == 1   # path_out needed
    assert tv(MIS, vsd.BF16, a, a, a, 4, 8, 100, a, a, a, a, a, big, None) == 4
    need = wb(vsd.OP_TREE_VERIFY, 4, 8, 100, 0)
    assert tv(a, vsd.BF16, a, a, a, 4, 8, 100, a, a, a, a, a, need - 1, None) == 9
    assert tv(a, vsd.BF16, a, a, a, 4, 8, 100, a, a, a, a, None, big, None) == 9


def test_draft_block_topk_rejects_bad_arguments(lib):
    wb = lib.spec_workspace_bytes
    assert wb(vsd.OP_DRAFT_TOPK, 32, 7, 248320, 256) > 0
    assert wb(vsd.OP_DRAFT_TOPK, 0, 7, 100, 0) == 0
    a, big = A, 1 << 30
    f = lib.spec_draft_block_topk
    args = lambda **kw: dict(dict(l=a, ldt=vsd.BF16, anc=a, U=a, Wt=a, wdt=vsd.BF16, r=16, B=2, G=3, V=100, k=20,
                                  tp=0.95, seeds=a, tok=a, conf=a, q=a, ws=a, wsb=big), **kw)
    call = lambda d: f(d["l"], d["ldt"], d["anc"], d["U"], d["Wt"], d["wdt"], d["r"], d["B"], d["G"], d["V"], d["k"],
                       d["tp"], d["seeds"], d["tok"], d["conf"], d["q"], d["ws"], d["wsb"], None)
    assert call(args(r=24)) == 2                  # r not a multiple of 16
    assert call(args(r=272)) == 2                 # r beyond SPEC_MAX_RANK
    assert call(args(k=0)) == 2 and call(args(k=33)) == 2
    assert call(args(tp=0.0)) == 1 and call(args(tp=1.5)) == 1
    assert call(args(wdt=vsd.F32)) == 3           # weights must be bf16
    assert call(args(seeds=None)) == 1
    assert call(args(l=MIS)) == 4
    assert call(args(wsb=wb(vsd.OP_DRAFT_TOPK, 2, 3, 100, 16) - 1)) == 9
    assert call(args(G=65)) == 2
    assert call(args(V=(1 << 19) + 1)) == 2       # beyond SPEC_MAX_V_DRAFT_TOPK
    assert wb(vsd.OP_DRAFT_TOPK, 2, 3, (1 << 19) + 1, 16) == 0
    # the workspace holds each position's biased logits: about B * V * 4 bytes
    assert wb(vsd.OP_DRAFT_TOPK, 32, 7, 248320, 256) >= 32 * 248320 * 4
