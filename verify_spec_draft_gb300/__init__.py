"""GB300 (sm_103a) hot path of block speculative decoding: Python binding.

The compute lives in ``libspecgb300.so`` (CUDA kernels behind the C ABI declared in
``include/spec.h``).  This module only marshals arguments: it checks tensor dtypes,
devices and shapes, allocates outputs and workspaces with PyTorch, and passes raw
device pointers and the current CUDA stream to the library.  There is no CPU or
PyTorch fallback: every call fails loudly if the library is not built.

    import verify_spec_draft_gb300 as vsd
    vsd.load()                                   # after vsd.build.build()
    out = vsd.draft_block(logits, anchor, U, Wt, temperature=0)
    res = vsd.verify(target, None, out["tokens"], temperature=0)
    tv  = vsd.e2etv(target_rows, draft_rows, n_branches, Wb)
"""

import ctypes
import os

from . import build as _build

OK = 0
STATUS = {
    0: "SPEC_OK", 1: "SPEC_ERR_INVALID_ARG", 2: "SPEC_ERR_SHAPE", 3: "SPEC_ERR_DTYPE",
    4: "SPEC_ERR_ALIGN", 5: "SPEC_ERR_CUDA", 6: "SPEC_ERR_TIMEOUT", 7: "SPEC_ERR_NONFINITE",
    8: "SPEC_ERR_TOKEN", 9: "SPEC_ERR_WORKSPACE",
}
F32, BF16 = 0, 1
OP_DRAFT, OP_VERIFY, OP_E2ETV, OP_DRAFT_VERIFY, OP_BRANCH_PLAN, OP_VERIFY_TOPK, OP_TREE_VERIFY, OP_DRAFT_TOPK = (
    0, 1, 2, 3, 4, 5, 6, 7)
DEV_TIMEOUT, DEV_NONFINITE, DEV_TOKEN = 1, 2, 4

# C signatures of include/spec.h, as ctypes types
_vp, _i32, _sz, _u32p = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.POINTER(ctypes.c_uint32)
SIGNATURES = {
    "spec_workspace_bytes": (_sz, [_i32, _i32, _i32, _i32, _i32]),
    "spec_workspace_init": (_i32, [_vp, _sz, _vp]),
    "spec_get_device_status": (_i32, [_vp, _vp, _u32p]),
    "spec_status_string": (ctypes.c_char_p, [_i32]),
    "spec_last_cuda_error": (_i32, []),
    "spec_last_cuda_error_string": (ctypes.c_char_p, []),
    "spec_draft_block": (_i32, [_vp, _i32, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _i32, _vp,
                                _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp]),
    "spec_verify": (_i32, [_vp, _i32, _vp, _i32, _vp, _i32, _i32, _i32, _i32, _vp,
                           _vp, _vp, _vp, _vp, _vp, _sz, _vp]),
    "spec_e2etv": (_i32, [_vp, _vp, _i32, _i32, _i32, _vp, _vp, _vp, _vp, _vp, _sz, _vp]),
    "spec_verify_noalloc": (_i32, [_vp, _i32, _vp, _i32, _vp, _i32, _i32, _i32, _i32, _vp,
                                   _vp, _vp, _vp, _vp, _vp]),
    "spec_draft_verify": (_i32, [_vp, _i32, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _vp, _i32,
                                 _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp]),
    "spec_verify_budget": (_i32, [_vp, _i32, _i32, _i32, _vp, _vp, _vp, _vp]),
    "spec_verify_topk": (_i32, [_vp, _i32, _vp, _i32, _vp, _i32, _i32, _i32, _i32, ctypes.c_double, _vp, _vp, _vp,
                                _vp, _vp, _vp, _sz, _vp]),
    "spec_e2etv_shard": (_i32, [_vp, _vp, _i32, _i32, _i32, _i32, _vp, _vp, _vp, _vp, _vp, _sz, _vp]),
    "spec_branch_plan": (_i32, [_vp, _vp, _i32, _i32, _i32, _i32, ctypes.c_uint64, _vp, _vp, _vp, _vp,
                                _vp, _sz, _vp]),
    "spec_tree_select": (_i32, [_vp, _vp, _i32, _i32, _i32, _vp, _vp, _vp, _vp]),
    "spec_draft_block_topk": (_i32, [_vp, _i32, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _i32, ctypes.c_double,
                                     _vp, _vp, _vp, _vp, _vp, _sz, _vp]),
    "spec_tree_verify": (_i32, [_vp, _i32, _vp, _vp, _vp, _i32, _i32, _i32, _vp, _vp, _vp, _vp, _vp, _sz, _vp]),
}

_lib = None


class SpecError(RuntimeError):
    def __init__(self, code, what):
        msg = f"{what}: {STATUS.get(code, code)} ({status_string(code)})"
        if code == 5 and _lib is not None:
            msg += f" [cuda error {_lib.spec_last_cuda_error()}: {_lib.spec_last_cuda_error_string().decode()}]"
        super().__init__(msg)
        self.code = code


def library_path():
    return _build.LIB


def load(path=None):
    """Load the compiled library (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or library_path()
    if not os.path.exists(path):
        raise RuntimeError(f"libspecgb300.so not found at {path}: run verify_spec_draft_gb300.build.build() "
                           "(or __graft_entry__.build()) first; there is no fallback implementation")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def status_string(code):
    if _lib is None:
        return STATUS.get(code, "unknown")
    return _lib.spec_status_string(code).decode()


def _check(code, what):
    if code != OK:
        raise SpecError(code, what)


# ---------------------------------------------------------------------------------
# tensor marshalling helpers (no arithmetic)
# ---------------------------------------------------------------------------------
def _torch():
    import torch
    return torch


def _dtype_code(t):
    torch = _torch()
    if t.dtype == torch.float32:
        return F32
    if t.dtype == torch.bfloat16:
        return BF16
    raise TypeError(f"logits/weights must be float32 or bfloat16, got {t.dtype}")


def _ptr(t):
    return ctypes.c_void_p(0 if t is None else t.data_ptr())


def _need(t, name, device=None, dtype=None, shape=None):
    if t is None:
        raise ValueError(f"{name} is required")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (the library has no CPU path)")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    return t


def _stream(stream=None):
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def workspace_bytes(op, B, gamma, V, r=0):
    n = load().spec_workspace_bytes(op, B, gamma, V, r)
    if n == 0:
        raise SpecError(2, f"workspace_bytes(op={op}, B={B}, gamma={gamma}, V={V}, r={r})")
    return n


def workspace(op, B, gamma, V, r=0, device=None, stream=None):
    """Allocate a device workspace for one operation and zero it (spec_workspace_init).

    Calls of that operation and shape can reuse it as it is; zero it again (or take a
    new one) before a call with another operation or shape."""
    torch = _torch()
    n = workspace_bytes(op, B, gamma, V, r)
    ws = torch.empty(n, dtype=torch.uint8, device=device or torch.device("cuda"))
    _check(load().spec_workspace_init(_ptr(ws), n, _stream(stream)), "spec_workspace_init")
    return ws


def device_status(ws, stream=None):
    """Synchronise and return the raw SPEC_DEV_* flags of a workspace."""
    flags = ctypes.c_uint32(0)
    load().spec_get_device_status(_ptr(ws), _stream(stream), ctypes.byref(flags))
    return flags.value


# ---------------------------------------------------------------------------------
# the three operations
# ---------------------------------------------------------------------------------
def draft_block(logits, anchor, U=None, Wt=None, temperature=0, seeds=None, ws=None,
                qlogits=False, out=None, stream=None):
    """spec_draft_block.  logits [B, gamma, V] f32/bf16; anchor [B] int32; U, Wt [V, r]
    (same dtype) or None; seeds [B] int64 (uint64 bits) at T=1.  Returns a dict of
    device tensors: tokens, conf, qtok, passes and (if ``qlogits``) the float32 z rows."""
    torch = _torch()
    lib = load()
    _need(logits, "logits")
    dev = logits.device
    B, gamma, V = logits.shape
    _need(anchor, "anchor", dev, torch.int32, (B,))
    r = 0
    if U is not None:
        _need(U, "U", dev)
        _need(Wt, "Wt", dev, U.dtype, tuple(U.shape))
        if U.shape[0] != V:
            raise ValueError("U and Wt must have V rows")
        r = U.shape[1]
    wdt = _dtype_code(U) if U is not None else F32
    if temperature == 1:
        _need(seeds, "seeds", dev, torch.int64, (B,))
    if out is None:
        out = dict(
            tokens=torch.empty((B, gamma), dtype=torch.int32, device=dev),
            conf=torch.empty((B, gamma), dtype=torch.float32, device=dev),
            qtok=torch.empty((B, gamma), dtype=torch.float32, device=dev),
            passes=torch.zeros((1,), dtype=torch.int32, device=dev),
        )
        if qlogits:
            out["qlogits"] = torch.empty((B, gamma, V), dtype=torch.float32, device=dev)
    if ws is None:
        ws = workspace(OP_DRAFT, B, gamma, V, r, dev, stream)
    code = lib.spec_draft_block(
        _ptr(logits), _dtype_code(logits), _ptr(anchor), _ptr(U), _ptr(Wt), wdt, r, B, gamma, V,
        int(temperature), _ptr(seeds), _ptr(out["tokens"]), _ptr(out["conf"]), _ptr(out.get("qtok")),
        _ptr(out.get("qlogits")), _ptr(out.get("passes")), _ptr(ws), ws.numel(), _stream(stream))
    _check(code, "spec_draft_block")
    out["ws"] = ws
    return out


def verify(target, draft, tokens, temperature=0, seeds=None, ws=None, out=None, stream=None):
    """spec_verify.  target [B, gamma+1, V]; draft [B, gamma, V] (T=1, else None);
    tokens [B, gamma] int32; seeds [B] int64 at T=1.  Returns a dict of device tensors:
    n (accepted drafts), committed, bonus, near."""
    torch = _torch()
    lib = load()
    _need(target, "target")
    dev = target.device
    B, g1, V = target.shape
    gamma = g1 - 1
    _need(tokens, "tokens", dev, torch.int32, (B, gamma))
    ddt = F32
    if temperature == 1:
        _need(draft, "draft", dev, None, (B, gamma, V))
        ddt = _dtype_code(draft)
        _need(seeds, "seeds", dev, torch.int64, (B,))
    if out is None:
        out = dict(
            n=torch.empty((B,), dtype=torch.int32, device=dev),
            committed=torch.empty((B, gamma + 1), dtype=torch.int32, device=dev),
            bonus=torch.empty((B,), dtype=torch.int32, device=dev),
            near=torch.empty((B,), dtype=torch.int32, device=dev),
        )
    if ws is None:
        ws = workspace(OP_VERIFY, B, gamma, V, 0, dev, stream)
    code = lib.spec_verify(
        _ptr(target), _dtype_code(target), _ptr(draft if temperature == 1 else None), ddt, _ptr(tokens),
        B, gamma, V, int(temperature), _ptr(seeds), _ptr(out["n"]), _ptr(out["committed"]), _ptr(out["bonus"]),
        _ptr(out.get("near")), _ptr(ws), ws.numel(), _stream(stream))
    _check(code, "spec_verify")
    out["ws"] = ws
    return out


def draft_verify(logits, target, anchor, U=None, Wt=None, ws=None, out=None, stream=None):
    """spec_draft_verify (T=0).  logits [B, gamma, V]; target [B, gamma+1, V]; anchor [B]
    int32; U, Wt [V, r] or None.  Returns a dict of device tensors: the draft's tokens,
    conf, qtok, passes and verify's n, committed, bonus."""
    torch = _torch()
    lib = load()
    _need(logits, "logits")
    dev = logits.device
    B, gamma, V = logits.shape
    _need(target, "target", dev, None, (B, gamma + 1, V))
    _need(anchor, "anchor", dev, torch.int32, (B,))
    r = 0
    if U is not None:
        _need(U, "U", dev)
        _need(Wt, "Wt", dev, U.dtype, tuple(U.shape))
        if U.shape[0] != V:
            raise ValueError("U and Wt must have V rows")
        r = U.shape[1]
    wdt = _dtype_code(U) if U is not None else F32
    if out is None:
        out = dict(
            tokens=torch.empty((B, gamma), dtype=torch.int32, device=dev),
            conf=torch.empty((B, gamma), dtype=torch.float32, device=dev),
            qtok=torch.empty((B, gamma), dtype=torch.float32, device=dev),
            passes=torch.zeros((1,), dtype=torch.int32, device=dev),
            n=torch.empty((B,), dtype=torch.int32, device=dev),
            committed=torch.empty((B, gamma + 1), dtype=torch.int32, device=dev),
            bonus=torch.empty((B,), dtype=torch.int32, device=dev),
        )
    if ws is None:
        ws = workspace(OP_DRAFT_VERIFY, B, gamma, V, r, dev, stream)
    code = lib.spec_draft_verify(
        _ptr(logits), _dtype_code(logits), _ptr(anchor), _ptr(U), _ptr(Wt), wdt, r, B, gamma, V,
        _ptr(target), _dtype_code(target), _ptr(out["tokens"]), _ptr(out["conf"]), _ptr(out.get("qtok")),
        _ptr(out.get("passes")), _ptr(out["n"]), _ptr(out["committed"]), _ptr(out["bonus"]), _ptr(ws),
        ws.numel(), _stream(stream))
    _check(code, "spec_draft_verify")
    out["ws"] = ws
    return out


def verify_budget(conf, budget, cost=None, out=None, stream=None):
    """spec_verify_budget.  conf [B, gamma] float32 (spec_draft_block's conf); budget:
    most draft positions verified in all; cost: float32 [budget + 1] time per total, or
    None.  Returns a dict of device tensors: gamma [B] int32, expected [1] float32."""
    torch = _torch()
    lib = load()
    _need(conf, "conf", None, torch.float32)
    if conf.dim() != 2:
        raise ValueError("conf must be [B, gamma]")
    dev = conf.device
    B, gamma = conf.shape
    if cost is not None:
        _need(cost, "cost", dev, torch.float32, (int(budget) + 1,))
    if out is None:
        out = dict(gamma=torch.empty((B,), dtype=torch.int32, device=dev),
                   expected=torch.empty((1,), dtype=torch.float32, device=dev))
    code = lib.spec_verify_budget(_ptr(conf), B, gamma, int(budget), _ptr(cost), _ptr(out["gamma"]),
                                  _ptr(out.get("expected")), _stream(stream))
    _check(code, "spec_verify_budget")
    return out


def branch_plan(trunk, lengths, n_anchors, W, seed, ws=None, out=None, stream=None):
    """spec_branch_plan.  trunk int32 [n_refs, Lmax] reference tokens; lengths int32
    [n_refs].  Returns a dict of device tensors: anchors, anchor_tok [n_refs, n_anchors]
    and parent, position [n_refs, n_anchors * W] (int32)."""
    torch = _torch()
    lib = load()
    _need(trunk, "trunk", None, torch.int32)
    if trunk.dim() != 2:
        raise ValueError("trunk must be [n_refs, Lmax]")
    dev = trunk.device
    R, Lmax = trunk.shape
    _need(lengths, "lengths", dev, torch.int32, (R,))
    if out is None:
        out = dict(anchors=torch.empty((R, n_anchors), dtype=torch.int32, device=dev),
                   anchor_tok=torch.empty((R, n_anchors), dtype=torch.int32, device=dev),
                   parent=torch.empty((R, n_anchors * W), dtype=torch.int32, device=dev),
                   position=torch.empty((R, n_anchors * W), dtype=torch.int32, device=dev))
    if ws is None:
        ws = workspace(OP_BRANCH_PLAN, R, W, Lmax, 0, dev, stream)
    code = lib.spec_branch_plan(_ptr(trunk), _ptr(lengths), R, Lmax, int(n_anchors), int(W), int(seed),
                                _ptr(out["anchors"]), _ptr(out["anchor_tok"]), _ptr(out["parent"]),
                                _ptr(out["position"]), _ptr(ws), ws.numel(), _stream(stream))
    _check(code, "spec_branch_plan")
    out["ws"] = ws
    return out


def verify_topk(target, draft, tokens, top_k, top_p, seeds, ws=None, out=None, stream=None):
    """spec_verify_topk (T=1 against top-k / top-p filtered rows).  target [B, gamma+1, V]
    and draft [B, gamma, V] f32/bf16; tokens [B, gamma] int32; seeds [B] int64.  Returns
    a dict of device tensors: n [B], committed [B, gamma+1], bonus [B], near [B]."""
    torch = _torch()
    lib = load()
    _need(target, "target")
    dev = target.device
    B, G1, V = target.shape
    G = G1 - 1
    _need(draft, "draft", dev, None, (B, G, V))
    _need(tokens, "tokens", dev, torch.int32, (B, G))
    _need(seeds, "seeds", dev, torch.int64, (B,))
    if out is None:
        out = dict(n=torch.empty((B,), dtype=torch.int32, device=dev),
                   committed=torch.empty((B, G1), dtype=torch.int32, device=dev),
                   bonus=torch.empty((B,), dtype=torch.int32, device=dev),
                   near=torch.empty((B,), dtype=torch.int32, device=dev))
    if ws is None:
        ws = workspace(OP_VERIFY_TOPK, B, G, V, 0, dev, stream)
    code = lib.spec_verify_topk(_ptr(target), _dtype_code(target), _ptr(draft), _dtype_code(draft), _ptr(tokens), B, G,
                                V, int(top_k), float(top_p), _ptr(seeds), _ptr(out["n"]), _ptr(out["committed"]),
                                _ptr(out["bonus"]), _ptr(out.get("near")), _ptr(ws), ws.numel(), _stream(stream))
    _check(code, "spec_verify_topk")
    out["ws"] = ws
    return out


def e2etv_shard(target, draft, n_branches, Wb, total_branches, ws=None, out=None, stream=None):
    """spec_e2etv_shard: one shard of a batch of ``total_branches`` branches.  target, draft
    bf16 [n_branches*Wb, V].  Returns a dict of device tensors: a, surv [R] float32,
    msum [1] float32 (this shard's part of the mean survival), grad bf16 [R, V]."""
    torch = _torch()
    lib = load()
    _need(target, "target", None, torch.bfloat16)
    dev = target.device
    R, V = target.shape
    if R != n_branches * Wb:
        raise ValueError("target must have n_branches * Wb rows")
    _need(draft, "draft", dev, torch.bfloat16, (R, V))
    if out is None:
        out = dict(
            a=torch.empty((R,), dtype=torch.float32, device=dev),
            surv=torch.empty((R,), dtype=torch.float32, device=dev),
            msum=torch.empty((1,), dtype=torch.float32, device=dev),
            grad=torch.empty((R, V), dtype=torch.bfloat16, device=dev),
        )
    if ws is None:
        ws = workspace(OP_E2ETV, n_branches, Wb, V, 0, dev, stream)
    code = lib.spec_e2etv_shard(_ptr(target), _ptr(draft), n_branches, Wb, V, int(total_branches), _ptr(out["a"]),
                                _ptr(out["surv"]), _ptr(out["msum"]), _ptr(out["grad"]), _ptr(ws), ws.numel(),
                                _stream(stream))
    _check(code, "spec_e2etv_shard")
    out["ws"] = ws
    return out


def e2etv(target, draft, n_branches, Wb, ws=None, out=None, stream=None):
    """spec_e2etv.  target, draft bf16 [n_branches*Wb, V] branch-major.  Returns a dict of
    device tensors: a, surv [R] float32, loss [1] float32, grad bf16 [R, V]."""
    torch = _torch()
    lib = load()
    _need(target, "target", None, torch.bfloat16)
    dev = target.device
    R, V = target.shape
    if R != n_branches * Wb:
        raise ValueError("target must have n_branches * Wb rows")
    _need(draft, "draft", dev, torch.bfloat16, (R, V))
    if out is None:
        out = dict(
            a=torch.empty((R,), dtype=torch.float32, device=dev),
            surv=torch.empty((R,), dtype=torch.float32, device=dev),
            loss=torch.empty((1,), dtype=torch.float32, device=dev),
            grad=torch.empty((R, V), dtype=torch.bfloat16, device=dev),
        )
    if ws is None:
        ws = workspace(OP_E2ETV, n_branches, Wb, V, 0, dev, stream)
    code = lib.spec_e2etv(_ptr(target), _ptr(draft), n_branches, Wb, V, _ptr(out["a"]), _ptr(out["surv"]),
                          _ptr(out["loss"]), _ptr(out["grad"]), _ptr(ws), ws.numel(), _stream(stream))
    _check(code, "spec_e2etv")
    out["ws"] = ws
    return out


def tree_select(parent, conf, m, out=None, stream=None):
    """spec_tree_select.  parent int32 [n_trees, n_nodes], conf float32 [n_trees, n_nodes].
    Returns a dict of device tensors: score float64 [n_trees, n_nodes], keep int32
    [n_trees, n_nodes] (1 = kept), selected int32 [n_trees, m] (ascending, then -1)."""
    torch = _torch()
    lib = load()
    _need(parent, "parent", None, torch.int32)
    if parent.dim() != 2:
        raise ValueError("parent must be [n_trees, n_nodes]")
    dev = parent.device
    T, n = parent.shape
    _need(conf, "conf", dev, torch.float32, (T, n))
    m = int(m)
    if out is None:
        out = dict(score=torch.empty((T, n), dtype=torch.float64, device=dev),
                   keep=torch.empty((T, n), dtype=torch.int32, device=dev),
                   selected=torch.empty((T, max(m, 0)), dtype=torch.int32, device=dev))
    code = lib.spec_tree_select(_ptr(parent), _ptr(conf), T, n, m, _ptr(out.get("score")), _ptr(out["keep"]),
                                _ptr(out.get("selected")) if m > 0 else _ptr(None), _stream(stream))
    _check(code, "spec_tree_select")
    return out


def tree_verify(target, parent, token, keep=None, ws=None, out=None, stream=None):
    """spec_tree_verify (T=0).  target f32/bf16 [n_trees, n_nodes + 1, V] (root row first);
    parent, token int32 [n_trees, n_nodes]; keep int32 [n_trees, n_nodes] or None (all).
    Returns a dict of device tensors: n [n_trees], path [n_trees, n_nodes], committed
    [n_trees, n_nodes + 1], bonus [n_trees]."""
    torch = _torch()
    lib = load()
    _need(target, "target")
    if target.dim() != 3:
        raise ValueError("target must be [n_trees, n_nodes + 1, V]")
    dev = target.device
    T, R, V = target.shape
    n = R - 1
    if n > 0:
        _need(parent, "parent", dev, torch.int32, (T, n))
        _need(token, "token", dev, torch.int32, (T, n))
        if keep is not None:
            _need(keep, "keep", dev, torch.int32, (T, n))
    if out is None:
        out = dict(n=torch.empty((T,), dtype=torch.int32, device=dev),
                   path=torch.empty((T, n), dtype=torch.int32, device=dev),
                   committed=torch.empty((T, R), dtype=torch.int32, device=dev),
                   bonus=torch.empty((T,), dtype=torch.int32, device=dev))
    if ws is None:
        ws = workspace(OP_TREE_VERIFY, T, n, V, 0, dev, stream)
    code = lib.spec_tree_verify(_ptr(target), _dtype_code(target), _ptr(parent if n > 0 else None),
                                _ptr(token if n > 0 else None), _ptr(keep if n > 0 else None), T, n, V,
                                _ptr(out["n"]), _ptr(out["path"]) if n > 0 else _ptr(None), _ptr(out["committed"]),
                                _ptr(out["bonus"]), _ptr(ws), ws.numel(), _stream(stream))
    _check(code, "spec_tree_verify")
    out["ws"] = ws
    return out


def draft_block_topk(logits, anchor, U, Wt, top_k, top_p, seeds, ws=None, out=None, stream=None):
    """spec_draft_block_topk (T=1, filtered draws).  logits [B, gamma, V] f32/bf16; anchor
    [B] int32; U, Wt bf16 [V, r] or None; seeds [B] int64.  Returns a dict of device
    tensors: tokens [B, gamma] int32, conf and qtok [B, gamma] float32."""
    torch = _torch()
    lib = load()
    _need(logits, "logits")
    dev = logits.device
    B, G, V = logits.shape
    _need(anchor, "anchor", dev, torch.int32, (B,))
    _need(seeds, "seeds", dev, torch.int64, (B,))
    r = 0
    if U is not None:
        r = U.shape[1]
        _need(U, "U", dev, torch.bfloat16, (V, r))
        _need(Wt, "Wt", dev, torch.bfloat16, (V, r))
    if out is None:
        out = dict(tokens=torch.empty((B, G), dtype=torch.int32, device=dev),
                   conf=torch.empty((B, G), dtype=torch.float32, device=dev),
                   qtok=torch.empty((B, G), dtype=torch.float32, device=dev))
    if ws is None:
        ws = workspace(OP_DRAFT_TOPK, B, G, V, r, dev, stream)
    code = lib.spec_draft_block_topk(_ptr(logits), _dtype_code(logits), _ptr(anchor), _ptr(U), _ptr(Wt), BF16, r, B, G,
                                     V, int(top_k), float(top_p), _ptr(seeds), _ptr(out["tokens"]), _ptr(out["conf"]),
                                     _ptr(out.get("qtok")), _ptr(ws), ws.numel(), _stream(stream))
    _check(code, "spec_draft_block_topk")
    out["ws"] = ws
    return out
