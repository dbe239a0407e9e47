"""Seeded synthetic inputs shaped like the pages' workloads.

This module holds none of the method's arithmetic: it only draws random logits,
weights, anchors and tokens.  Tests, the benchmark and the oracle-side checks all take
their inputs from here, so both the CUDA path and the oracle see the same numbers.

The pages evaluate on public benchmarks and trained checkpoints that are not
available here; these generators stand in for them with the shapes the pages give:
gamma = 7 (sionic.ai launch example: block size 7, 8 verify tokens; SpecOPD summary:
7 draft tokens), block 16 (DSpine card), V = 248,320 (DSpine card parameter
breakdown), r = 256 (VESSL page, DSpark bias equation).

Distributions (generated in float32, rounded once to bf16 where the config says so):

* gaussian: target logits N(0, 3^2) per entry;
* zipf: logit = -4 ln(rank) + N(0, 1), ranks 1..V placed by an independent random
  permutation per row;
* draft rows = target rows + N(0, sigma^2) (draft row j-1 pairs with target row j-1,
  both describing position j);
* Markov weights U, Wt ~ N(0, 0.02^2);
* anchors uniform in [0, V);
* standalone-verify draft tokens: argmax of the draft row (T=0, a greedy drafter) or
  the Gumbel-max draw argmax(d + G), G standard Gumbel (T=1, a sample from the draft
  row's softmax without computing one);
* draft trees: node i's parent uniform among the root (-1) and the nodes before it (or
  node i-1 for a chain); its token the argmax of its parent's target row with a given
  probability (a drafter that often agrees), else uniform in [0, V); confidences
  uniform in [0.05, 1).
"""

from dataclasses import dataclass, field

import torch


@dataclass
class Config:
    name: str
    B: int
    gamma: int
    V: int
    r: int
    dtype: torch.dtype
    temperatures: tuple
    dist: str               # "gaussian" or "zipf"
    draft_sigma: object     # float, or (lo, hi) for a per-request uniform sigma
    seed: int
    note: str = ""
    extra: dict = field(default_factory=dict)


CONFIGS = {
    1: Config("tiny B1 g7 V32000 r32 fp32", 1, 7, 32000, 32, torch.float32, (0, 1), "gaussian", 0.5, 1001),
    2: Config("batch-verify B8 g7 V151936 r128 bf16", 8, 7, 151936, 128, torch.bfloat16, (0, 1), "zipf", 0.8, 1002),
    3: Config("latency B1 g15 V248320 r256 bf16", 1, 15, 248320, 256, torch.bfloat16, (0,), "zipf", 0.6, 1003),
    4: Config("throughput B32 g7 V248320 r256 bf16", 32, 7, 248320, 256, torch.bfloat16, (1,), "zipf", (0.3, 1.5),
              1004),
    5: Config("e2etv 16x64x7 rows V248320 bf16", 1024, 7, 248320, 0, torch.bfloat16, (1,), "gaussian", 1.0, 1005,
              note="B = branches (16 references x 64 anchors), gamma = branch length Wb"),
}


def generator(seed, device):
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _base_logits(rows, V, dist, g, device):
    if dist == "gaussian":
        return torch.randn((rows, V), generator=g, device=device, dtype=torch.float32) * 3.0
    if dist == "zipf":
        out = torch.empty((rows, V), device=device, dtype=torch.float32)
        ranks = torch.arange(1, V + 1, device=device, dtype=torch.float32)
        zipf = -4.0 * torch.log(ranks)
        for i in range(rows):
            perm = torch.randperm(V, generator=g, device=device)
            out[i, perm] = zipf
        out += torch.randn((rows, V), generator=g, device=device, dtype=torch.float32)
        return out
    raise ValueError(dist)


def _sigmas(cfg_sigma, B, g, device):
    if isinstance(cfg_sigma, tuple):
        lo, hi = cfg_sigma
        return lo + (hi - lo) * torch.rand((B,), generator=g, device=device, dtype=torch.float32)
    return torch.full((B,), float(cfg_sigma), device=device, dtype=torch.float32)


def target_and_draft(B, gamma, V, dist="gaussian", sigma=0.5, dtype=torch.float32, seed=0, device="cpu"):
    """target [B, gamma+1, V] and draft [B, gamma, V] logits (draft row j-1 = target
    row j-1 + noise)."""
    g = generator(seed, device)
    tgt = _base_logits(B * (gamma + 1), V, dist, g, device).view(B, gamma + 1, V)
    sig = _sigmas(sigma, B, g, device).view(B, 1, 1)
    noise = torch.randn((B, gamma, V), generator=g, device=device, dtype=torch.float32)
    drf = tgt[:, :gamma] + sig * noise
    return tgt.to(dtype).contiguous(), drf.to(dtype).contiguous()


def markov_weights(V, r, dtype=torch.float32, seed=0, device="cpu", scale=0.02):
    """U and Wt, both [V, r] (Wt row v is column v of W_2)."""
    g = generator(seed + 7919, device)
    U = torch.randn((V, r), generator=g, device=device, dtype=torch.float32) * scale
    Wt = torch.randn((V, r), generator=g, device=device, dtype=torch.float32) * scale
    return U.to(dtype).contiguous(), Wt.to(dtype).contiguous()


def anchors(B, V, seed=0, device="cpu"):
    g = generator(seed + 104729, device)
    return torch.randint(0, V, (B,), generator=g, device=device, dtype=torch.int32)


def seeds_for(B, base=0, device="cpu"):
    """Per-request Philox keys seed_b = base + b."""
    return (torch.arange(B, device=device, dtype=torch.int64) + int(base)).contiguous()


def draft_tokens(draft, temperature, seed=0):
    """Tokens a drafter would propose from its rows: greedy at T=0, Gumbel-max at T=1."""
    d = draft.float()
    if temperature == 0:
        return d.argmax(-1).to(torch.int32).contiguous()
    g = generator(seed + 15485863, d.device)
    u = torch.rand(d.shape, generator=g, device=d.device, dtype=torch.float32).clamp_(1e-20, 1.0 - 1e-7)
    gumbel = -torch.log(-torch.log(u))
    return (d + gumbel).argmax(-1).to(torch.int32).contiguous()


def e2etv_rows(n_branches, Wb, V, sigma=1.0, dtype=torch.bfloat16, seed=0, device="cpu"):
    """Branch-major target and draft rows [n_branches*Wb, V] from the gaussian
    distribution, draft = target + N(0, sigma^2)."""
    g = generator(seed, device)
    R = n_branches * Wb
    tgt = _base_logits(R, V, "gaussian", g, device)
    drf = tgt + sigma * torch.randn((R, V), generator=g, device=device, dtype=torch.float32)
    return tgt.to(dtype).contiguous(), drf.to(dtype).contiguous()


# The SpecOPD anchor-branch sampler (beyond the numbered configurations): 16 reference
# responses of 4096 tokens (the pages give no length; 4096 is this workload's choice),
# 64 anchors each, branches of W = 7 (the SpecOPD summary's 7 draft tokens), drafted at
# T=1 with the rank-256 bias over V = 248,320; drafter rows from the zipf distribution.
BRANCH_CONFIG = Config("anchor branches 16 refs x 64 anchors x W7 V248320 r256 bf16", 1024, 7, 248320, 256,
                       torch.bfloat16, (1,), "zipf", 0.0, 1006,
                       extra=dict(n_refs=16, n_anchors=64, Lmax=4096))


def branch_inputs(n_refs, n_anchors, W, V, r, Lmax, dtype=torch.bfloat16, seed=0, device="cpu", dist="zipf",
                  lengths=None):
    """Inputs of the anchor-branch sampler: reference tokens [n_refs, Lmax] uniform in
    [0, V), lengths [n_refs] (all Lmax unless given), drafter logits
    [n_refs * n_anchors, W, V], Markov weights U, Wt [V, r] and per-branch seeds."""
    g = generator(seed, device)
    trunk = torch.randint(0, V, (n_refs, Lmax), generator=g, device=device, dtype=torch.int32)
    if lengths is None:
        lengths = torch.full((n_refs,), Lmax, dtype=torch.int32, device=device)
    else:
        lengths = torch.as_tensor(lengths, dtype=torch.int32).to(device)
    B = n_refs * n_anchors
    logits = _base_logits(B * W, V, dist, g, device).view(B, W, V).to(dtype).contiguous()
    U, Wt = markov_weights(V, r, dtype, seed, device)
    return dict(trunk=trunk.contiguous(), lengths=lengths.contiguous(), logits=logits, U=U, Wt=Wt,
                seeds=seeds_for(B, seed, device))


def config_inputs(cfg_id, device="cpu"):
    """All inputs of a numbered configuration (see CONFIGS)."""
    c = CONFIGS[cfg_id]
    if cfg_id == 5:
        t, d = e2etv_rows(c.B, c.gamma, c.V, c.draft_sigma, c.dtype, c.seed, device)
        return dict(cfg=c, target=t, draft=d)
    t, d = target_and_draft(c.B, c.gamma, c.V, c.dist, c.draft_sigma, c.dtype, c.seed, device)
    U, Wt = markov_weights(c.V, c.r, c.dtype, c.seed, device)
    return dict(cfg=c, target=t, draft=d, U=U, Wt=Wt, anchor=anchors(c.B, c.V, c.seed, device),
                seeds=seeds_for(c.B, 0, device))


# Draft trees (beyond the numbered configurations): the pages give no tree sizes; this
# workload verifies 32 trees of 64 nodes over V = 248,320 (zipf rows, bf16), i.e. 2080
# target rows, about the size of an EAGLE-2 tree per request in a batch of 32.
TREE_CONFIG = Config("draft trees 32 x 64 nodes V248320 bf16", 32, 64, 248320, 0, torch.bfloat16, (0,), "zipf",
                     0.0, 1007)


def tree_inputs(n_trees, n_nodes, V, dtype=torch.bfloat16, seed=0, device="cpu", dist="zipf", p_match=0.7,
                shape="bushy"):
    """Draft trees and their target rows: parent, token int32 [n_trees, n_nodes], conf
    float32 [n_trees, n_nodes] and target [n_trees, n_nodes + 1, V] (the root's row
    first, then node i's at 1 + i)."""
    g = generator(seed, device)
    T, n = n_trees, n_nodes
    rows = _base_logits(T * (n + 1), V, dist, g, device).view(T, n + 1, V).to(dtype).contiguous()
    i = torch.arange(n, device=device, dtype=torch.float32)
    if shape == "chain":
        parent = (torch.arange(n, device=device, dtype=torch.int64) - 1).expand(T, n)
    else:
        u = torch.rand((T, n), generator=g, device=device, dtype=torch.float32)
        parent = torch.floor(u * (i + 1)).to(torch.int64) - 1      # uniform in [-1, i)
    am = rows.float().argmax(-1)                                   # [T, n + 1]
    parent_am = torch.gather(am, 1, parent + 1)
    rand_tok = torch.randint(0, V, (T, n), generator=g, device=device, dtype=torch.int64)
    match = torch.rand((T, n), generator=g, device=device, dtype=torch.float32) < p_match
    token = torch.where(match, parent_am, rand_tok)
    conf = 0.05 + 0.95 * torch.rand((T, n), generator=g, device=device, dtype=torch.float32)
    return dict(parent=parent.to(torch.int32).contiguous(), token=token.to(torch.int32).contiguous(),
                conf=conf.contiguous(), target=rows)
