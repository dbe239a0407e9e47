"""Launch one operation a few times on a synthetic workload, for profiler captures.

    python -m verify_spec_draft_gb300.profile_cases CASE [--launches N]

Nothing is timed here; the point is a short process with a handful of launches of one
kernel, on inputs larger than L2 (129 MB) but only a few hundred MB on the device:

  draft      spec_draft_block, B=1, gamma=15, V=248320, r=256, T=0 (151 MB: logits, U, Wt)
  draft_t1   spec_draft_block, B=32, gamma=7, V=248320, r=256, T=1 (365 MB: logits, U, Wt)
  verify_t0  spec_verify T=0 on the 16 target rows of the same workload (8 MB; below L2)
  verify_t1  spec_verify T=1, B=32, gamma=7, V=248320 (238 MB of target and draft rows)
  verify_topk spec_verify_topk on the same rows, top_k 20, top_p 0.95
  e2etv      spec_e2etv on 64 branches x Wb=7 = 448 rows, V=248320 (445 MB in, 222 MB out):
             a 64-anchor slice of the 16 x 64 x 7 layout
  tree_verify spec_tree_verify on 32 trees x 64 nodes, V=248320 (2080 rows, 1.03 GB)
  draft_topk spec_draft_block_topk, B=32, gamma=7, V=248320, r=256, top_k 20, top_p 0.95
             (365 MB: logits, U, Wt)
  draft_pos  spec_draft_block at T=1 on 512 requests x gamma=2, V=248320, r=256: the
             position-by-position path for batches over 256 rows (509 MB of logits)
  sampler    spec_draft_block at T=1 on the anchor-branch workload, 1024 branches x W=7
             (3.56 GB of logits): for launch lists only (one metric, one pass)
  budget     spec_verify_budget, B=32, gamma=16, budget 256, a linear cost curve (2 KB)
"""

import argparse

import torch

from . import draft_block, draft_block_topk, e2etv, load, synth, tree_verify, verify, verify_budget, verify_topk

CASES = ("draft", "draft_t1", "verify_t0", "verify_t1", "verify_topk", "e2etv", "tree_verify", "draft_topk",
         "draft_pos", "sampler", "budget")


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("case", choices=CASES)
    ap.add_argument("--launches", type=int, default=3)
    args = ap.parse_args(argv)
    load()
    dev = torch.device("cuda")
    if args.case in ("draft", "verify_t0"):
        inp = synth.config_inputs(3, device=dev)
        out = draft_block(inp["draft"], inp["anchor"], inp["U"], inp["Wt"], 0)
        if args.case == "draft":
            run = lambda: draft_block(inp["draft"], inp["anchor"], inp["U"], inp["Wt"], 0, ws=out["ws"], out=out)
        else:
            ref = verify(inp["target"], None, out["tokens"], 0)
            run = lambda: verify(inp["target"], None, out["tokens"], 0, ws=ref["ws"], out=ref)
    elif args.case == "draft_t1":
        inp = synth.config_inputs(4, device=dev)
        out = draft_block(inp["draft"], inp["anchor"], inp["U"], inp["Wt"], 1, inp["seeds"])
        run = lambda: draft_block(inp["draft"], inp["anchor"], inp["U"], inp["Wt"], 1, inp["seeds"], ws=out["ws"],
                                  out=out)
    elif args.case == "verify_topk":
        inp = synth.config_inputs(4, device=dev)
        tok = synth.draft_tokens(inp["draft"], 1, seed=inp["cfg"].seed)
        ref = verify_topk(inp["target"], inp["draft"], tok, 20, 0.95, inp["seeds"])
        run = lambda: verify_topk(inp["target"], inp["draft"], tok, 20, 0.95, inp["seeds"], ws=ref["ws"], out=ref)
    elif args.case == "verify_t1":
        inp = synth.config_inputs(4, device=dev)
        tok = synth.draft_tokens(inp["draft"], 1, seed=inp["cfg"].seed)
        ref = verify(inp["target"], inp["draft"], tok, 1, inp["seeds"])
        run = lambda: verify(inp["target"], inp["draft"], tok, 1, inp["seeds"], ws=ref["ws"], out=ref)
    elif args.case == "tree_verify":
        c = synth.TREE_CONFIG
        x = synth.tree_inputs(c.B, c.gamma, c.V, c.dtype, seed=c.seed, device=dev, p_match=0.75)
        ref = tree_verify(x["target"], x["parent"], x["token"])
        run = lambda: tree_verify(x["target"], x["parent"], x["token"], ws=ref["ws"], out=ref)
    elif args.case in ("draft_pos", "sampler"):
        V, r = 248320, 256
        if args.case == "sampler":
            c = synth.BRANCH_CONFIG
            x = c.extra
            B = x["n_refs"] * x["n_anchors"]
            inp = synth.branch_inputs(x["n_refs"], x["n_anchors"], c.gamma, c.V, c.r, x["Lmax"], c.dtype, c.seed, dev)
            L, U, Wt, seeds = inp["logits"], inp["U"], inp["Wt"], inp["seeds"]
        else:
            B, G = 512, 2
            L, _ = synth.target_and_draft(B, G - 1, V, "zipf", 0.0, torch.bfloat16, seed=1011, device=dev)
            L = L[:, :G].contiguous()
            U, Wt = synth.markov_weights(V, r, torch.bfloat16, seed=1011, device=dev)
            seeds = synth.seeds_for(B, 1011).to(dev)
        anchor = synth.anchors(B, V, seed=1011).to(dev)
        ref = draft_block(L, anchor, U, Wt, 1, seeds)
        run = lambda: draft_block(L, anchor, U, Wt, 1, seeds, ws=ref["ws"], out=ref)
    elif args.case == "budget":
        g = torch.Generator(device=dev)
        g.manual_seed(1006)
        conf = (0.4 + 0.6 * torch.rand((32, 16), generator=g, device=dev)).contiguous()
        cost = (40.0 + 0.1 * torch.arange(257, device=dev, dtype=torch.float32)).contiguous()
        ref = verify_budget(conf, 256, cost)
        run = lambda: verify_budget(conf, 256, cost, out=ref)
    elif args.case == "draft_topk":
        inp = synth.config_inputs(4, device=dev)
        ref = draft_block_topk(inp["draft"], inp["anchor"], inp["U"], inp["Wt"], 20, 0.95, inp["seeds"])
        run = lambda: draft_block_topk(inp["draft"], inp["anchor"], inp["U"], inp["Wt"], 20, 0.95, inp["seeds"],
                                       ws=ref["ws"], out=ref)
    else:
        c = synth.CONFIGS[5]
        n_branches = 64
        t, d = synth.e2etv_rows(n_branches, c.gamma, c.V, c.draft_sigma, c.dtype, c.seed, dev)
        ref = e2etv(t, d, n_branches, c.gamma)
        run = lambda: e2etv(t, d, n_branches, c.gamma, ws=ref["ws"], out=ref)
    torch.cuda.synchronize()
    for _ in range(args.launches):
        run()
    torch.cuda.synchronize()
    print(f"{args.case}: {args.launches} launches done")


if __name__ == "__main__":
    main()
