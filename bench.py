#!/usr/bin/env python3
"""Benchmark of the block-speculative-decoding hot path on GB300.

Headline workload (one step = the whole path of a decode step at B=1):
    spec_draft_block (gamma=15, V=248320, rank-256 Markov bias, T=0)
  + spec_verify      (16 target rows, T=0)
timed as spec_draft_verify, the one-call form of the two (the verify kernel is the
programmatic dependent of the draft kernel, so its target-row pass overlaps the
draft), in one CUDA graph; the two calls made separately are timed too (same
outputs); on seeded synthetic logits (verify_spec_draft_gb300/synth.py,
configuration 3).
Metric: verify rows per second over the whole draft+verify step, with the step's
microseconds alongside, and the dominant kernel's fraction of the HBM roofline.

Secondary numbers measured in the same run (not separate bench lines):
    verify T=1 at B=32, gamma=7, V=248320 (configuration 4), rows/s and HBM fraction;
    E2E-TV over 16x64x7 rows, V=248320 (configuration 5), tokens/s and HBM fraction.

Usage:  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
For N > 1 run it under torch.distributed.run; every rank processes its own
independent requests (weak scaling, no collective on the data path).
"""

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "verify rows/s (V-wide) + % HBM roofline; draft+verify µs @B1 γ15 V248320"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
L2_FLUSH_BYTES = 512 << 20
# DRAM bytes (read + written) per launch of draft_tc_kernel<1, bf16> on the headline
# workload, from an ncu capture (ncu --set full, one launch); None once the kernel
# changes, until it is captured again
DRAFT_TC_TRAFFIC_BYTES = 138_496_512


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-secondary", action="store_true", help="skip the configuration 4 and 5 numbers")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    return ap.parse_args()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# ---------------------------------------------------------------------------------
# clocks sampled while the GPU works
# ---------------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.samples = []
        self.proc = None
        self.thread = None
        self.active = False

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 8:
                self.samples.append((self.active, parts))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=2)

    def summary(self):
        busy = [p for a, p in self.samples if a] or [p for _, p in self.samples]
        if not busy:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(p[0]) for p in busy if num(p[0]) is not None]
        smax = [num(p[1]) for p in busy if num(p[1]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for p in busy for i in range(4) if p[4 + i].lower().startswith("active")})
        power = [num(p[2]) for p in busy if num(p[2]) is not None]
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(busy), "power_w_max": max(power) if power else None}


# ---------------------------------------------------------------------------------
# our implementation
# ---------------------------------------------------------------------------------
def capture(fn, torch):
    """CUDA-graph capture of a call sequence; falls back to eager replay."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    try:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, capture_error_mode="thread_local"):
            fn()
        torch.cuda.synchronize()
        return g.replay, True
    except Exception as e:  # noqa: BLE001
        print(f"[bench] graph capture failed ({e}); timing eager calls", file=sys.stderr)
        torch.cuda.synchronize()
        return fn, False


def time_steps(torch, replay, steps, flush=None, parts=None):
    """Per-step CUDA-event times (ms) on the current stream.  ``parts`` is a list of
    callables making up the step, each timed on its own; ``flush`` runs between steps
    outside the events."""
    parts = parts or [replay]
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(parts) + 1)] for _ in range(steps)]
    for k in range(steps):
        if flush is not None:
            flush()
        evs[k][0].record()
        for i, p in enumerate(parts):
            p()
            evs[k][i + 1].record()
    torch.cuda.synchronize()
    per_part = [[evs[k][i].elapsed_time(evs[k][i + 1]) for k in range(steps)] for i in range(len(parts))]
    total = [evs[k][0].elapsed_time(evs[k][-1]) for k in range(steps)]
    return total, per_part


def run_ours(args, rank, world, torch, dist):
    from verify_spec_draft_gb300 import shard
    import verify_spec_draft_gb300 as vsd
    from verify_spec_draft_gb300 import synth

    vsd.load()
    dev = torch.device("cuda", torch.cuda.current_device())
    hbm, hbm_kind = peaks()
    sampler = ClockSampler(torch.cuda.current_device())
    sampler.start()

    # ---- headline: configuration 3 (B=1, gamma=15, V=248320, r=256), draft + verify, T=0
    inp = synth.config_inputs(3, device=dev)
    c = inp["cfg"]
    B, G, V, r = c.B, c.gamma, c.V, c.r
    L, tgt, U, Wt, anchor = inp["draft"], inp["target"], inp["U"], inp["Wt"], inp["anchor"]
    ws_d = vsd.workspace(vsd.OP_DRAFT, B, G, V, r, dev)
    ws_v = vsd.workspace(vsd.OP_VERIFY, B, G, V, 0, dev)
    ws_f = vsd.workspace(vsd.OP_DRAFT_VERIFY, B, G, V, r, dev)
    out_d = dict(tokens=torch.empty((B, G), dtype=torch.int32, device=dev),
                 conf=torch.empty((B, G), dtype=torch.float32, device=dev),
                 qtok=torch.empty((B, G), dtype=torch.float32, device=dev),
                 passes=torch.zeros((1,), dtype=torch.int32, device=dev))
    out_v = dict(n=torch.empty((B,), dtype=torch.int32, device=dev),
                 committed=torch.empty((B, G + 1), dtype=torch.int32, device=dev),
                 bonus=torch.empty((B,), dtype=torch.int32, device=dev),
                 near=torch.empty((B,), dtype=torch.int32, device=dev))

    out_f = dict(out_d)
    out_f.update({k: torch.empty_like(v) for k, v in out_d.items()})
    out_f.update({k: torch.empty_like(v) for k, v in out_v.items() if k != "near"})

    def do_fused():
        vsd.draft_verify(L, tgt, anchor, U, Wt, ws=ws_f, out=out_f)

    def do_draft():
        vsd.draft_block(L, anchor, U, Wt, 0, None, ws=ws_d, out=out_d)

    def do_verify():
        vsd.verify(tgt, None, out_d["tokens"], 0, None, ws=ws_v, out=out_v)

    flush_buf = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    def flush():
        flush_buf.zero_()

    def do_step():
        do_draft()
        do_verify()

    # the headline step: spec_draft_verify in one graph (its verify kernel overlaps the
    # draft kernel); then the two calls made separately, and each call alone
    g_fused, graphed_f = capture(do_fused, torch)
    g_step, graphed_s = capture(do_step, torch)
    g_draft, graphed_d = capture(do_draft, torch)
    g_verify, graphed_v = capture(do_verify, torch)
    for _ in range(args.warmup):
        flush()
        g_fused()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    sampler.active = True
    t_wall = time.perf_counter()
    total, _ = time_steps(torch, g_fused, args.steps, flush=flush)
    t_wall = time.perf_counter() - t_wall
    sampler.active = False
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    n_part = max(20, min(args.steps, 200))
    t_two, _ = time_steps(torch, g_step, n_part, flush=flush)
    t_draft, _ = time_steps(torch, g_draft, n_part, flush=flush)
    t_verify, _ = time_steps(torch, g_verify, n_part, flush=flush)
    ms_step = sum(total) / len(total)
    ms_two = sum(t_two) / len(t_two)
    ms_draft = sum(t_draft) / len(t_draft)
    ms_verify = sum(t_verify) / len(t_verify)
    if world > 1:
        ms_step, ms_two, ms_draft, ms_verify = (shard.max_over_ranks(x, dev) for x in (ms_step, ms_two, ms_draft,
                                                                                      ms_verify))
    passes = int(out_f["passes"].item())
    rows = B * (G + 1)
    # algorithmic bytes of one draft launch (the dominant kernel): the draft rows and Wt
    # read once, plus the U rows of the gamma previous tokens; verify: the 16 target rows
    draft_bytes = B * G * V * 2 + V * r * 2 + B * G * r * 2
    verify_bytes = B * (G + 1) * V * 2
    dom_bytes, dom_ms = draft_bytes, ms_draft
    achieved = dom_bytes / (dom_ms * 1e-3) / 1e9
    n_acc = out_f["n"].cpu().tolist()
    assert torch.equal(out_f["tokens"], out_d["tokens"]) and torch.equal(out_f["n"], out_v["n"])

    result = {
        "metric": METRIC,
        "value": rows * world / (ms_step * 1e-3),
        "unit": "rows/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_step,
        "draft_verify_us": ms_step * 1e3,
        "two_call_step_us": ms_two * 1e3,
        "draft_us": ms_draft * 1e3,
        "verify_us": ms_verify * 1e3,
        "note_parts": "draft_verify_us: spec_draft_verify (the headline step); two_call_step_us: spec_draft_block "
                      "then spec_verify in one graph (same outputs); draft_us and verify_us time each call alone",
        "verify_only_rows_per_s": rows / (ms_verify * 1e-3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16 storage, f32 accumulate",
        "data": "synthetic (seeded zipf-skewed logits and N(0,0.02^2) Markov weights, shaped like the pages' workloads)",
        "config": {
            "workload": "latency: draft block + verify, B=1, gamma=15 (block 16), V=248320, r=256, T=0",
            "B": B, "gamma": G, "V": V, "r": r, "temperature": 0,
            "fixed_point_passes": passes,
            "accepted_n": n_acc,
            "cuda_graphs": bool(graphed_f and graphed_s and graphed_d and graphed_v),
            "step": "one CUDA graph of spec_draft_verify: the draft kernel, then the verify kernel as its "
                    "programmatic dependent (its target-row pass overlaps the draft; it waits for the draft "
                    "before reading the tokens)",
            "l2": f"flushed between steps ({L2_FLUSH_BYTES >> 20} MiB write), outside the timed events",
            "parallelism": f"replicas x{world} (independent requests per GPU, no collective)",
        },
        "roofline": {
            "kernel": "spec::draft_tc_kernel",
            "bound": "hbm",
            "achieved": achieved,
            "peak": hbm,
            "peak_kind": hbm_kind,
            "unit": "GB/s",
            "frac": achieved / hbm,
            "frac_of_nominal_8tbs": achieved / NOMINAL_HBM_GBS,
            "algorithmic_bytes_per_launch": dom_bytes,
            # dram__bytes_read.sum + dram__bytes_write.sum of this kernel on this workload,
            # from one ncu capture
            "traffic": DRAFT_TC_TRAFFIC_BYTES,
        },
        "gpu_launches": 2 * args.steps,
        "wall_s_timed_loop": t_wall,
    }

    # ---- end to end through the public API with host buffers (pinned), copies timed
    if not args.no_e2e:
        h_L = L.cpu().pin_memory()
        h_t = tgt.cpu().pin_memory()
        h_a = anchor.cpu().pin_memory()
        d_L, d_t, d_a = torch.empty_like(L), torch.empty_like(tgt), torch.empty_like(anchor)
        h_out = torch.empty((B * (G + 1) + 2 * B + B * G,), dtype=torch.int32).pin_memory()
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        e2e_steps = min(args.steps, 200)

        def e2e_fused():
            # every input copied, then spec_draft_verify
            d_L.copy_(h_L, non_blocking=True)
            d_t.copy_(h_t, non_blocking=True)
            d_a.copy_(h_a, non_blocking=True)
            vsd.draft_verify(d_L, d_t, d_a, U, Wt, ws=ws_f, out=out_f)
            packed = torch.cat([out_f["n"], out_f["committed"].flatten(), out_f["bonus"], out_f["tokens"].flatten()])
            h_out.copy_(packed, non_blocking=True)

        copy_s = torch.cuda.Stream()
        # the drafter rows and the anchors in one pinned buffer (the anchors after the rows,
        # 4-byte aligned), so one copy brings both; device views of the same layout
        nb_l = h_L.numel() * h_L.element_size()
        h_la = torch.empty((nb_l + 4 * B,), dtype=torch.uint8).pin_memory()
        h_la[:nb_l].view(h_L.dtype).copy_(h_L.flatten())
        h_la[nb_l:].view(torch.int32).copy_(h_a)
        d_la = torch.empty_like(h_la, device=dev)
        d_L2 = d_la[:nb_l].view(h_L.dtype).view(h_L.shape)
        d_a2 = d_la[nb_l:].view(torch.int32)
        # the results the host reads, written by the calls into one int32 buffer (views in
        # the packed order: n, committed, bonus, tokens), so one copy brings them back
        e2e_i32 = torch.empty((h_out.numel(),), dtype=torch.int32, device=dev)
        o0, o1, o2 = B, B + B * (G + 1), B + B * (G + 1) + B
        out_de = dict(tokens=e2e_i32[o2:].view(B, G), conf=torch.empty_like(out_d["conf"]),
                      qtok=torch.empty_like(out_d["qtok"]), passes=torch.zeros_like(out_d["passes"]))
        out_ve = dict(n=e2e_i32[:o0], committed=e2e_i32[o0:o1].view(B, G + 1), bonus=e2e_i32[o1:o2],
                      near=torch.empty_like(out_v["near"]))

        def e2e_overlap():
            # the target rows copied on a second stream while spec_draft_block runs on the
            # drafter rows; spec_verify once both are in
            main = torch.cuda.current_stream()
            copy_s.wait_stream(main)   # after the step's start (and the last step's reads)
            with torch.cuda.stream(copy_s):
                d_t.copy_(h_t, non_blocking=True)
            d_la.copy_(h_la, non_blocking=True)
            vsd.draft_block(d_L2, d_a2, U, Wt, 0, None, ws=ws_d, out=out_de)
            main.wait_stream(copy_s)
            vsd.verify(d_t, None, out_de["tokens"], 0, None, ws=ws_v, out=out_ve)
            h_out.copy_(e2e_i32, non_blocking=True)

        def time_e2e(step_fn):
            for _ in range(5):
                flush()
                step_fn()
            torch.cuda.synchronize()
            times = []
            for _ in range(e2e_steps):
                flush()
                ev[0].record()
                step_fn()
                ev[1].record()
                ev[1].synchronize()
                times.append(ev[0].elapsed_time(ev[1]))
            return sum(times) / len(times)

        ms_fused = time_e2e(e2e_fused)
        ref_out = h_out.clone()
        ms_e2e = time_e2e(e2e_overlap)
        assert torch.equal(h_out, ref_out), "the two end-to-end paths disagree"
        result["e2e"] = {"value": rows * world / (ms_e2e * 1e-3), "unit": "rows/s", "us_per_step": ms_e2e * 1e3,
                         "h2d_bytes_per_step": h_la.numel() + h_t.numel() * 2,
                         "d2h_bytes_per_step": h_out.numel() * 4,
                         "path": "pinned host buffers -> cudaMemcpyAsync (target rows on a second stream, "
                                 "overlapping spec_draft_block) -> spec_verify -> results (written into one "
                                 "buffer) to pinned host, eager C-ABI calls (Markov weights resident)",
                         "us_per_step_copies_first": ms_fused * 1e3,
                         "note": "us_per_step_copies_first: every input copied first, then one spec_draft_verify call"}
    del flush_buf

    # ---- secondary: verify T=1 at B=32 (configuration 4) and E2E-TV (configuration 5)
    if not args.no_secondary:
        result["secondary"] = secondary(args, torch, vsd, synth, dev, hbm, hbm_kind, sampler, rank, world)

    sampler.stop()
    result["clocks"] = sampler.summary()
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(inp, budget_s=20.0)
    result["summary"] = summary(result)
    return result


def summary(result):
    """The numbers of every workload in a few hundred characters, last on the line (so
    that a tail of the output still holds all of them)."""
    r3 = lambda x: None if x is None else float(f"{x:.4g}")
    out = {"draft_verify_us": r3(result["draft_verify_us"]), "draft_us": r3(result["draft_us"]),
           "draft_frac": r3(result["roofline"]["frac"])}
    sec = result.get("secondary", {})
    for key, name, scale, unit in (("verify_t1_b32", "verify_t1_b32", 1e-6, "Mrows_s"),
                                   ("verify_t1_topk_b32", "verify_topk_b32", 1e-6, "Mrows_s"),
                                   ("e2etv_cfg5", "e2etv", 1e-6, "Mtok_s"),
                                   ("tree_verify_t0", "tree_verify", 1e-6, "Mrows_s"),
                                   ("draft_t1_b32", "draft_t1_b32", 1e-6, "Mrows_s"),
                                   ("draft_t1_topk_b32", "draft_topk_b32", 1e-6, "Mrows_s"),
                                   ("anchor_branches", "sampler", 1e-3, "kbranch_s")):
        v = sec.get(key)
        if not v:
            continue
        t = v.get("us_per_step")
        out[name + ("_us" if t is not None else "_ms")] = r3(t if t is not None else v.get("ms_per_step"))
        out[f"{name}_{unit}"] = r3(v["value"] * scale)
        out[name + "_frac"] = r3(v["roofline"].get("frac"))
    cb = result.get("cpu_baseline", {})
    for k, v in cb.get("configs", {}).items():
        out["oracle_" + k] = [r3(v.get("value_1core")), r3(v.get("value_all")), v.get("unit")]
    return out


def secondary(args, torch, vsd, synth, dev, hbm, hbm_kind, sampler, rank=0, world=1):
    from verify_spec_draft_gb300 import shard
    out = {}
    steps = max(5, min(args.steps, 50))
    # configuration 4: verify T=1, B=32, gamma=7, V=248320; inputs 238 MB > L2
    inp = synth.config_inputs(4, device=dev)
    c = inp["cfg"]
    B, G, V = c.B, c.gamma, c.V
    t, d, seeds = inp["target"], inp["draft"], inp["seeds"]
    tok = synth.draft_tokens(d, 1, seed=c.seed)
    ws = vsd.workspace(vsd.OP_VERIFY, B, G, V, 0, dev)
    o = dict(n=torch.empty((B,), dtype=torch.int32, device=dev),
             committed=torch.empty((B, G + 1), dtype=torch.int32, device=dev),
             bonus=torch.empty((B,), dtype=torch.int32, device=dev),
             near=torch.empty((B,), dtype=torch.int32, device=dev))
    fn, graphed = capture(lambda: vsd.verify(t, d, tok, 1, seeds, ws=ws, out=o), torch)
    for _ in range(3):
        fn()
    torch.cuda.synchronize()
    sampler.active = True
    total, _ = time_steps(torch, fn, steps)
    sampler.active = False
    ms = sum(total) / len(total)
    rows = B * (G + 1)
    byts = (B * (G + 1) + B * G) * V * 2
    ach = byts / (ms * 1e-3) / 1e9
    out["verify_t1_b32"] = {
        "workload": "verify T=1, B=32, gamma=7, V=248320, bf16, per-request seeds",
        "value": rows / (ms * 1e-3), "unit": "rows/s", "us_per_step": ms * 1e3, "cuda_graphs": graphed,
        "accepted_mean_n": float(o["n"].float().mean().item()),
        "roofline": {"bound": "hbm", "achieved": ach, "peak": hbm, "peak_kind": hbm_kind, "unit": "GB/s",
                     "frac": ach / hbm, "frac_of_nominal_8tbs": ach / NOMINAL_HBM_GBS,
                     "algorithmic_bytes_per_launch": byts},
        "gpu_launches": 2 * steps,
    }
    # the same rows verified against top-k / top-p filtered distributions (the DSpine
    # card's sampling setting: top_k 20, top_p 0.95)
    k, top_p = 20, 0.95
    otk = vsd.verify_topk(t, d, tok, k, top_p, seeds)
    fn, graphed = capture(lambda: vsd.verify_topk(t, d, tok, k, top_p, seeds, ws=otk["ws"], out=otk), torch)
    for _ in range(3):
        fn()
    torch.cuda.synchronize()
    sampler.active = True
    total, _ = time_steps(torch, fn, steps)
    sampler.active = False
    ms = sum(total) / len(total)
    ach = byts / (ms * 1e-3) / 1e9
    out["verify_t1_topk_b32"] = {
        "workload": "verify T=1 with top_k 20, top_p 0.95, B=32, gamma=7, V=248320, bf16, per-request seeds",
        "value": rows / (ms * 1e-3), "unit": "rows/s", "us_per_step": ms * 1e3, "cuda_graphs": graphed,
        "accepted_mean_n": float(otk["n"].float().mean().item()),
        "roofline": {"bound": "hbm", "achieved": ach, "peak": hbm, "peak_kind": hbm_kind, "unit": "GB/s",
                     "frac": ach / hbm, "frac_of_nominal_8tbs": ach / NOMINAL_HBM_GBS,
                     "algorithmic_bytes_per_launch": byts},
        "gpu_launches": 3 * steps,
    }
    del t, d, inp
    torch.cuda.empty_cache()

    # draft trees: 32 trees x 64 nodes over V = 248320 bf16 rows (2080 rows, 1.03 GB > L2):
    # T=0 verification of every node, then the EAGLE-2 step of keeping the top 24 nodes
    # by path product and verifying only those
    tc = synth.TREE_CONFIG
    x = synth.tree_inputs(tc.B, tc.gamma, tc.V, tc.dtype, seed=tc.seed, device=dev, p_match=0.75)
    T_, n_ = tc.B, tc.gamma
    ws_t = vsd.workspace(vsd.OP_TREE_VERIFY, T_, n_, tc.V, 0, dev)
    ot_ = vsd.tree_verify(x["target"], x["parent"], x["token"], ws=ws_t)
    fn, graphed = capture(lambda: vsd.tree_verify(x["target"], x["parent"], x["token"], ws=ws_t, out=ot_), torch)
    for _ in range(3):
        fn()
    torch.cuda.synchronize()
    sampler.active = True
    total, _ = time_steps(torch, fn, steps)
    sampler.active = False
    ms = sum(total) / len(total)
    rows = T_ * (n_ + 1)
    byts = rows * tc.V * 2
    ach = byts / (ms * 1e-3) / 1e9
    out["tree_verify_t0"] = {
        "workload": "tree verify T=0: 32 trees x 64 nodes, V=248320 bf16 (root + 64 node rows per tree)",
        "value": rows / (ms * 1e-3), "unit": "rows/s", "us_per_step": ms * 1e3, "cuda_graphs": graphed,
        "accepted_mean_n": float(ot_["n"].float().mean().item()),
        "roofline": {"bound": "hbm", "achieved": ach, "peak": hbm, "peak_kind": hbm_kind, "unit": "GB/s",
                     "frac": ach / hbm, "frac_of_nominal_8tbs": ach / NOMINAL_HBM_GBS,
                     "algorithmic_bytes_per_launch": byts},
        "gpu_launches": steps,
    }
    m_ = 24
    os_ = vsd.tree_select(x["parent"], x["conf"], m_)
    op_ = vsd.tree_verify(x["target"], x["parent"], x["token"], keep=os_["keep"], ws=ws_t)

    def select_verify():
        vsd.tree_select(x["parent"], x["conf"], m_, out=os_)
        vsd.tree_verify(x["target"], x["parent"], x["token"], keep=os_["keep"], ws=ws_t, out=op_)

    fn, graphed = capture(select_verify, torch)
    for _ in range(3):
        fn()
    torch.cuda.synchronize()
    flush_buf = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    sampler.active = True
    total, _ = time_steps(torch, fn, steps, flush=lambda: flush_buf.zero_())
    sampler.active = False
    del flush_buf
    ms = sum(total) / len(total)
    rows = T_ * (m_ + 1)
    byts = rows * tc.V * 2
    ach = byts / (ms * 1e-3) / 1e9
    out["tree_select_verify_m24"] = {
        "workload": "EAGLE-2 step: top-24 of 64 nodes by path product (32 trees), then T=0 verification of the "
                    "kept nodes, V=248320 bf16 (L2 flushed)",
        "value": rows / (ms * 1e-3), "unit": "rows/s", "us_per_step": ms * 1e3, "cuda_graphs": graphed,
        "accepted_mean_n": float(op_["n"].float().mean().item()),
        "roofline": {"bound": "hbm", "achieved": ach, "peak": hbm, "peak_kind": hbm_kind, "unit": "GB/s",
                     "frac": ach / hbm, "frac_of_nominal_8tbs": ach / NOMINAL_HBM_GBS,
                     "algorithmic_bytes_per_launch": byts},
        "gpu_launches": 2 * steps,
    }
    del x, ws_t, ot_, os_, op_
    torch.cuda.empty_cache()

    # configuration 5: E2E-TV, 16 x 64 x 7 rows, V=248320; 7.1 GB of inputs.  With N > 1
    # ranks the 1024 branches are split across them (strong scaling for this line): each
    # rank runs its shard and the loss takes one scalar all-reduce per step
    inp = synth.config_inputs(5, device=dev)
    c = inp["cfg"]
    N_all, Wb, V = c.B, c.gamma, c.V
    b0, N = shard.shard_range(N_all, rank, world)
    t = inp["target"][b0 * Wb:(b0 + N) * Wb]
    d = inp["draft"][b0 * Wb:(b0 + N) * Wb]
    ws = vsd.workspace(vsd.OP_E2ETV, N, Wb, V, 0, dev)
    R = N * Wb
    o = dict(a=torch.empty((R,), dtype=torch.float32, device=dev),
             surv=torch.empty((R,), dtype=torch.float32, device=dev),
             loss=torch.empty((1,), dtype=torch.float32, device=dev),
             grad=torch.empty((R, V), dtype=torch.bfloat16, device=dev))
    if world == 1:
        fn, graphed = capture(lambda: vsd.e2etv(t, d, N, Wb, ws=ws, out=o), torch)
    else:
        o["msum"] = o["loss"]

        def sharded():
            r = shard.e2etv_rank(t, d, N, Wb, N_all, ws=ws, out=o)
            o["loss_all"] = r["loss"]

        fn, graphed = sharded, False
    for _ in range(3):
        fn()
    torch.cuda.synchronize()
    steps5 = max(5, min(args.steps, 30))
    sampler.active = True
    total, _ = time_steps(torch, fn, steps5)
    sampler.active = False
    ms = sum(total) / len(total)
    if world > 1:
        ms = shard.max_over_ranks(ms, dev)
    byts = 3 * R * V * 2
    ach = byts / (ms * 1e-3) / 1e9
    out["e2etv_cfg5"] = {
        "workload": "E2E-TV, 16 refs x 64 anchors x Wb=7 = 7168 rows, V=248320, bf16 in/out",
        "value": N_all * Wb / (ms * 1e-3), "unit": "supervised tokens/s", "ms_per_step": ms, "cuda_graphs": graphed,
        "loss": float((o["loss_all"] if world > 1 else o["loss"]).item()),
        "scaling": "strong" if world > 1 else None,
        "branches_per_rank": N,
        "roofline": {"bound": "hbm", "achieved": ach, "peak": hbm, "peak_kind": hbm_kind, "unit": "GB/s",
                     "frac": ach / hbm, "frac_of_nominal_8tbs": ach / NOMINAL_HBM_GBS,
                     "algorithmic_bytes_per_launch": byts},
        "gpu_launches": steps5,
    }
    del t, d, inp, o
    torch.cuda.empty_cache()

    # configuration 4's draft: B=32, gamma=7, V=248320, r=256 bf16, T=1 (224 rows, the
    # tcgen05 kernel with two M tiles); 111 MB of drafter rows and 127 MB of Wt
    inp = synth.config_inputs(4, device=dev)
    c = inp["cfg"]
    B, G, V = c.B, c.gamma, c.V
    L4, U4, Wt4, a4, s4 = inp["draft"], inp["U"], inp["Wt"], inp["anchor"], inp["seeds"]
    ws4 = vsd.workspace(vsd.OP_DRAFT, B, G, V, c.r, dev)
    o4 = vsd.draft_block(L4, a4, U4, Wt4, 1, s4, ws=ws4)
    fn, graphed = capture(lambda: vsd.draft_block(L4, a4, U4, Wt4, 1, s4, ws=ws4, out=o4), torch)
    for _ in range(3):
        fn()
    torch.cuda.synchronize()
    flush_buf = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    sampler.active = True
    total, _ = time_steps(torch, fn, steps, flush=lambda: flush_buf.zero_())
    sampler.active = False
    ms = sum(total) / len(total)
    passes = int(o4["passes"].item())
    byts = B * G * V * 2 + passes * V * c.r * 2 + B * G * c.r * 2
    ach = byts / (ms * 1e-3) / 1e9
    out["draft_t1_b32"] = {
        "workload": "draft block T=1, B=32, gamma=7, V=248320, r=256 bf16, per-request seeds (L2 flushed)",
        "value": B * G / (ms * 1e-3), "unit": "rows/s", "us_per_step": ms * 1e3, "cuda_graphs": graphed,
        "passes": passes,
        "roofline": {"bound": "hbm", "achieved": ach, "peak": hbm, "peak_kind": hbm_kind, "unit": "GB/s",
                     "frac": ach / hbm, "frac_of_nominal_8tbs": ach / NOMINAL_HBM_GBS,
                     "algorithmic_bytes_per_launch": byts,
                     "note": "drafter rows once, W once per biased pass; pass 0 and the biased pass both read the rows"},
        "gpu_launches": steps,
    }
    # the same draft with the DSpine card's filtered draws (top_k 20, top_p 0.95): the chain
    # position by position, the weights read once per position
    wsk = vsd.workspace(vsd.OP_DRAFT_TOPK, B, G, V, c.r, dev)
    ok_ = vsd.draft_block_topk(L4, a4, U4, Wt4, 20, 0.95, s4, ws=wsk)
    fn, graphed = capture(lambda: vsd.draft_block_topk(L4, a4, U4, Wt4, 20, 0.95, s4, ws=wsk, out=ok_), torch)
    for _ in range(3):
        fn()
    torch.cuda.synchronize()
    sampler.active = True
    total, _ = time_steps(torch, fn, steps, flush=lambda: flush_buf.zero_())
    sampler.active = False
    ms = sum(total) / len(total)
    byts = B * G * V * 2 + G * V * c.r * 2
    ach = byts / (ms * 1e-3) / 1e9
    out["draft_t1_topk_b32"] = {
        "workload": "draft block T=1 with top_k 20, top_p 0.95, B=32, gamma=7, V=248320, r=256 bf16 (L2 flushed)",
        "value": B * G / (ms * 1e-3), "unit": "rows/s", "us_per_step": ms * 1e3, "cuda_graphs": graphed,
        "roofline": {"bound": "hbm", "achieved": ach, "peak": hbm, "peak_kind": hbm_kind, "unit": "GB/s",
                     "frac": ach / hbm, "frac_of_nominal_8tbs": ach / NOMINAL_HBM_GBS,
                     "algorithmic_bytes_per_launch": byts,
                     "note": "drafter rows once and W once per position (the chain is walked position by position)"},
        "gpu_launches": 2 * G * steps,
    }
    del inp, L4, U4, Wt4, o4, ws4, flush_buf, wsk, ok_
    torch.cuda.empty_cache()

    # the SpecOPD anchor-branch sampler: 16 references x 64 anchors, W = 7, V = 248320,
    # r = 256, T = 1: the plan, then the draft block over the 1024 branches (3.56 GB of
    # drafter rows, more than L2), walked position by position on the tensor cores
    c = synth.BRANCH_CONFIG
    x = c.extra
    inp = synth.branch_inputs(x["n_refs"], x["n_anchors"], c.gamma, c.V, c.r, x["Lmax"], c.dtype, c.seed, dev)
    nb = x["n_refs"] * x["n_anchors"]
    op = vsd.branch_plan(inp["trunk"], inp["lengths"], x["n_anchors"], c.gamma, c.seed)
    anchor = op["anchor_tok"].view(-1)
    wsd = vsd.workspace(vsd.OP_DRAFT, nb, c.gamma, c.V, c.r, dev)
    ob = vsd.draft_block(inp["logits"], anchor, inp["U"], inp["Wt"], 1, inp["seeds"], ws=wsd)

    def sampler_step():
        vsd.branch_plan(inp["trunk"], inp["lengths"], x["n_anchors"], c.gamma, c.seed, ws=op["ws"], out=op)
        vsd.draft_block(inp["logits"], anchor, inp["U"], inp["Wt"], 1, inp["seeds"], ws=wsd, out=ob)

    fn, graphed = capture(sampler_step, torch)
    for _ in range(3):
        fn()
    torch.cuda.synchronize()
    steps6 = max(5, min(args.steps, 30))
    sampler.active = True
    total, _ = time_steps(torch, fn, steps6)
    sampler.active = False
    ms = sum(total) / len(total)
    passes = int(ob["passes"].item())
    # more than 256 rows take the position-by-position path: per slice of at most 1024
    # branches a gather, then a tiles kernel and a draw per position (passes = gamma:
    # W read once per position)
    launches = 1 + ((nb + 1023) // 1024) * (1 + 2 * c.gamma)
    # algorithmic: the drafter rows once, W once per pass over the positions, the outputs
    byts = nb * c.gamma * c.V * 2 + passes * c.V * c.r * 2
    ach = byts / (ms * 1e-3) / 1e9
    out["anchor_branches"] = {
        "workload": "SpecOPD anchor-branch sampler: 16 refs x 4096 tokens, 64 anchors each, W=7, V=248320, "
                    "r=256 bf16, T=1 (plan + draft block over 1024 branches)",
        "value": nb / (ms * 1e-3), "unit": "branches/s", "ms_per_step": ms, "cuda_graphs": graphed,
        "passes": passes, "draft_launches_per_step": launches - 1, "path": "position by position (tcgen05)",
        "roofline": {"bound": "hbm", "achieved": ach, "peak": hbm, "peak_kind": hbm_kind, "unit": "GB/s",
                     "frac": ach / hbm, "frac_of_nominal_8tbs": ach / NOMINAL_HBM_GBS,
                     "algorithmic_bytes_per_launch": byts,
                     "note": "per step: the drafter rows once and W once per position"},
        "gpu_launches": launches * steps6,
    }
    del inp, ob, wsd
    torch.cuda.empty_cache()

    # the verify budget across a batch: B=32 requests, gamma=16 confidences in [0.4, 1),
    # budget 256 positions, a linear cost curve; a few KB of input, L2 flushed between
    # steps
    g = torch.Generator(device=dev)
    g.manual_seed(1006)
    conf = (0.4 + 0.6 * torch.rand((32, 16), generator=g, device=dev)).contiguous()
    budget = 256
    cost = (40.0 + 0.1 * torch.arange(budget + 1, device=dev, dtype=torch.float32)).contiguous()
    ob = dict(gamma=torch.empty((32,), dtype=torch.int32, device=dev),
              expected=torch.empty((1,), dtype=torch.float32, device=dev))
    fn, graphed = capture(lambda: vsd.verify_budget(conf, budget, cost, out=ob), torch)
    flush_buf = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    for _ in range(3):
        fn()
    torch.cuda.synchronize()
    total, _ = time_steps(torch, fn, steps, flush=lambda: flush_buf.zero_())
    ms = sum(total) / len(total)
    out["verify_budget_b32_g16"] = {
        "workload": "verify budget: B=32, gamma=16 confidences, budget 256, linear cost curve",
        "value": ms * 1e3, "unit": "us/call", "higher_is_better": False, "cuda_graphs": graphed,
        "verified_positions": int(ob["gamma"].sum().item()), "expected_committed": float(ob["expected"].item()),
        "roofline": {"bound": "latency", "note": "2 KB of confidences; one CTA sorts 512 candidates"},
        "gpu_launches": steps,
    }
    del flush_buf
    torch.cuda.empty_cache()
    return out


# ---------------------------------------------------------------------------------
# CPU baseline: the float64 oracle, as it stands
# ---------------------------------------------------------------------------------
def oracle_step(L, anchor, U, Wt, tgt):
    from oracle import draft as od, verify as ov
    d = od.draft_block(L, anchor, U, Wt, 0, [0])
    ov.verify(tgt, None, d["tokens"], 0, None)


def blas_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 1) for i in threadpool_info() if i.get("user_api") == "blas"]
        return max(n) if n else 1
    except Exception:
        return int(os.environ.get("OPENBLAS_NUM_THREADS", os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1)))


def cpu_model():
    """The host CPU as /proc/cpuinfo names it (Arm cores list implementer and part)."""
    arm_parts = {"0xd4f": "Arm Neoverse-V2", "0xd40": "Arm Neoverse-V1", "0xd0c": "Arm Neoverse-N1"}
    try:
        with open("/proc/cpuinfo") as f:
            info = f.read()
    except OSError:
        return None
    for line in info.splitlines():
        if line.lower().startswith("model name"):
            return line.split(":", 1)[1].strip()
    for line in info.splitlines():
        if line.startswith("CPU part"):
            part = line.split(":", 1)[1].strip()
            return arm_parts.get(part, f"Arm CPU part {part}")
    return None


# Oracle work units for the CPU baseline, run in worker processes started with "spawn"
# (the parent has initialised CUDA) and BLAS limited to one thread per process.  Inputs
# are generated on the host with the same recipe as the GPU run (synthetic, seeded;
# the host generator draws other numbers than the CUDA one, with the same shapes and
# distributions).  Returns (seconds spent in the oracle, units done).
def _oracle_work(kind, units, seed):
    import numpy as np
    import torch
    from verify_spec_draft_gb300 import synth
    if kind == "cfg3":       # draft + verify steps, B=1, gamma=15, V=248320, r=256
        inp = synth.config_inputs(3, device="cpu")
        L = inp["draft"].double().numpy()
        tgt = inp["target"].double().numpy()
        U = inp["U"].double().numpy()
        Wt = inp["Wt"].double().numpy()
        anchor = inp["anchor"].numpy()
        t0 = time.perf_counter()
        for _ in range(units):
            oracle_step(L, anchor, U, Wt, tgt)
        return time.perf_counter() - t0, units * 16
    if kind == "cfg4":       # verify T=1 of `units` requests, gamma=7, V=248320, Zipf rows
        from oracle import verify as ov
        t, d = synth.target_and_draft(units, 7, 248320, "zipf", 0.9, torch.bfloat16, seed=seed)
        tok = synth.draft_tokens(d, 1, seed=seed)
        T, D, X = t.double().numpy(), d.double().numpy(), tok.numpy()
        seeds = np.arange(units, dtype=np.uint64)
        t0 = time.perf_counter()
        ov.verify(T, D, X, 1, seeds)
        return time.perf_counter() - t0, units * 8
    if kind == "cfg5":       # E2E-TV with the gradient over `units` branches of 7 rows
        from oracle import e2etv as oe
        t, d = synth.e2etv_rows(units, 7, 248320, 1.0, seed=seed)
        T, D = t.double().numpy(), d.double().numpy()
        t0 = time.perf_counter()
        oe.e2etv(T, D, units, 7)
        return time.perf_counter() - t0, units * 7
    raise ValueError(kind)


def _timed_pool(kind, units, workers):
    """Wall time of `workers` spawn processes doing `units` each, all in parallel; the
    oracle time is the slowest worker's (set-up excluded)."""
    import multiprocessing as mp
    from concurrent.futures import ProcessPoolExecutor
    saved = {k: os.environ.get(k) for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")}
    for k in saved:
        os.environ[k] = "1"
    try:
        with ProcessPoolExecutor(max_workers=workers, mp_context=mp.get_context("spawn")) as ex:
            res = list(ex.map(_oracle_work, [kind] * workers, [units] * workers, range(workers)))
    finally:
        for k, v in saved.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
    return max(r[0] for r in res), sum(r[1] for r in res)


def cpu_baseline(inp, budget_s=20.0):
    c = inp["cfg"]
    L = inp["draft"].double().cpu().numpy()
    tgt = inp["target"].double().cpu().numpy()
    U = inp["U"].double().cpu().numpy()
    Wt = inp["Wt"].double().cpu().numpy()
    anchor = inp["anchor"].cpu().numpy()
    done, t0 = 0, time.perf_counter()
    while True:
        oracle_step(L, anchor, U, Wt, tgt)
        done += 1
        el = time.perf_counter() - t0
        if el >= budget_s or done >= 20:
            break
    rows = done * c.B * (c.gamma + 1)
    out = {"value": rows / el, "unit": "rows/s", "cores": blas_threads(), "kind": "oracle",
           "sample": f"{done} full draft+verify steps of the headline workload (float64 numpy oracle, "
                     f"{el:.1f} s)", "host_cpus": os.cpu_count(), "nproc": os.cpu_count(), "cpu_model": cpu_model()}
    # every configuration's oracle on one core and on all cores (one process per core,
    # independent requests / branches / steps in parallel), units as the GPU's
    nproc = os.cpu_count() or 1
    # (name, work, units on one core, units per process on all cores, process cap, unit);
    # configuration 3 holds 1 GB of float64 weights per process, hence its cap
    plan = (("cfg3_draft_verify", "cfg3", 6, 3, 8, "rows/s"), ("cfg4_verify_t1", "cfg4", 256, 32, nproc, "rows/s"),
            ("cfg5_e2etv", "cfg5", 96, 24, nproc, "tokens/s"))
    configs = {}
    try:
        for name, kind, n1, nall, cap, unit in plan:
            procs = max(1, min(nproc, cap))
            t1, u1 = _timed_pool(kind, n1, 1)
            ta, ua = _timed_pool(kind, nall, procs)
            configs[name] = {"value_1core": u1 / t1, "value_all": ua / ta, "unit": unit, "cores_all": procs,
                             "sample": f"1 core: {u1} units in {t1:.1f} s; {procs} processes x {nall} work items "
                                       f"each in {ta:.1f} s (BLAS 1 thread per process)"}
    except Exception as e:  # noqa: BLE001
        configs["error"] = {"unit": None, "note": f"{type(e).__name__}: {e}"[:200]}
    out["configs"] = configs
    return out


def run_reference(args, rank, world):
    """The oracle timed on the host cores on the headline workload (bounded sample)."""
    import torch
    from verify_spec_draft_gb300 import synth
    inp = synth.config_inputs(3, device="cpu")
    c = inp["cfg"]
    L = inp["draft"].double().numpy()
    tgt = inp["target"].double().numpy()
    U = inp["U"].double().numpy()
    Wt = inp["Wt"].double().numpy()
    anchor = inp["anchor"].numpy()
    w = min(args.warmup, 1)
    for _ in range(w):
        oracle_step(L, anchor, U, Wt, tgt)
    budget = 90.0
    done, t0 = 0, time.perf_counter()
    while done < args.steps:
        oracle_step(L, anchor, U, Wt, tgt)
        done += 1
        if time.perf_counter() - t0 > budget:
            break
    el = time.perf_counter() - t0
    rows = done * c.B * (c.gamma + 1)
    v = rows / el
    cores = blas_threads()
    return {"impl": "reference", "metric": METRIC, "value": v, "unit": "rows/s", "n_gpus": world,
            "steps": done, "warmup": w, "ms_per_step": el / done * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": "latency: draft block + verify, B=1, gamma=15, V=248320, r=256, T=0",
                       "B": c.B, "gamma": c.gamma, "V": c.V, "r": c.r},
            "cpu_baseline": {"value": v, "unit": "rows/s", "cores": cores, "kind": "oracle",
                             "sample": f"{done} of {args.steps} requested steps (capped at {budget:.0f} s)"},
            "e2e": {"value": v, "unit": "rows/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    args = parse()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args, rank, world)))
        return
    import torch
    dist = None
    if world > 1:
        import torch.distributed as dist
        local = int(os.environ.get("LOCAL_RANK", "0"))
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device (the library has no CPU path)")
    res = run_ours(args, rank, world, torch, dist)
    if rank == 0:
        print(json.dumps(res))
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
