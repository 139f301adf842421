"""Benchmark of the token-tree verification step on GB300.

A step is the whole hot path over one batch: tv_tree_build ->
tv_tree_attention_verify -> tv_accept_commit (greedy accept + KV commit with
block release), after the block-table refill a serving loop's allocator does.

The headline workload (config 5) is the Llama-3-8B attention geometry, batch
64 ragged, prompts log-uniform in [4096, 32768], random EAGLE-style trees of
16-128 nodes (+ root), run as eight evolving steps: each step commits the
accepted path, releases blocks past the new end, the host allocator hands the
next tree's slots out of the free list, and the next tree is verified at
P + 1 + a. The eight steps are generated once, then replayed in order; the
timed steps cycle through them. Configs 2, 3 and 4 are measured as one
verification step each (`sub_workloads`). ``--config C`` makes config C the
headline instead.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--config C]

Under torchrun every rank runs its own batch (requests are independent: no
data-path collective); rank 0 prints one JSON line. ``--impl reference`` times
the CPU oracle on the host cores instead.
"""

from __future__ import annotations

import argparse
import hashlib
import re
import json
import math
import multiprocessing as mp
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "tree-verify tokens/s at 1 GB300; attention HBM GB/s & % roofline per step"
UNIT = "tokens/s"
L2_FLUSH_BYTES = 512 << 20
MULTISTEP = 8                 # config 5: verification steps of one request cycle
SUB_CONFIGS = (2, 3, 4)
ATTN_SOURCES = ("attention_tc.cu", "tv_sm100.cuh", "tv_common.cuh")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=80,
                    help="timed verification steps (config 5: the eight evolving steps in turn)")
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", type=int, default=5)
    ap.add_argument("--attn-iters", type=int, default=30,
                    help="timed launches of each step's attention call")
    ap.add_argument("--sub-iters", type=int, default=200,
                    help="timed steps of each of the other workloads (configs 2-4)")
    ap.add_argument("--no-sub", action="store_true", help="skip the other workloads")
    ap.add_argument("--e2e-steps", type=int, default=40)
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--sampling-steps", type=int, default=200,
                    help="timed launches of each sampling-acceptance and DDTree-construction "
                         "call (0 = skip)")
    return ap.parse_args()


def workload_config(w):
    plen = np.asarray(w["prompt_len"])
    cu = np.asarray(w["cu_nodes"])
    return {
        "workload": {2: "llama3-8b-attn-medusa", 3: "llama3-8b-attn-eagle2",
                     4: "llama3-70b-attn-ddtree", 5: "llama3-8b-attn-ragged-eagle",
                     1: "tiny-medusa"}.get(w["config"], str(w["config"])),
        "description": __import__("gen.workloads",
                                  fromlist=["CONFIG_NAMES"]).CONFIG_NAMES[w["config"]],
        "batch": int(w["batch"]), "num_q_heads": w["num_q_heads"],
        "num_kv_heads": w["num_kv_heads"], "head_dim": w["head_dim"],
        "block_size": w["block_size"], "tree_nodes_per_request": sorted(set(np.diff(cu).tolist())),
        "prompt_len_mean": float(plen.mean()), "prompt_len_min": int(plen.min()),
        "prompt_len_max": int(plen.max()), "seed": 1000 + int(w["config"]),
        "l2": ("flushed before every timed step: 512 MiB write, then a 256 MiB read of another "
               "buffer, so each step starts with a cold and clean L2 (no dirty lines from the "
               "flush write-back during the step)"),
    }


def attention_algorithmic(w, depth):
    """Algorithmic bytes and FLOPs of one tv_tree_attention_verify launch."""
    hq, hkv, d = w["num_q_heads"], w["num_kv_heads"], w["head_dim"]
    cu = np.asarray(w["cu_nodes"])
    nbytes = 0
    flops = 0
    for b in range(w["batch"]):
        n = int(cu[b + 1] - cu[b])
        p = int(w["prompt_len"][b])
        nbytes += 2 * hkv * d * 2 * p                # prompt K + V read
        nbytes += n * (hq + 2 * hkv) * d * 2         # raw q, k, v read
        nbytes += n * 2 * hkv * d * 2                # rotated K + V written to the cache
        nbytes += n * hq * d * 2                     # output written
        flops += 4 * hq * d * n * p
        flops += 4 * hq * d * int(np.sum(depth[cu[b]:cu[b + 1]] + 1))
    return nbytes, flops


def attn_source_sha():
    return source_sha(ATTN_SOURCES)


SAMPLE_SOURCES = ("sample.cu", "tv_cluster.cuh", "tv_common.cuh")


DDTREE_SOURCES = ("ddtree.cu", "tv_common.cuh")


def measure_dense_mask(w, db, stream, flush, iters, hbm_peak):
    """Dense FULL_MASK export of the bench workload's trees (bool and additive
    float32), write-bound; CUDA events, L2 flushed before each launch."""
    import torch

    import speculative_decoding_tree_build_gb300 as tvb

    n_el = tvb.dense_mask_elements(w["cu_nodes"], w["prompt_len"], tvb.MASK_FULL)
    res = {}
    for name, dt, tdt, size in (("bool", tvb.MASK_BOOL, torch.uint8, 1),
                                ("additive_f32", tvb.MASK_ADDITIVE_F32, torch.float32, 4)):
        out = torch.empty(n_el, dtype=tdt, device=db.mask.device)
        st = torch.zeros_like(db.status)

        def fn():
            tvb.tree_mask_dense(db.mask, db.cu_nodes, db.prompt_len, st, int(w["max_nodes"]), out,
                                tvb.MASK_FULL, dt, stream)
        for _ in range(3):
            flush.zero_()
            fn()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(iters)]
        torch.cuda.synchronize()
        for a, b in evs:
            flush.zero_()
            a.record(stream)
            fn()
            b.record(stream)
        torch.cuda.synchronize()
        us = float(np.mean([a.elapsed_time(b) for a, b in evs])) * 1e3
        gbs = n_el * size / (us * 1e-6) / 1e9
        res[name] = {"us_per_launch": us, "bytes_written": n_el * size, "achieved_gbs": gbs,
                     "frac_of_hbm": gbs / hbm_peak}
    return res


def measure_eagle(dev, stream, flush, iters):
    """EAGLE-2 selection with the EAGLE-2 workload's recipe: 32 requests, six
    layers of top-8 expansion (328 candidates each; drafter log-probs from
    log_softmax of N(0, 2) logits), global top 64. Times one layer's
    tv_eagle_expand_select and tv_eagle_rerank (CUDA events, L2 flushed)."""
    import torch

    import speculative_decoding_tree_build_gb300 as tvb
    from gen import workloads as wl

    rng = np.random.default_rng(3003)
    batch, layers, k, keep = 32, 6, 8, 64
    reqs = [wl.eagle_candidates(rng, layers, k, 32000, 2.0) for _ in range(batch)]
    m = max(len(r[0]) for r in reqs)
    lp = np.zeros((batch, m), np.float32)
    par = np.full((batch, m), -1, np.int32)
    tok = np.zeros((batch, m), np.int32)
    cnt = np.zeros(batch, np.int32)
    for i, (l, p, t) in enumerate(reqs):
        lp[i, :len(l)], par[i, :len(l)], tok[i, :len(l)], cnt[i] = l, p, t, len(l)
    i32 = dict(dtype=torch.int32, device=dev)
    d_lp, d_par, d_tok, d_cnt = (torch.from_numpy(a).to(dev) for a in (lp, par, tok, cnt))
    sel = torch.empty((batch, k), **i32)
    st = torch.zeros(batch, **i32)
    parents = torch.empty(batch * (keep + 1), **i32)
    tokens = torch.empty(batch * (keep + 1), **i32)
    cu = torch.empty(batch + 1, **i32)

    def run_select():
        tvb.eagle_expand_select(d_lp, d_par, d_cnt, layers - 1, k, sel, st, stream)

    def run_rerank():
        tvb.eagle_rerank(d_lp, d_par, d_tok, d_cnt, keep, parents, tokens, cu, st, stream=stream)

    def timed(fn):
        for _ in range(3):
            flush.zero_()
            fn()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(iters)]
        torch.cuda.synchronize()
        for a, b in evs:
            flush.zero_()
            a.record(stream)
            fn()
            b.record(stream)
        torch.cuda.synchronize()
        return float(np.mean([a.elapsed_time(b) for a, b in evs])) * 1e3

    us_sel, us_rr = timed(run_select), timed(run_rerank)
    if int(st.abs().sum()) != 0:
        raise RuntimeError("EAGLE selection produced status flags")
    return {"workload": f"32 requests, {m} candidates each (6 layers x top-8), keep 64",
            "expand_select_us": us_sel, "rerank_us": us_rr,
            "note": "latency-bound: one CTA per request, candidates ranked in shared memory"}


def measure_ddtree(dev, stream, flush, iters, hbm_peak):
    """DDTree draft-tree construction with the DDTree workload's drafter
    recipe: 16 requests x L = 16 positions, vocabulary 151936, logits
    N(0, 3) (float32), budget B = 256 (K = 256). Times tv_ddtree_topk (HBM:
    every logit read once) and tv_ddtree_build (B dependent heap pops per
    request) with CUDA events, L2 flushed before each launch."""
    import torch

    import speculative_decoding_tree_build_gb300 as tvb

    batch, L, V, B = 16, 16, 151936, 256
    rng = np.random.default_rng(4004)
    logits_h = np.empty((batch * L, V), np.float32)
    rng.standard_normal(dtype=np.float32, out=logits_h)
    logits_h *= np.float32(3.0)
    logits = torch.from_numpy(logits_h).to(dev)
    i32 = dict(dtype=torch.int32, device=dev)
    tt = torch.empty((batch * L, B), **i32)
    tq = torch.empty((batch * L, B), dtype=torch.float32, device=dev)
    n = tvb.ddtree_nodes(L, B, B)
    par, tok = torch.empty(batch * n, **i32), torch.empty(batch * n, **i32)
    cu = torch.empty(batch + 1, **i32)

    def run_topk():
        tvb.ddtree_topk(logits, B, tt, tq, stream)

    def run_build():
        tvb.ddtree_build(tq.view(batch, L, B), tt.view(batch, L, B), B, par, tok, cu,
                         stream=stream)

    def timed(fn):
        for _ in range(3):
            flush.zero_()
            fn()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(iters)]
        torch.cuda.synchronize()
        for a, b in evs:
            flush.zero_()
            a.record(stream)
            fn()
            b.record(stream)
        torch.cuda.synchronize()
        return float(np.mean([a.elapsed_time(b) for a, b in evs])) * 1e3

    us_topk = timed(run_topk)
    us_build = timed(run_build)
    nbytes = batch * L * V * 4 + batch * L * B * 8
    gbs = nbytes / (us_topk * 1e-6) / 1e9
    return {
        "workload": "16 requests x 16 positions, vocabulary 151936, N(0,3) float32 logits, B=256",
        "ddtree_topk": {"us_per_launch": us_topk, "algorithmic_bytes": nbytes,
                        "roofline": {"bound": "hbm", "achieved": gbs, "peak": hbm_peak,
                                     "unit": "GB/s", "frac": gbs / hbm_peak,
                                     "traffic": recorded_traffic(4, "ddtree_topk",
                                                                 DDTREE_SOURCES)}},
        "ddtree_build": {"us_per_launch": us_build, "pops_per_request": B,
                         "ns_per_pop": us_build * 1e3 / B,
                         "note": "latency-bound: B dependent best-first pops per request, "
                                 "one warp per request, all requests in parallel"},
        "trees_per_s": batch / ((us_topk + us_build) * 1e-6),
    }


def measure_sampling(w, dev, stream, flush, iters, hbm_peak):
    """Sampling acceptance on the bench workload's trees: per-node target
    logits over the workload's vocabulary (float32, N(0, 1) with a boosted
    child token) and float32 Gumbel noise, every request at temperature 1.
    Times tv_sample_tokens (all nodes) and tv_sampled_accept (the walk, which
    reads only the visited nodes' rows) with CUDA events, L2 flushed before
    each launch."""
    import torch

    import speculative_decoding_tree_build_gb300 as tvb
    from gen import workloads as wl

    rng = np.random.default_rng(4242 + int(w["config"]))
    logits_h, gumbel_h = wl.sampling_inputs(rng, w)
    vocab = int(w["vocab"])
    bsz = int(w["batch"])
    total = int(w["cu_nodes"][-1])
    logits = torch.from_numpy(logits_h).to(dev)
    gumbel = torch.from_numpy(gumbel_h).to(dev)
    i32 = dict(dtype=torch.int32, device=dev)
    cu = torch.from_numpy(np.asarray(w["cu_nodes"], np.int32)).to(dev)
    parents = torch.from_numpy(np.asarray(w["parents"], np.int32)).to(dev)
    draft = torch.from_numpy(np.asarray(w["draft_tokens"], np.int32)).to(dev)
    temps = torch.ones(bsz, dtype=torch.float32, device=dev)
    status = torch.zeros(bsz, **i32)
    tokens = torch.empty(total, **i32)
    md = int(w["max_depth"])
    path = torch.empty((bsz, md + 1), **i32)
    alen, bonus = torch.empty(bsz, **i32), torch.empty(bsz, **i32)
    mn = int(w["max_nodes"])

    def run_sample():
        tvb.sample_tokens(logits, gumbel, cu, temps, mn, tokens, status, stream)

    def run_walk():
        tvb.sampled_accept(logits, gumbel, cu, temps, parents, draft, mn, path, alen, bonus,
                           status, stream)

    def timed(fn):
        for _ in range(3):
            flush.zero_()
            fn()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(iters)]
        torch.cuda.synchronize()
        for a, b in evs:
            flush.zero_()
            a.record(stream)
            fn()
            b.record(stream)
        torch.cuda.synchronize()
        return float(np.mean([a.elapsed_time(b) for a, b in evs])) * 1e3

    us_sample = timed(run_sample)
    us_walk = timed(run_walk)
    if int(status.abs().sum()) != 0:
        raise RuntimeError("sampling produced status flags")
    visited = int((alen.cpu().numpy() + 1).sum())
    bytes_sample = total * vocab * 8 + total * 4
    bytes_walk = visited * vocab * 8
    gbs_sample = bytes_sample / (us_sample * 1e-6) / 1e9
    gbs_walk = bytes_walk / (us_walk * 1e-6) / 1e9
    return {
        "vocab": vocab, "temperature": 1.0, "nodes": total,
        "inputs": "float32 logits N(0,1) + boosted child token, float32 Gumbel noise",
        "sample_tokens": {
            "us_per_launch": us_sample, "algorithmic_bytes": bytes_sample,
            "roofline": {"bound": "hbm", "achieved": gbs_sample, "peak": hbm_peak,
                         "unit": "GB/s", "frac": gbs_sample / hbm_peak,
                         "traffic": recorded_traffic(w["config"], "sample_tokens",
                                                     SAMPLE_SOURCES)},
            "nodes_per_s": total / (us_sample * 1e-6)},
        "sampled_accept": {
            "us_per_launch": us_walk, "visited_rows": visited, "algorithmic_bytes": bytes_walk,
            "achieved_gbs": gbs_walk, "frac_of_hbm": gbs_walk / hbm_peak,
            "speedup_vs_sample_all_then_walk": us_sample / us_walk,
            "note": "latency-bound: one row per step per request, steps in sequence"},
    }


def measure_rejection(w, dev, stream, flush, iters, hbm_peak):
    """Rejection-sampling acceptance on the bench workload's trees: drafter
    logits with boosted child tokens, target logits = drafter's + N(0, 0.5),
    Gumbel noise, uniforms, draft log-probabilities (float32), temperature 1.
    Times tv_rejection_accept with CUDA events, L2 flushed before each
    launch. Algorithmic bytes: the target and drafter rows of every visited
    node (the accepted prefix and the stop node) plus the stop node's noise
    row; the kernel also reads the chosen path's rows past the stop node
    (all path rows are reduced in parallel)."""
    import torch

    import speculative_decoding_tree_build_gb300 as tvb
    from gen import workloads as wl

    rng = np.random.default_rng(5151 + int(w["config"]))
    logits_h, draft_h, gumbel_h, unif_h, logp_h = wl.rejection_inputs(rng, w)
    vocab = int(w["vocab"])
    bsz = int(w["batch"])
    logits, draft_l, gumbel = (torch.from_numpy(a).to(dev) for a in (logits_h, draft_h, gumbel_h))
    unif, logp = torch.from_numpy(unif_h).to(dev), torch.from_numpy(logp_h).to(dev)
    i32 = dict(dtype=torch.int32, device=dev)
    cu = torch.from_numpy(np.asarray(w["cu_nodes"], np.int32)).to(dev)
    parents = torch.from_numpy(np.asarray(w["parents"], np.int32)).to(dev)
    tokens = torch.from_numpy(np.asarray(w["draft_tokens"], np.int32)).to(dev)
    temps = torch.ones(bsz, dtype=torch.float32, device=dev)
    status = torch.zeros(bsz, **i32)
    md = int(w["max_depth"])
    path = torch.empty((bsz, md + 1), **i32)
    alen, bonus = torch.empty(bsz, **i32), torch.empty(bsz, **i32)
    mn = int(w["max_nodes"])

    def run():
        tvb.rejection_accept(logits, draft_l, gumbel, unif, cu, temps, parents, tokens, logp, mn,
                             path, alen, bonus, status, stream)

    for _ in range(3):
        flush.zero_()
        run()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(iters)]
    torch.cuda.synchronize()
    for a, b in evs:
        flush.zero_()
        a.record(stream)
        run()
        b.record(stream)
    torch.cuda.synchronize()
    us = float(np.mean([a.elapsed_time(b) for a, b in evs])) * 1e3
    if int(status.abs().sum()) != 0:
        raise RuntimeError("rejection walk produced status flags")
    acc = alen.cpu().numpy()
    visited = int((acc + 1).sum())
    algo = visited * vocab * 8 + bsz * vocab * 4
    gbs = algo / (us * 1e-6) / 1e9
    return {
        "vocab": vocab, "temperature": 1.0, "requests": bsz,
        "mean_accepted": float(acc.mean()),
        "inputs": "float32 drafter logits N(0,1) + boosted children, target = drafter + N(0,0.5), "
                  "float32 Gumbel noise and uniforms",
        "us_per_launch": us, "visited_rows": visited, "algorithmic_bytes": algo,
        "achieved_gbs": gbs, "frac_of_hbm": gbs / hbm_peak,
        "requests_per_s": bsz / (us * 1e-6)}


def _code_only(text):
    """Source text without comments and blank lines, so that a comment edit
    does not disown the counters taken on the same code."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    lines = (re.sub(r"//.*$", "", ln).rstrip() for ln in text.splitlines())
    return "\n".join(ln for ln in lines if ln.strip())


def source_sha(files):
    """Hash of the code (comments stripped) of the given csrc files."""
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "speculative_decoding_tree_build_gb300", "csrc", f), encoding="utf-8") as fh:
            h.update(_code_only(fh.read()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(config, name="tree_attention_verify", sources=ATTN_SOURCES,
                     key="dram_bytes_per_launch"):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the current source of that kernel."""
    path = os.path.join(ROOT, "profiles", f"{name}_config{config}.md")
    if not os.path.exists(path):
        return None
    vals = {}
    with open(path, encoding="utf-8") as fh:
        for line in fh:
            if ":" in line and line.startswith("- "):
                k, v = line[2:].split(":", 1)
                vals[k.strip()] = v.strip().strip("`")
    if vals.get("source_sha", vals.get("attention_source_sha")) != source_sha(sources):
        return None
    try:
        return float(vals[key])
    except (KeyError, ValueError):
        return None


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as fh:
            d = json.load(fh)
        return d.get("hbm_gbs", 6800.0), d.get("bf16_tflops", 1900.0), "measured"
    return 6800.0, 1900.0, "fallback"


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during a region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.idx = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(self.idx), "-lms", "100"], stdout=subprocess.PIPE,
                stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=5)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": float(max(mx)),
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ CPU oracle

def _oracle_worker(args):
    os.environ["OPENBLAS_NUM_THREADS"] = "1"
    w, req_ids, node_limit = args
    from oracle import verify_step_ref
    t0 = time.perf_counter()
    nodes = 0
    cu = np.asarray(w["cu_nodes"])
    for b in req_ids:
        n = int(cu[b + 1] - cu[b])
        use = n if node_limit is None else min(n, node_limit)
        sub = _sub_workload(w, b)
        pairs = {0: [(i, h) for i in range(use) for h in range(w["num_q_heads"])]}
        verify_step_ref(sub, sample=pairs)
        nodes += use
    return nodes, time.perf_counter() - t0


def _sub_workload(w, b):
    cu = np.asarray(w["cu_nodes"])
    t0, t1 = int(cu[b]), int(cu[b + 1])
    sub = dict(w)
    sub.update(batch=1, cu_nodes=np.array([0, t1 - t0], np.int32),
               parents=w["parents"][t0:t1], prompt_len=w["prompt_len"][b:b + 1],
               draft_tokens=w["draft_tokens"][t0:t1], target_ids=w["target_ids"][t0:t1],
               q=w["q"][t0:t1], k_new=w["k_new"][t0:t1], v_new=w["v_new"][t0:t1],
               block_table=w["block_table"][b:b + 1], n_blocks=w["n_blocks"][b:b + 1])
    return sub


def cpu_baseline(w, seconds, node_limit=None):
    """Time the oracle (as it stands) on the host cores: one spawn worker per
    core, single-threaded BLAS, each worker verifying requests (all query
    heads of the first ``node_limit`` nodes of each, or every node)."""
    cores = os.cpu_count() or 1
    ctx = mp.get_context("spawn")
    batch = w["batch"]
    # calibrate on one request
    n0, t_one = _oracle_worker((w, [0], node_limit))
    per_req = max(t_one, 1e-3)
    reqs_total = max(1, int(seconds * cores / per_req))
    order = [i % batch for i in range(reqs_total)]
    chunks = [order[i::cores] for i in range(cores)]
    chunks = [c for c in chunks if c]
    t0 = time.perf_counter()
    with ctx.Pool(len(chunks)) as pool:
        res = pool.map(_oracle_worker, [(w, c, node_limit) for c in chunks])
    wall = time.perf_counter() - t0
    nodes = sum(r[0] for r in res)
    what = "every node" if node_limit is None else f"the first {node_limit} nodes"
    return {"value": nodes / wall, "unit": UNIT, "cores": len(chunks), "kind": "oracle",
            "sample": f"{reqs_total} requests of the workload's first step ({what} of each, all query "
                      f"heads: {nodes} tree nodes verified, full step per request) over "
                      f"{len(chunks)} spawn workers, {wall:.1f} s wall"}


def rank_seed(config, rank):
    """Each rank verifies its own batch (requests are independent)."""
    return 1000 + config + 7919 * rank


def reduce_over_ranks(times_ms, tokens, world, device):
    """Whole-job numbers of a weak-scaling run: every time is the maximum over
    ranks (the job ends with its slowest rank), the token count the sum."""
    import torch
    import torch.distributed as dist

    if world <= 1:
        return [float(t) for t in times_ms], float(tokens)
    mx = torch.tensor([float(t) for t in times_ms], dtype=torch.float64, device=device)
    sm = torch.tensor([float(tokens)], dtype=torch.float64, device=device)
    dist.all_reduce(mx, op=dist.ReduceOp.MAX)
    dist.all_reduce(sm, op=dist.ReduceOp.SUM)
    return [float(t) for t in mx.tolist()], float(sm[0])


# oracle sample for the CPU baseline and the reference arm: config 5's
# requests have prompts of 4K-32K tokens, so a few nodes of each
ORACLE_NODE_LIMIT = {5: 4}


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from gen import workloads as wl
    w = wl.make_config(args.config)
    cores = os.cpu_count() or 1
    # each step: one request's verification on the oracle (a bounded number of
    # its nodes); sized so the whole run ends in minutes
    cap = ORACLE_NODE_LIMIT.get(args.config)
    n_first, t_first = _oracle_worker((w, [0], cap))
    budget = 150.0
    per_step = budget / max(1, args.steps + args.warmup)
    node_limit = max(1, int(n_first * min(1.0, per_step / max(t_first, 1e-6))))
    times, nodes = [], 0
    for s in range(args.warmup + args.steps):
        b = s % w["batch"]
        n, dt = _oracle_worker((w, [b], node_limit))
        if s >= args.warmup:
            times.append(dt)
            nodes += n
    total = sum(times)
    value = nodes / total
    ref_config = workload_config(w)
    if args.config == 5:
        # the GPU arm's headline is this workload's eight evolving steps; the
        # oracle's bounded sample comes from the first of them
        ref_config = dict(ref_config, workload="llama3-8b-attn-ragged-eagle-8steps", steps_per_cycle=MULTISTEP,
                          oracle_sample="requests of the first of the eight steps")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": ref_config,
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": f"each step verifies {node_limit} node(s) (all query heads) "
                                   f"of one request of the workload's first step on the CPU "
                                   f"oracle, single process"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "host_cores_available": cores,
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ GPU arm

def make_flush(dev):
    import torch

    flush_w = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=dev)
    flush_r = torch.ones(L2_FLUSH_BYTES // 8, dtype=torch.int32, device=dev)
    flush_sink = torch.zeros((), dtype=torch.int64, device=dev)

    class _Flush:
        """Evict the L2 before a timed step: write a buffer larger than the
        126 MB L2, then read another one so the lines left behind are clean
        (otherwise the step would pay for writing the flush data back)."""

        @staticmethod
        def zero_():
            flush_w.zero_()
            flush_sink.add_(flush_r.sum())

    return _Flush()


def timed_replays(graphs, stream, flush, n):
    """CUDA-event time (ms) of n replays cycling through ``graphs``, the L2
    flushed (outside the events) before each."""
    import torch

    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(n)]
    torch.cuda.synchronize()
    for i in range(n):
        flush.zero_()
        evs[i][0].record(stream)
        graphs[i % len(graphs)].replay()
        evs[i][1].record(stream)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in evs]


def e2e_pipelined(steps, stream, n, dev):
    """End to end over n steps cycling through ``steps`` = [(DeviceBatch,
    CUDAGraph)]: each step's inputs are copied in from pinned host memory (one
    copy) on an upload stream while the previous step computes, and its
    results are copied out (one copy) on a download stream while the next one
    computes. Timed with CUDA events from the first copy in to the last copy
    out. Returns (ms per step, mean H2D bytes, mean D2H bytes, host outputs)."""
    import torch

    m = len(steps)
    h_in = [db.inputs.cpu().pin_memory() for db, _ in steps]
    h_out = [torch.empty_like(db.outputs, device="cpu").pin_memory() for db, _ in steps]
    up, down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(n)]
    ev_done = [torch.cuda.Event() for _ in range(n)]
    ev_out = [torch.cuda.Event() for _ in range(n)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def copy_in(i):
        k = i % m
        with torch.cuda.stream(up):
            if i >= m:
                up.wait_event(ev_done[i - m])          # the last step that read this buffer
            steps[k][0].inputs.copy_(h_in[k], non_blocking=True)
            ev_in[i].record(up)

    torch.cuda.synchronize()
    t0.record(stream)
    up.wait_stream(stream)
    down.wait_stream(stream)
    copy_in(0)
    for i in range(n):
        k = i % m
        stream.wait_event(ev_in[i])
        if i >= m:
            stream.wait_event(ev_out[i - m])           # its outputs were read out
        steps[k][1].replay()
        ev_done[i].record(stream)
        if i + 1 < n:
            copy_in(i + 1)
        with torch.cuda.stream(down):
            down.wait_event(ev_done[i])
            h_out[k].copy_(steps[k][0].outputs, non_blocking=True)
            ev_out[i].record(down)
    stream.wait_stream(down)
    t1.record(stream)
    torch.cuda.synchronize()
    h2d = float(np.mean([t.numel() * t.element_size() for t in h_in]))
    d2h = float(np.mean([t.numel() * t.element_size() for t in h_out]))
    return t0.elapsed_time(t1) / n, h2d, d2h, h_out


def e2e_sequential(db, graph, stream, flush, n):
    """End to end, one step at a time: flush L2, then per step the inputs
    copied in from pinned host memory (one copy), the step's graph, its
    results copied out (one copy), bracketed by CUDA events."""
    import torch

    h_in = db.inputs.cpu().pin_memory()
    h_out = torch.empty_like(db.outputs, device="cpu").pin_memory()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    torch.cuda.synchronize()
    for i in range(n):
        flush.zero_()
        evs[i][0].record(stream)
        db.inputs.copy_(h_in, non_blocking=True)
        graph.replay()
        h_out.copy_(db.outputs, non_blocking=True)
        evs[i][1].record(stream)
    torch.cuda.synchronize()
    ms = float(np.mean([a.elapsed_time(b) for a, b in evs]))
    return ms, float(h_in.numel() * h_in.element_size()), float(h_out.numel() * h_out.element_size()), h_out


def roofline_of(nbytes, flops, attn_s, hbm_peak, tf_peak, src):
    ridge = tf_peak * 1e12 / (hbm_peak * 1e9)
    roof_s = max(nbytes / (hbm_peak * 1e9), flops / (tf_peak * 1e12))
    gbs = nbytes / attn_s / 1e9
    tfs = flops / attn_s / 1e12
    if flops / nbytes < ridge:
        roof = {"bound": "hbm", "achieved": gbs, "peak": hbm_peak, "unit": "GB/s", "frac": gbs / hbm_peak}
    else:
        roof = {"bound": "tensor", "achieved": tfs, "peak": tf_peak, "unit": "TFLOP/s",
                "frac": tfs / tf_peak}
    roof.update(peak_source=src, algorithmic_bytes=nbytes, algorithmic_flops=flops,
                attention_us=attn_s * 1e6, roofline_us=roof_s * 1e6,
                frac_of_roofline_time=roof_s / attn_s, frac_of_nominal_8tbs=gbs / 8000.0)
    return roof


def prepare_multistep(w0, dev, nsteps, seed):
    """Run the config-5 loop once, untimed: verify -> accept + commit (block
    release) -> host allocator (released blocks back on the free list, blocks
    for the next tree's slots taken from it) -> next tree at P + 1 + a, with
    fresh EAGLE-style trees. Returns per step (DeviceBatch, block-table
    snapshot the step starts from, inputs); every step's batch shares one KV
    pool, block table and workspace. A replay of the steps in order repeats
    the same work: step k reads only prompt slots no later step writes."""
    import torch

    from gen import workloads as wl
    from speculative_decoding_tree_build_gb300.step import DeviceBatch

    rng = np.random.default_rng(seed)
    out = []
    w = w0
    base = None
    for k in range(nsteps):
        db = DeviceBatch(w, device=dev) if base is None else DeviceBatch(w, device=dev, share=base)
        base = base or db
        snap = torch.from_numpy(np.concatenate([np.ascontiguousarray(w["block_table"], np.int32).reshape(-1),
                                                np.asarray(w["n_blocks"], np.int32)])).to(dev)
        db.table_state.copy_(snap)
        db.status.zero_()
        db.tree_build()
        db.attention()
        db.accept_commit()
        torch.cuda.synchronize()
        st = db.status.cpu().numpy()
        if np.any(st != 0):
            raise RuntimeError(f"multi-step workload: step {k} produced status flags {st}")
        out.append((db, snap, w))
        if k == nsteps - 1:
            break
        new_len = db.new_len.cpu().numpy()
        bonus = db.bonus.cpu().numpy()
        rel = db.released.cpu().numpy()
        cnt = db.released_count.cpu().numpy()
        tab = db.table_state.cpu().numpy()
        nb = w["block_table"].size
        free = list(w["free_blocks"])
        for b in range(w["batch"]):
            free.extend(int(x) for x in rel[b][:cnt[b]])
        state = dict(w, block_table=tab[:nb].reshape(w["block_table"].shape).copy(),
                     n_blocks=tab[nb:].copy(), free_blocks=free)
        trees = []
        for b in range(w["batch"]):
            n_tree = int(rng.choice([16, 32, 64, 128]))
            trees.append(wl.eagle_tree(rng, 0, int(rng.integers(4, 11)), n_tree, wl.VOCAB_LLAMA,
                                       2.0, until_count=True)[:2])
        w = wl.next_step_inputs(rng, state, new_len, bonus, trees)
    return out


def measure_single(cfg, dev, stream, flush, rank, iters, hbm_peak, tf_peak, src):
    """One verification step of workload ``cfg``, replayed as one CUDA graph
    from a restored block table; its attention call timed in its own loop."""
    import torch

    from gen import workloads as wl
    from speculative_decoding_tree_build_gb300.step import DeviceBatch

    w = wl.make_config(cfg, seed=rank_seed(cfg, rank))
    db = DeviceBatch(w, device=dev)
    table0 = db.table_state.clone()

    def pre():
        db.table_state.copy_(table0, non_blocking=True)   # allocator refill
        db.tree_build()

    def step():
        pre()
        db.attention()
        db.accept_commit()

    side = torch.cuda.Stream(dev)
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        for _ in range(3):
            flush.zero_()
            step()
    stream.wait_stream(side)
    torch.cuda.synchronize()
    if int(db.status.abs().sum()) != 0:
        raise RuntimeError(f"config {cfg}: status flags")
    depth = db.depth.cpu().numpy()
    g_step, g_pre, g_attn = (torch.cuda.CUDAGraph() for _ in range(3))
    with torch.cuda.graph(g_step, stream=side):
        step()
    with torch.cuda.graph(g_pre, stream=side):
        pre()
    with torch.cuda.graph(g_attn, stream=side):
        db.attention()
    torch.cuda.synchronize()
    for _ in range(3):
        flush.zero_()
        g_step.replay()
    step_ms = float(np.mean(timed_replays([g_step], stream, flush, iters)))
    g_pre.replay()
    attn_ms = float(np.mean(timed_replays([g_attn], stream, flush, iters)))
    if int(db.status.abs().sum()) != 0:
        raise RuntimeError(f"config {cfg}: replay status flags")
    tokens = int(w["cu_nodes"][-1])
    nbytes, flops = attention_algorithmic(w, depth)
    roof = roofline_of(nbytes, flops, attn_ms * 1e-3, hbm_peak, tf_peak, src)
    roof["traffic"] = recorded_traffic(cfg)
    e2e_ms, h2d, d2h, h_out = e2e_sequential(db, g_step, stream, flush, max(3, min(iters, 40)))
    if int(h_out[:4 * int(w["batch"])].view(torch.int32).abs().sum()) != 0:
        raise RuntimeError(f"config {cfg}: end-to-end status flags")
    return w, db, {"workload": workload_config(w)["workload"], "config": workload_config(w),
                   "tokens_per_step": tokens, "ms_per_step": step_ms,
                   "tokens_per_s": tokens / (step_ms * 1e-3),
                   "attention_tokens_per_s": tokens / (attn_ms * 1e-3), "roofline": roof,
                   "e2e": {"value": tokens / (e2e_ms * 1e-3), "unit": UNIT, "h2d_bytes_per_step": h2d,
                           "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                           "mode": "L2 flushed, then per step the pinned host inputs copied in (one copy), "
                                   "the step's CUDA graph, the results copied out (one copy), CUDA events"},
                   "timing": f"{iters} flushed replays of the step's CUDA graph, and of the "
                             f"attention call's, CUDA events"}


def run_ours(args):
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    from __graft_entry__ import build
    build()
    from gen import workloads as wl

    hbm_peak, tf_peak, src = measured_peaks()
    stream = torch.cuda.current_stream(dev)
    flush = make_flush(dev)
    sampler = ClockSampler(local) if rank == 0 else None
    if sampler:
        sampler.start()

    if args.config != 5:
        # a single-step workload as the headline
        w, db, single = measure_single(args.config, dev, stream, flush, rank, args.steps,
                                       hbm_peak, tf_peak, src)
        multi = None
    else:
        w = wl.make_config(5, seed=rank_seed(5, rank))
        multi = prepare_multistep(w, dev, MULTISTEP, seed=rank_seed(5, rank) + 77)
    side = torch.cuda.Stream(dev)

    if multi is not None:
        # ---- the eight evolving steps, each its own CUDA graph: restore the
        # step's block table (the allocator's result), tree_build, attention,
        # accept + commit with block release; timed steps cycle through them
        graphs, attn_graphs, pre_graphs = [], [], []
        for db, snap, wk in multi:
            def pre(db=db, snap=snap):
                db.table_state.copy_(snap, non_blocking=True)
                db.tree_build()

            def step(db=db, pre=pre):
                pre()
                db.attention()
                db.accept_commit()
            side.wait_stream(stream)
            g, ga, gp = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=side):
                step()
            with torch.cuda.graph(gp, stream=side):
                pre()
            with torch.cuda.graph(ga, stream=side):
                db.attention()
            graphs.append(g)
            pre_graphs.append(gp)
            attn_graphs.append(ga)
        torch.cuda.synchronize()
        for _ in range(max(3, args.warmup)):
            for g in graphs:
                flush.zero_()
                g.replay()
        torch.cuda.synchronize()
        tokens = [int(wk["cu_nodes"][-1]) for _, _, wk in multi]
        if world > 1:
            dist.barrier()
        times = timed_replays(graphs, stream, flush, args.steps)
        if world > 1:
            dist.barrier()
        step_ms = float(np.sum(times)) / args.steps
        tokens_timed = float(sum(tokens[i % MULTISTEP] for i in range(args.steps)))
        # each step's attention call in its own loop (table and tree of that step)
        attn_ms, per_step = [], []
        tot_b = tot_f = 0
        for k, (db, snap, wk) in enumerate(multi):
            pre_graphs[k].replay()
            ms = float(np.mean(timed_replays([attn_graphs[k]], stream, flush, args.attn_iters)))
            depth = db.depth.cpu().numpy()
            nb, nf = attention_algorithmic(wk, depth)
            attn_ms.append(ms)
            tot_b += nb
            tot_f += nf
            per_step.append({"step": k, "tokens": tokens[k], "attention_us": ms * 1e3,
                             "algorithmic_bytes": nb, "prompt_len_mean": float(np.mean(wk["prompt_len"])),
                             "hbm_frac": nb / (ms * 1e-3) / 1e9 / hbm_peak})
        for db, _, _ in multi:
            if int(db.status.abs().sum()) != 0:
                raise RuntimeError("multi-step replay produced status flags")
        attn_total_s = float(np.sum(attn_ms)) * 1e-3
        roof = roofline_of(tot_b, tot_f, attn_total_s, hbm_peak, tf_peak, src)
        roof.update(traffic=recorded_traffic(5), per_step=per_step,
                    attention_timing=("each step's attention call in its own loop of graph replays "
                                      "on the step's stream, L2 flushed before each, CUDA events; "
                                      "the eight steps' algorithmic bytes over the sum of their times"))
        # end to end: every step's inputs copied in from pinned host memory and
        # its results copied out, the copies of one step overlapping the
        # neighbouring steps' compute (each step has its own buffers)
        n_e2e = max(MULTISTEP, args.e2e_steps)
        e2e_ms, h2d, d2h, h_out = e2e_pipelined([(db, graphs[k]) for k, (db, _, _) in enumerate(multi)],
                                                stream, n_e2e, dev)
        for k, (db, _, wk) in enumerate(multi):
            if int(h_out[k][:4 * int(wk["batch"])].view(torch.int32).abs().sum()) != 0:
                raise RuntimeError("end-to-end step produced status flags")
        (step_ms, e2e_ms), tokens_all = reduce_over_ranks([step_ms, e2e_ms], tokens_timed / args.steps,
                                                          world, dev)
        headline_cfg = dict(workload_config(w), workload="llama3-8b-attn-ragged-eagle-8steps",
                            steps_per_cycle=MULTISTEP,
                            loop=("verify -> greedy accept + KV commit with block release -> host "
                                  "allocator (released blocks back on the free list, the next tree's "
                                  "slots allocated) -> next EAGLE-style tree at P + 1 + a; the eight "
                                  "steps precomputed once, then replayed in order (each timed step "
                                  "restores its step's block table, as the allocator leaves it)"),
                            tokens_per_step=tokens,
                            prompt_len_mean_per_step=[float(np.mean(wk["prompt_len"])) for _, _, wk in multi])
        line = {
            "metric": METRIC, "value": tokens_all / (step_ms * 1e-3), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic", "config": headline_cfg, "roofline": roof,
            "e2e": {"value": tokens_all / (e2e_ms * 1e-3), "unit": UNIT, "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                    "mode": "every step's pinned host inputs copied in (one copy) on an upload stream while "
                            "the previous step computes, its results copied out (one copy) on a download "
                            "stream while the next one computes, the step's library calls replayed from its "
                            "CUDA graph; timed from the first copy in to the last copy out (no L2 flush: each "
                            "step streams ~3.8 GB of K/V, 30x the L2)"},
            "gpu_launches": 5 * args.steps,   # tree_build, rope_append, attn_tc, attn_merge, accept_commit
            "attention_tokens_per_s": float(sum(tokens)) / attn_total_s,
        }
        w0, db0 = multi[0][2], multi[0][0]
    else:
        (step_ms,), tokens_all = reduce_over_ranks([single["ms_per_step"]], single["tokens_per_step"],
                                                   world, dev)
        line = {
            "metric": METRIC, "value": tokens_all / (step_ms * 1e-3), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic", "config": single["config"], "roofline": single["roofline"],
            "e2e": single["e2e"],
            "gpu_launches": 5 * args.steps,
            "attention_tokens_per_s": single["attention_tokens_per_s"],
        }
        w0, db0 = w, db

    # ---- the other workloads, one verification step each
    if not args.no_sub and rank == 0:
        subs = {}
        for cfg in SUB_CONFIGS:
            if cfg == args.config:
                continue
            _, _, res = measure_single(cfg, dev, stream, flush, rank, args.sub_iters, hbm_peak, tf_peak,
                                       src)
            subs[f"config{cfg}"] = res
        line["sub_workloads"] = subs
    clocks = sampler.stop() if sampler else None
    line["clocks"] = clocks
    if world > 1:
        dist.destroy_process_group()
    if rank != 0:
        return
    if args.sampling_steps > 0:
        # the NEXT-row kernels on the config-2 workload's trees (small rows)
        w2 = wl.make_config(2, seed=rank_seed(2, rank))
        from speculative_decoding_tree_build_gb300.step import DeviceBatch
        db2 = DeviceBatch(w2, device=dev)
        db2.tree_build()
        torch.cuda.synchronize()
        line["sampling"] = measure_sampling(w2, dev, stream, flush, args.sampling_steps, hbm_peak)
        line["rejection_acceptance"] = measure_rejection(w2, dev, stream, flush, args.sampling_steps,
                                                         hbm_peak)
        line["ddtree_construction"] = measure_ddtree(dev, stream, flush, args.sampling_steps, hbm_peak)
        line["eagle_selection"] = measure_eagle(dev, stream, flush, args.sampling_steps)
        line["dense_mask_export"] = measure_dense_mask(w2, db2, stream, flush, args.sampling_steps,
                                                       hbm_peak)
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w0, args.cpu_seconds, ORACLE_NODE_LIMIT.get(args.config))
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
