"""Benchmark of one token-tree verification step on GB300.

A step is the whole hot path over one batch: tv_tree_build ->
tv_tree_attention_verify -> tv_greedy_accept -> tv_kv_commit (plus the
block-table refill a serving loop's allocator does before the next step).
The default workload is the Llama-3-8B attention geometry, batch 8, prompt
lengths U[512, 2048], Medusa 4x3x2 trees (41 nodes incl. root), paged KV
block 16 with a shuffled block table.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--config C]

Under torchrun every rank runs its own batch (requests are independent: no
data-path collective); rank 0 prints one JSON line. ``--impl reference`` times
the CPU oracle on the host cores instead.
"""

from __future__ import annotations

import argparse
import hashlib
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
ATTN_SOURCES = ("attention_tc.cu", "tv_sm100.cuh", "tv_common.cuh")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", type=int, default=2)
    ap.add_argument("--e2e-steps", type=int, default=200)
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


def source_sha(files):
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "speculative_decoding_tree_build_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
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


def cpu_baseline(w, seconds):
    """Time the oracle (as it stands) on the host cores: one spawn worker per
    core, single-threaded BLAS, each worker verifying whole requests."""
    cores = os.cpu_count() or 1
    ctx = mp.get_context("spawn")
    batch = w["batch"]
    # calibrate on one request
    n0, t_one = _oracle_worker((w, [0], None))
    per_req = max(t_one, 1e-3)
    reqs_total = max(1, int(seconds * cores / per_req))
    order = [i % batch for i in range(reqs_total)]
    chunks = [order[i::cores] for i in range(cores)]
    chunks = [c for c in chunks if c]
    t0 = time.perf_counter()
    with ctx.Pool(len(chunks)) as pool:
        res = pool.map(_oracle_worker, [(w, c, None) for c in chunks])
    wall = time.perf_counter() - t0
    nodes = sum(r[0] for r in res)
    return {"value": nodes / wall, "unit": UNIT, "cores": len(chunks), "kind": "oracle",
            "sample": f"{reqs_total} requests of the workload ({nodes} tree nodes, all query "
                      f"heads, full step per request) over {len(chunks)} spawn workers, "
                      f"{wall:.1f} s wall"}


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


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from gen import workloads as wl
    w = wl.make_config(args.config)
    cores = os.cpu_count() or 1
    # each step: one request's verification on the oracle; size so the run ends in minutes
    n_first, t_first = _oracle_worker((w, [0], None))
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
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": workload_config(w),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": f"each step verifies {node_limit} node(s) (all query heads) "
                                   f"of one request on the CPU oracle, single process"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "host_cores_available": cores,
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ GPU arm

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
    from speculative_decoding_tree_build_gb300.step import DeviceBatch

    w = wl.make_config(args.config, seed=rank_seed(args.config, rank))
    db = DeviceBatch(w, device=dev)
    stream = torch.cuda.current_stream(dev)
    table0 = db.table_state.clone()          # block table + block counts, one buffer
    tokens_per_step = int(w["cu_nodes"][-1])
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

    flush = _Flush()

    def pre():
        db.table_state.copy_(table0, non_blocking=True)   # allocator refill
        db.tree_build()

    def post():
        db.accept_commit()                   # greedy_accept + kv_commit, one kernel

    def step():
        pre()
        db.attention()
        post()

    sampler = ClockSampler(local) if rank == 0 else None
    if sampler:
        sampler.start()
    side = torch.cuda.Stream(dev)
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        for _ in range(max(3, args.warmup)):
            flush.zero_()
            step()
    stream.wait_stream(side)
    torch.cuda.synchronize()
    depth = db.depth.cpu().numpy()
    st = db.status.cpu().numpy()
    if np.any(st != 0):
        raise RuntimeError(f"bench workload produced status flags {st}")

    # The step's library calls are captured once into one CUDA graph (one graph
    # per tree-size bucket is how a serving loop would run them) and replayed,
    # so the timed region measures the GPU, not Python call overhead. The
    # attention call alone is captured too, to time it in its own loop (an
    # event between the step's grids would split the step into several graph
    # launches, each with its own launch latency).
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
    torch.cuda.synchronize()
    if int(db.status.abs().sum()) != 0:
        raise RuntimeError("graph replay produced status flags")

    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    ev_a = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            for _ in range(args.steps)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    for i in range(args.steps):
        flush.zero_()
        ev[i][0].record(stream)
        g_step.replay()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    # the attention call on its own: the block table as the step leaves it
    # before the commit (refill + tree_build), then flushed replays
    g_pre.replay()
    for i in range(args.steps):
        flush.zero_()
        ev_a[i][0].record(stream)
        g_attn.replay()
        ev_a[i][1].record(stream)
    torch.cuda.synchronize()
    if int(db.status.abs().sum()) != 0:
        raise RuntimeError("attention replay produced status flags")
    clocks = sampler.stop() if sampler else None
    step_ms = float(np.mean([a.elapsed_time(b) for a, b in ev]))
    attn_ms = float(np.mean([a.elapsed_time(b) for a, b in ev_a]))

    # end to end through the public API: host inputs in, results out. The
    # step's inputs (tree, tokens, raw q/k/v) sit in one device buffer and
    # its results in another, so each direction is one copy per step.
    h_in = db.inputs.cpu().pin_memory()
    h_out = torch.empty_like(db.outputs, device="cpu").pin_memory()
    h2d = h_in.numel() * h_in.element_size()
    d2h = h_out.numel() * h_out.element_size()
    e2e_steps = max(3, args.e2e_steps)

    def e2e_loop(run_step):
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(e2e_steps)]
        for i in range(e2e_steps):
            flush.zero_()
            evs[i][0].record(stream)
            db.inputs.copy_(h_in, non_blocking=True)
            run_step()
            h_out.copy_(db.outputs, non_blocking=True)
            evs[i][1].record(stream)
        torch.cuda.synchronize()
        if int(h_out[:4 * int(w["batch"])].view(torch.int32).abs().sum()) != 0:
            raise RuntimeError("end-to-end step produced status flags")
        return float(np.mean([a.elapsed_time(b) for a, b in evs]))

    def graph_step():
        g_step.replay()

    e2e_ms = e2e_loop(graph_step)          # host buffers in/out, graph-replayed API calls
    e2e_eager_ms = e2e_loop(step)          # host buffers in/out, one Python call per API entry

    (step_ms, attn_ms, e2e_ms), tokens_all = reduce_over_ranks(
        [step_ms, attn_ms, e2e_ms], tokens_per_step, world, dev)
    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return

    nbytes, flops = attention_algorithmic(w, depth)
    hbm_peak, tf_peak, src = measured_peaks()
    attn_gbs = nbytes / (attn_ms * 1e-3) / 1e9
    attn_tfs = flops / (attn_ms * 1e-3) / 1e12
    ridge = tf_peak * 1e12 / (hbm_peak * 1e9)
    bound = "hbm" if flops / nbytes < ridge else "tensor"
    roof_s = max(nbytes / (hbm_peak * 1e9), flops / (tf_peak * 1e12))
    if bound == "hbm":
        roof = {"bound": "hbm", "achieved": attn_gbs, "peak": hbm_peak, "unit": "GB/s",
                "frac": attn_gbs / hbm_peak}
    else:
        roof = {"bound": "tensor", "achieved": attn_tfs, "peak": tf_peak, "unit": "TFLOP/s",
                "frac": attn_tfs / tf_peak}
    roof.update(traffic=recorded_traffic(args.config), peak_source=src,
                algorithmic_bytes=nbytes, algorithmic_flops=flops,
                attention_us=attn_ms * 1e3, roofline_us=roof_s * 1e6,
                attention_timing=("the attention call's own loop of graph replays on the step's "
                                  "stream, L2 flushed before each, CUDA events"),
                frac_of_roofline_time=roof_s / (attn_ms * 1e-3),
                frac_of_nominal_8tbs=attn_gbs / 8000.0)
    line = {
        "metric": METRIC, "value": tokens_all / (step_ms * 1e-3), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic", "config": workload_config(w), "roofline": roof,
        "e2e": {"value": tokens_all / (e2e_ms * 1e-3), "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                "mode": "pinned host inputs copied in (one copy), results copied out (one copy), library calls "
                        "replayed from CUDA graphs",
                "eager_value": tokens_all / (e2e_eager_ms * 1e-3),
                "eager_ms_per_step": e2e_eager_ms},
        "gpu_launches": 5 * args.steps,     # tree_build, rope_append, attn_tc, attn_merge, accept_commit
        "attention_tokens_per_s": tokens_all / (attn_ms * 1e-3),
        "clocks": clocks,
    }
    if args.sampling_steps > 0:
        line["sampling"] = measure_sampling(w, dev, stream, flush, args.sampling_steps, hbm_peak)
        line["rejection_acceptance"] = measure_rejection(w, dev, stream, flush,
                                                         args.sampling_steps, hbm_peak)
        line["ddtree_construction"] = measure_ddtree(dev, stream, flush, args.sampling_steps,
                                                     hbm_peak)
        line["eagle_selection"] = measure_eagle(dev, stream, flush, args.sampling_steps)
        line["dense_mask_export"] = measure_dense_mask(w, db, stream, flush, args.sampling_steps,
                                                       hbm_peak)
    if world > 1:
        dist.destroy_process_group()
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, args.cpu_seconds)
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
