"""Seeded synthetic workloads for the token-tree verification step.

This module only makes inputs: candidate trees (parent lists), draft and
target token ids, bf16 Q/K/V drawn from N(0, 1), prompt lengths and a paged KV
pool with a shuffled block table. It holds none of the step's arithmetic (no
masks, RoPE, attention, acceptance or commit), so both the CUDA path and the
CPU oracle can be fed from it.

Tree shapes follow the proposal methods the pages describe:
  * Medusa cartesian trees - "02 · Token Tree 与 Tree Attention", §3: head k
    contributes its top-s_k tokens under every depth-(k-1) node.
  * EAGLE-2 dynamic trees - same page §3 and §5: each layer expands the top-k
    nodes of the previous layer by cumulative (prefix survival) log-probability
    and the global top-N nodes are kept.
  * DDTree trees - "Accelerating Speculative Decoding with Block Diffusion
    Draft Trees", §4-§5: factorised per-position marginals, per-depth top-K
    (Lemma 1) and a best-first heap over rank tuples (Algorithm 1) that pops
    the B most probable prefixes.

Readings where the workload descriptions are silent: N(0, s) means standard
deviation s; "the target matches the draft child with probability p" means a
node with children gets, with probability p, the token of a uniformly chosen
child as its target id, otherwise a uniform id (leaves always get a uniform
id); ties in the tree selections go to the shallower node, then the earlier
generated one.
"""

from __future__ import annotations

import concurrent.futures
import heapq
import math
import os
from dataclasses import dataclass

import numpy as np
import torch

VOCAB_LLAMA = 32000
VOCAB_QWEN = 151936


def bf16_bits_from_f32(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (torch's round-to-nearest-even) and return
    the uint16 bit patterns."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def normal_bf16(rng: np.random.Generator, shape, chunk=1 << 24) -> np.ndarray:
    """bf16 bit patterns of N(0, 1) draws, generated in chunks to bound memory.

    Up to one chunk comes from ``rng`` itself. Larger arrays (the paged KV
    pools) are split into chunks of their own seeded streams - chunk i draws
    from a generator seeded with (one draw of ``rng``, i) - and generated on
    several threads; the result depends only on ``rng``'s state, not on the
    thread count."""
    total = int(np.prod(shape))
    out = np.empty(total, dtype=np.uint16)
    if total <= chunk:
        out[:] = bf16_bits_from_f32(rng.standard_normal(total, dtype=np.float32))
        return out.reshape(shape)
    base = int(rng.integers(0, 2 ** 62))

    def fill(i):
        s, e = i * chunk, min(total, (i + 1) * chunk)
        g = np.random.default_rng([base, i])
        out[s:e] = bf16_bits_from_f32(g.standard_normal(e - s, dtype=np.float32))

    n = -(-total // chunk)
    with concurrent.futures.ThreadPoolExecutor(max_workers=min(16, os.cpu_count() or 1, n)) as ex:
        list(ex.map(fill, range(n)))
    return out.reshape(shape)


# --------------------------------------------------------------------------
# tree shapes


def medusa_tree(rng, sizes, vocab):
    """Cartesian Medusa tree in BFS order: returns (parents, tokens) without
    the root's token (node 0 is the root; tokens[0] is filled by the caller)."""
    parents, tokens = [-1], [0]
    frontier = [0]
    for s in sizes:
        head_tokens = rng.choice(vocab, size=s, replace=False)
        nxt = []
        for p in frontier:
            for t in head_tokens:
                parents.append(p)
                tokens.append(int(t))
                nxt.append(len(parents) - 1)
        frontier = nxt
    return np.array(parents, np.int32), np.array(tokens, np.int32)


def _topk_logprobs(rng, vocab, k, sigma):
    logits = rng.standard_normal(vocab) * sigma
    m = logits.max()
    lse = m + math.log(np.exp(logits - m).sum())
    idx = np.argpartition(-logits, k - 1)[:k]
    idx = idx[np.lexsort((idx, -logits[idx]))]        # descending, ties by id
    return idx.astype(np.int64), logits[idx] - lse


def eagle_tree(rng, depth, topk, keep, vocab, sigma=2.0, until_count=False,
               max_layers=32, return_candidates=False):
    """EAGLE-2 style dynamic tree.

    Layer 1 is the root's top-k children; layer l expands the top-k nodes of
    layer l-1 (by cumulative log-prob) with their own top-k children. With
    ``until_count`` layers are added until at least ``keep`` candidates exist
    (at most ``max_layers``) instead of exactly ``depth`` layers. The global
    top-``keep`` candidates by cumulative score are kept (prefix-closed because
    every child scores strictly below its parent) and packed in BFS order.
    Returns (parents, tokens, scores) with node 0 the root; with
    ``return_candidates`` also (logp, parent, token) of every generated
    candidate in generation order (parent -1 for the root's children).
    """
    # candidate: (score, depth, gen, parent_gen, rank, token)
    cands = []
    toks, lps = _topk_logprobs(rng, vocab, topk, sigma)
    layer = []
    for r in range(topk):
        c = (float(lps[r]), 1, len(cands), -1, r, int(toks[r]))
        cands.append(c)
        layer.append(c)
    n_layers = 1
    while True:
        if until_count:
            if len(cands) >= keep or n_layers >= max_layers:
                break
        elif n_layers >= depth:
            break
        best = sorted(layer, key=lambda c: (-c[0], c[2]))[:topk]
        layer = []
        for pc in best:
            toks, lps = _topk_logprobs(rng, vocab, topk, sigma)
            for r in range(topk):
                c = (pc[0] + float(lps[r]), pc[1] + 1, len(cands), pc[2], r, int(toks[r]))
                cands.append(c)
                layer.append(c)
        n_layers += 1
    kept = sorted(cands, key=lambda c: (-c[0], c[1], c[2]))[:keep]
    kept_gen = {c[2] for c in kept}
    for c in kept:
        if c[3] != -1 and c[3] not in kept_gen:
            raise AssertionError("eagle_tree selection is not prefix-closed")
    # BFS packing: by depth, then parent's packed index, then child rank.
    packed_of = {-1: 0}
    order = []
    for dpt in range(1, max(c[1] for c in kept) + 1):
        level = [c for c in kept if c[1] == dpt]
        level.sort(key=lambda c: (packed_of[c[3]], c[4]))
        for c in level:
            packed_of[c[2]] = len(order) + 1
            order.append(c)
    parents = [-1] + [packed_of[c[3]] for c in order]
    tokens = [0] + [c[5] for c in order]
    scores = [0.0] + [c[0] for c in order]
    out = (np.array(parents, np.int32), np.array(tokens, np.int32), np.array(scores))
    if return_candidates:
        logp = np.array([c[0] - (cands[c[3]][0] if c[3] >= 0 else 0.0) for c in cands])
        out += ((logp, np.array([c[3] for c in cands], np.int32),
                 np.array([c[5] for c in cands], np.int32)),)
    return out


def eagle_candidates(rng, layers, topk, vocab, sigma=2.0, chooser=None):
    """Candidates of an EAGLE-style expansion, in generation order: layer 1 is
    the root's top-k children (drafter log-probs from log_softmax of N(0,
    sigma) logits); each later layer gives top-k children to the layer nodes
    named by ``chooser(logp, parent, layer)`` (default: the first topk nodes
    of the layer, generation order). Returns (logp float32, parent, token)."""
    logp, parent, token = [], [], []
    toks, lps = _topk_logprobs(rng, vocab, topk, sigma)
    layer_nodes = []
    for r in range(topk):
        layer_nodes.append(len(logp))
        logp.append(lps[r]); parent.append(-1); token.append(int(toks[r]))
    for lay in range(1, layers):
        lp = np.array(logp, np.float32)
        par = np.array(parent, np.int32)
        chosen = chooser(lp, par, lay) if chooser is not None else layer_nodes[:topk]
        layer_nodes = []
        for pc in chosen:
            toks, lps = _topk_logprobs(rng, vocab, topk, sigma)
            for r in range(topk):
                layer_nodes.append(len(logp))
                logp.append(lps[r]); parent.append(int(pc)); token.append(int(toks[r]))
    return (np.array(logp, np.float32), np.array(parent, np.int32), np.array(token, np.int32))


def ddtree_marginals(rng, length, vocab, sigma=3.0, k=None):
    """Per-position drafter marginals softmax(N(0, sigma) logits).

    Returns (top_tokens [L, K], top_logq [L, K]) holding the K most probable
    tokens per position in descending probability (Lemma 1 of the DDTree notes:
    only the per-depth top-K tokens, K = min(B, |V|), can appear in an optimal
    tree)."""
    k = vocab if k is None else min(k, vocab)
    toks = np.zeros((length, k), np.int64)
    logq = np.zeros((length, k))
    for i in range(length):
        t, lp = _topk_logprobs(rng, vocab, k, sigma)
        toks[i], logq[i] = t, lp
    return toks, logq


def ddtree_heap(logq, budget):
    """Best-first enumeration of the ``budget`` most probable prefixes over
    rank tuples (Algorithm 1 of the DDTree notes, §5).

    logq [L, K]: per-position log-probabilities sorted descending. Ranks are
    0-based here. Returns the popped rank tuples in pop order and their scores.
    Ties pop the shallower tuple first, then the lexicographically smaller one.
    """
    length, k = logq.shape
    heap = [(-logq[0, 0], 1, (0,))]
    popped, scores = [], []
    while heap and len(popped) < budget:
        neg, _, rho = heapq.heappop(heap)
        score = -neg
        popped.append(rho)
        scores.append(score)
        d = len(rho)
        last = rho[-1]
        if last + 1 < k:                               # next sibling
            sib = rho[:-1] + (last + 1,)
            s = score - logq[d - 1, last] + logq[d - 1, last + 1]
            heapq.heappush(heap, (-s, d, sib))
        if d < length:                                 # first child
            child = rho + (0,)
            heapq.heappush(heap, (-(score + logq[d, 0]), d + 1, child))
    return popped, scores


def ddtree_tree(rng, length, vocab, budget, sigma=3.0):
    """DDTree: (parents, tokens, rank_tuples) with node 0 the root and the
    popped prefixes packed in pop order (parents always precede children)."""
    toks, logq = ddtree_marginals(rng, length, vocab, sigma, k=budget)
    popped, _ = ddtree_heap(logq, budget)
    index = {(): 0}
    parents, tokens = [-1], [0]
    for rho in popped:
        index[rho] = len(parents)
        parents.append(index[rho[:-1]])
        tokens.append(int(toks[len(rho) - 1, rho[-1]]))
    return np.array(parents, np.int32), np.array(tokens, np.int32), popped


def target_ids_for(rng, parents, tokens, vocab, p_match):
    """Synthetic per-node target (greedy) ids: with probability ``p_match`` a
    node with children points at a uniformly chosen child's token."""
    n = len(parents)
    children = [[] for _ in range(n)]
    for j in range(1, n):
        children[int(parents[j])].append(j)
    tgt = rng.integers(0, vocab, size=n).astype(np.int32)
    for i in range(n):
        if children[i] and rng.random() < p_match:
            tgt[i] = tokens[children[i][int(rng.integers(len(children[i])))]]
    return tgt


def _fill_gumbel(rng, out):
    """Fill a C-contiguous float32 array with Gumbel(0, 1) draws g = -log(E),
    E ~ Exp(1) (the same law as -log(-log(u)), u ~ U(0, 1)); E is kept above
    1e-30 so g stays finite."""
    rng.standard_exponential(dtype=np.float32, out=out)
    np.maximum(out, np.float32(1e-30), out=out)
    np.log(out, out=out)
    np.negative(out, out=out)


def gumbel_noise(rng, shape) -> np.ndarray:
    """float32 Gumbel(0, 1) noise of the given shape."""
    out = np.empty(shape, np.float32)
    _fill_gumbel(rng, out)
    return out


def sampling_inputs(rng, w, vocab=None, sigma=1.0, boost=(8.0, 16.0), ld=None,
                    pad_value=np.nan):
    """Per-node target logits and Gumbel noise for the sampled walk.

    logits[t] ~ N(0, sigma) over the vocabulary; with the workload's match
    probability a node with children gets a uniformly chosen child's token
    raised by a boost drawn from U(boost), so the sampled token is that child
    often but not always. Rows have ``ld`` >= vocab columns; the columns past
    the vocabulary hold ``pad_value`` (NaN by default: a reader that strays
    there would pick it). Returns (logits, gumbel), float32 [T][ld]."""
    vocab = w["vocab"] if vocab is None else vocab
    ld = vocab if ld is None else ld
    cu = w["cu_nodes"]
    total = int(cu[-1])
    logits = np.empty((total, ld), np.float32)
    gumbel = np.empty((total, ld), np.float32)

    def rows(a):          # C-contiguous pieces covering a[:, :vocab]
        if ld == vocab:
            yield a.reshape(-1)
        else:
            for r in range(total):
                yield a[r, :vocab]

    for piece in rows(logits):
        rng.standard_normal(dtype=np.float32, out=piece)
        if sigma != 1.0:
            piece *= np.float32(sigma)
    for b in range(w["batch"]):
        t0, t1 = int(cu[b]), int(cu[b + 1])
        par = w["parents"][t0:t1]
        tok = w["draft_tokens"][t0:t1]
        children = [[] for _ in range(t1 - t0)]
        for j in range(1, t1 - t0):
            children[int(par[j])].append(j)
        for i in range(t1 - t0):
            if children[i] and rng.random() < w["p_match"]:
                c = children[i][int(rng.integers(len(children[i])))]
                if int(tok[c]) < vocab:
                    logits[t0 + i, int(tok[c])] += np.float32(rng.uniform(*boost))
    for piece in rows(gumbel):
        _fill_gumbel(rng, piece)
    if ld > vocab:
        logits[:, vocab:] = pad_value
        gumbel[:, vocab:] = pad_value
    return logits, gumbel


def rejection_inputs(rng, w, vocab=None, draft_sigma=1.0, draft_boost=(4.0, 10.0), tau=0.5,
                     ld=None, pad_value=np.nan):
    """Inputs of the rejection-sampling walk: the drafter's logits at every
    node, the target's, Gumbel noise, uniforms and draft log-probabilities.

    draft[t] ~ N(0, draft_sigma) with every child's token raised by a boost
    drawn from U(draft_boost) (the children are the drafter's likely tokens);
    the target's row is the drafter's plus N(0, tau) noise (a drafter that
    approximates the target); draft_logp[t] is the drafter's reported
    log-probability of node t's token, drawn as -Exp(1) (the root's entry is
    0 and unused); uniforms[t] ~ U(0, 1) in float32. Rows have ``ld`` >=
    vocab columns, the ones past the vocabulary hold ``pad_value``. Returns
    (logits, draft, gumbel, uniforms, draft_logp)."""
    vocab = w["vocab"] if vocab is None else vocab
    ld = vocab if ld is None else ld
    cu = w["cu_nodes"]
    total = int(cu[-1])
    draft = np.empty((total, ld), np.float32)
    logits = np.empty((total, ld), np.float32)
    gumbel = np.empty((total, ld), np.float32)
    noise = np.empty(vocab, np.float32)
    for r in range(total):
        rng.standard_normal(dtype=np.float32, out=draft[r, :vocab])
        if draft_sigma != 1.0:
            draft[r, :vocab] *= np.float32(draft_sigma)
    for b in range(w["batch"]):
        t0, t1 = int(cu[b]), int(cu[b + 1])
        par = w["parents"][t0:t1]
        tok = w["draft_tokens"][t0:t1]
        for j in range(1, t1 - t0):
            if 0 <= int(tok[j]) < vocab:
                draft[t0 + int(par[j]), int(tok[j])] += np.float32(rng.uniform(*draft_boost))
    for r in range(total):
        rng.standard_normal(dtype=np.float32, out=noise)
        noise *= np.float32(tau)
        np.add(draft[r, :vocab], noise, out=logits[r, :vocab])
        _fill_gumbel(rng, gumbel[r, :vocab])
    if ld > vocab:
        for a in (draft, logits, gumbel):
            a[:, vocab:] = pad_value
    draft_logp = (-rng.standard_exponential(total)).astype(np.float32)
    draft_logp[cu[:-1]] = 0.0
    uniforms = rng.random(total, dtype=np.float32)
    return logits, draft, gumbel, uniforms, draft_logp


# --------------------------------------------------------------------------
# batches


@dataclass
class Geometry:
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int = 16
    rope_base: float = 10000.0
    rope_style: int = 0


def assemble(rng, geom: Geometry, prompt_lens, trees, vocab, p_match,
             max_nodes=None, slack_blocks=None, extra_slots=0, cache_fill="normal"):
    """Build one batch.

    trees: list of (parents, tokens) per request (node 0 = root). Returns a
    dict with every array the step consumes (bf16 tensors as uint16 bits).
    ``extra_slots`` reserves block-table room for later steps.
    """
    bsz = len(trees)
    bs = geom.block_size
    counts = [len(t[0]) for t in trees]
    cu = np.zeros(bsz + 1, np.int32)
    cu[1:] = np.cumsum(counts)
    total = int(cu[-1])
    if max_nodes is None:
        max_nodes = max(counts)
    parents = np.concatenate([t[0] for t in trees]).astype(np.int32)
    tokens = np.concatenate([t[1] for t in trees]).astype(np.int32)
    # the root's token is the previous round's bonus token
    for b in range(bsz):
        tokens[cu[b]] = int(rng.integers(0, vocab))
    targets = np.concatenate([
        target_ids_for(rng, trees[b][0], tokens[cu[b]:cu[b + 1]], vocab, p_match)
        for b in range(bsz)]).astype(np.int32)
    plen = np.asarray(prompt_lens, np.int32)
    need = [-(-(int(plen[b]) + counts[b]) // bs) for b in range(bsz)]
    max_blocks = max(-(-(int(plen[b]) + counts[b] + extra_slots) // bs) for b in range(bsz))
    if slack_blocks is None:
        slack_blocks = max(16, sum(need) // 20)
    num_blocks = sum(need) + slack_blocks + bsz * max(0, max_blocks - max(need))
    perm = rng.permutation(num_blocks).astype(np.int32)
    table = np.full((bsz, max_blocks), -1, np.int32)
    used = 0
    for b in range(bsz):
        table[b, :need[b]] = perm[used:used + need[b]]
        used += need[b]
    free = [int(x) for x in perm[used:]]
    hq, hkv, d = geom.num_q_heads, geom.num_kv_heads, geom.head_dim
    pool_shape = (num_blocks, hkv, bs, d)
    if cache_fill == "normal":
        k_cache = normal_bf16(rng, pool_shape)
        v_cache = normal_bf16(rng, pool_shape)
    else:
        k_cache = np.zeros(pool_shape, np.uint16)
        v_cache = np.zeros(pool_shape, np.uint16)
    return {
        "num_q_heads": hq, "num_kv_heads": hkv, "head_dim": d, "block_size": bs,
        "rope_base": geom.rope_base, "rope_style": geom.rope_style,
        "batch": bsz, "max_nodes": int(max_nodes), "max_depth": int(max_nodes) - 1,
        "vocab": vocab, "cu_nodes": cu, "parents": parents, "prompt_len": plen,
        "draft_tokens": tokens, "target_ids": targets,
        "q": normal_bf16(rng, (total, hq, d)),
        "k_new": normal_bf16(rng, (total, hkv, d)),
        "v_new": normal_bf16(rng, (total, hkv, d)),
        "block_table": table, "n_blocks": np.array(need, np.int32),
        "max_blocks_per_req": int(max_blocks), "num_blocks": int(num_blocks),
        "k_cache": k_cache, "v_cache": v_cache, "free_blocks": free,
        "p_match": p_match,
    }


CONFIG_NAMES = {
    1: "tiny: B=1 Hq4/Hkv2/D64 P=7 Medusa 2x3 (9 nodes)",
    2: "llama3-8b-attn B=8 P~U[512,2048] Medusa 4x3x2 (41 nodes)",
    3: "llama3-8b-attn B=32 P~U[1024,8192] EAGLE-2 d6 k8 top-64 (65 nodes)",
    4: "llama3-70b-attn B=16 P~U[2048,4096] DDTree L16 V151936 B256 (257 nodes)",
    5: "llama3-8b-attn B=64 ragged P~logU[4096,32768] random EAGLE N in {16..128}",
}

GEOM_8B = Geometry(32, 8, 128)
GEOM_70B = Geometry(64, 8, 128)
GEOM_TINY = Geometry(4, 2, 64)


def make_config(idx: int, batch=None, seed=None, prompt_scale=1.0, cache_fill="normal"):
    """The five verification workloads (seed 1000 + idx by default).

    ``batch`` and ``prompt_scale`` shrink a workload for quick checks (the
    tree recipe is unchanged)."""
    rng = np.random.default_rng(1000 + idx if seed is None else seed)
    if idx == 1:
        bsz = batch or 1
        trees = [medusa_tree(rng, (2, 3), VOCAB_LLAMA) for _ in range(bsz)]
        plens = [7] * bsz
        return assemble(rng, GEOM_TINY, plens, trees, VOCAB_LLAMA, 0.5,
                        cache_fill=cache_fill) | {"config": 1}
    if idx == 2:
        bsz = batch or 8
        plens = rng.integers(512, 2049, size=bsz)
        trees = [medusa_tree(rng, (4, 3, 2), VOCAB_LLAMA) for _ in range(bsz)]
        geom = GEOM_8B
    elif idx == 3:
        bsz = batch or 32
        plens = rng.integers(1024, 8193, size=bsz)
        trees = [eagle_tree(rng, 6, 8, 64, VOCAB_LLAMA, 2.0)[:2] for _ in range(bsz)]
        geom = GEOM_8B
    elif idx == 4:
        bsz = batch or 16
        plens = rng.integers(2048, 4097, size=bsz)
        trees = [ddtree_tree(rng, 16, VOCAB_QWEN, 256, 3.0)[:2] for _ in range(bsz)]
        geom = GEOM_70B
        plens = (np.asarray(plens) * prompt_scale).astype(np.int64)
        return assemble(rng, geom, plens, trees, VOCAB_QWEN, 0.7,
                        cache_fill=cache_fill) | {"config": 4}
    elif idx == 5:
        bsz = batch or 64
        plens = np.exp(rng.uniform(math.log(4096), math.log(32768), size=bsz)).astype(np.int64)
        trees = []
        for _ in range(bsz):
            n_tree = int(rng.choice([16, 32, 64, 128]))
            k = int(rng.integers(4, 11))
            trees.append(eagle_tree(rng, 0, k, n_tree, VOCAB_LLAMA, 2.0, until_count=True)[:2])
        plens = (np.asarray(plens) * prompt_scale).astype(np.int64)
        return assemble(rng, GEOM_8B, plens, trees, VOCAB_LLAMA, 0.6, max_nodes=129,
                        extra_slots=8 * 130, cache_fill=cache_fill) | {"config": 5}
    else:
        raise ValueError(f"unknown config {idx}")
    plens = (np.asarray(plens) * prompt_scale).astype(np.int64)
    return assemble(rng, geom, plens, trees, VOCAB_LLAMA, 0.7,
                    cache_fill=cache_fill) | {"config": idx}


def next_step_inputs(rng, w, new_len, bonus, trees, p_match=None):
    """Inputs of the following verification step of a multi-step run.

    new_len / bonus come from the previous step's commit; ``trees`` are the new
    candidate trees. The paged pool, block table and free list in ``w`` are the
    post-commit state; blocks for the new tentative slots are taken from
    ``w['free_blocks']`` (front first). Returns a new dict (pool arrays shared).
    """
    bsz = w["batch"]
    bs = w["block_size"]
    vocab = w["vocab"]
    p_match = w["p_match"] if p_match is None else p_match
    counts = [len(t[0]) for t in trees]
    cu = np.zeros(bsz + 1, np.int32)
    cu[1:] = np.cumsum(counts)
    total = int(cu[-1])
    tokens = np.concatenate([t[1] for t in trees]).astype(np.int32)
    for b in range(bsz):
        tokens[cu[b]] = int(bonus[b])
    targets = np.concatenate([
        target_ids_for(rng, trees[b][0], tokens[cu[b]:cu[b + 1]], vocab, p_match)
        for b in range(bsz)]).astype(np.int32)
    table = np.array(w["block_table"], copy=True)
    n_blocks = np.array(w["n_blocks"], copy=True)
    free = list(w["free_blocks"])
    for b in range(bsz):
        need = -(-(int(new_len[b]) + counts[b]) // bs)
        if need > table.shape[1]:
            raise RuntimeError("block table too small for the next step")
        while n_blocks[b] < need:
            table[b, n_blocks[b]] = free.pop(0)
            n_blocks[b] += 1
    hq, hkv, d = w["num_q_heads"], w["num_kv_heads"], w["head_dim"]
    out = dict(w)
    out.update(
        cu_nodes=cu, parents=np.concatenate([t[0] for t in trees]).astype(np.int32),
        prompt_len=np.asarray(new_len, np.int32), draft_tokens=tokens, target_ids=targets,
        q=normal_bf16(rng, (total, hq, d)), k_new=normal_bf16(rng, (total, hkv, d)),
        v_new=normal_bf16(rng, (total, hkv, d)), block_table=table, n_blocks=n_blocks,
        free_blocks=free)
    return out
