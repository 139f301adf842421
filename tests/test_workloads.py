"""The seeded workload generators: tree-shape facts the pages state
(Medusa node count, DDTree Propositions 2-3 and Lemma 1, EAGLE-2 prefix
closure) and the batch layout invariants the library relies on."""

import itertools
import math

import numpy as np
import pytest

from gen import workloads as wl


def _is_topological(parents):
    return parents[0] == -1 and all(0 <= p < i for i, p in enumerate(parents) if i)


def test_medusa_node_count(golden):
    g = golden("medusa_count.json")
    rng = np.random.default_rng(0)
    for case in g["cases"]:
        parents, tokens = wl.medusa_tree(rng, case["sizes"], 1000)
        assert len(parents) - 1 == case["nodes"]
        assert sum(math.prod(case["sizes"][:k + 1]) for k in range(len(case["sizes"]))) == case["nodes"]
        leaves = [i for i in range(len(parents)) if i not in set(parents.tolist())]
        assert len(leaves) == case["paths"] == math.prod(case["sizes"])
        assert _is_topological(parents.tolist())


def test_eagle_tree_prefix_closed_and_sized():
    rng = np.random.default_rng(1)
    for _ in range(5):
        parents, tokens, scores = wl.eagle_tree(rng, 6, 8, 64, 32000, 2.0)
        assert len(parents) == 65 and _is_topological(parents.tolist())
        depth = [0] * len(parents)
        for i in range(1, len(parents)):
            depth[i] = depth[parents[i]] + 1
            assert scores[i] < scores[parents[i]]
        assert depth == sorted(depth) and max(depth) <= 6
    for n_tree in (16, 32, 64, 128):
        for k in (4, 10):
            parents, _, _ = wl.eagle_tree(rng, 0, k, n_tree, 32000, 2.0, until_count=True)
            assert len(parents) == n_tree + 1 and _is_topological(parents.tolist())


def _brute_top_prefixes(logq, budget):
    length, k = logq.shape
    allp = []
    for d in range(1, length + 1):
        for rho in itertools.product(range(k), repeat=d):
            allp.append((sum(logq[i, r] for i, r in enumerate(rho)), rho))
    allp.sort(key=lambda x: -x[0])
    return allp[:budget]


@pytest.mark.parametrize("seed", range(5))
def test_ddtree_heap_equals_brute_force(seed):
    """Algorithm 1 pops the B most probable prefixes (Prop. 3), in
    non-increasing order, without duplicates, prefix-closed (Prop. 2)."""
    rng = np.random.default_rng(seed)
    length, vocab, budget = 3, 4, 6 + seed * 3
    _, logq = wl.ddtree_marginals(rng, length, vocab, 3.0)
    popped, scores = wl.ddtree_heap(logq, budget)
    brute = _brute_top_prefixes(logq, budget)
    assert sorted(popped) == sorted(r for _, r in brute)
    assert np.allclose(sorted(scores, reverse=True), [s for s, _ in brute])
    assert all(a >= b for a, b in zip(scores, scores[1:]))
    assert len(set(popped)) == len(popped)
    s = set(popped)
    assert all(len(r) == 1 or r[:-1] in s for r in popped)


def test_ddtree_lemma1_topk_suffices():
    """Restricting each depth to its top-K tokens, K = min(B, |V|), does not
    change the top-B set (Lemma 1)."""
    rng = np.random.default_rng(7)
    length, vocab, budget = 3, 6, 4
    toks, logq_full = wl.ddtree_marginals(rng, length, vocab, 3.0)
    full = _brute_top_prefixes(logq_full, budget)
    popped, _ = wl.ddtree_heap(logq_full[:, :budget], budget)
    assert sorted(popped) == sorted(r for _, r in full)


def test_ddtree_tree_packing():
    rng = np.random.default_rng(3)
    parents, tokens, popped = wl.ddtree_tree(rng, 16, 5000, 64, 3.0)
    assert len(parents) == 65 and _is_topological(parents.tolist())
    for i, rho in enumerate(popped, start=1):
        depth = 0
        j = i
        while parents[j] != -1:
            j, depth = parents[j], depth + 1
        assert depth == len(rho)


def test_target_match_rate():
    rng = np.random.default_rng(4)
    parents, tokens = wl.medusa_tree(rng, (4, 3, 2), 32000)
    hits = tries = 0
    for _ in range(300):
        tgt = wl.target_ids_for(rng, parents, tokens, 32000, 0.7)
        for i in range(len(parents)):
            kids = [j for j in range(len(parents)) if parents[j] == i]
            if kids:
                tries += 1
                hits += int(tgt[i] in {int(tokens[j]) for j in kids})
    assert abs(hits / tries - 0.7) < 0.03


@pytest.mark.parametrize("cfg", [1, 2, 3])
def test_batch_layout(cfg):
    w = wl.make_config(cfg, batch=3 if cfg > 1 else None, prompt_scale=0.1 if cfg > 1 else 1.0,
                       cache_fill="zeros")
    bs = w["block_size"]
    cu = w["cu_nodes"]
    for b in range(w["batch"]):
        n = cu[b + 1] - cu[b]
        assert _is_topological(w["parents"][cu[b]:cu[b + 1]].tolist())
        need = -(-(int(w["prompt_len"][b]) + n) // bs)
        assert w["n_blocks"][b] == need
        row = w["block_table"][b]
        assert np.all(row[:need] >= 0) and np.all(row[need:] == -1)
    used = w["block_table"][w["block_table"] >= 0]
    assert len(set(used.tolist())) == used.size and used.max() < w["num_blocks"]
    assert not set(used.tolist()) & set(w["free_blocks"])
    assert w["q"].dtype == np.uint16 and w["q"].shape == (cu[-1], w["num_q_heads"], w["head_dim"])
    expected_nodes = {1: 9, 2: 41, 3: 65}[cfg]
    assert all(cu[b + 1] - cu[b] == expected_nodes for b in range(w["batch"]))
