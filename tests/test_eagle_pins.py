"""Pins of the EAGLE-2 selection oracle (oracle/eagle_ref.py) to what
"02 · Token Tree 与 Tree Attention" §3/§5 fixes: the kept set is the N most
probable prefixes and is prefix-closed (checked by brute force over every
prefix-closed subset of small candidate sets: it maximises the summed
survival probability); easy contexts give deep trees and divergent ones wide
trees; and it agrees with the independently written tree generator."""

import itertools

import numpy as np
import pytest

from oracle.eagle_ref import eagle_expand_select_ref, eagle_rerank_ref, eagle_scores_ref
from gen import workloads as wl


def random_candidates(rng, m):
    parent = np.full(m, -1, np.int32)
    for c in range(1, m):
        parent[c] = rng.integers(-1, c)
    logp = np.log(rng.uniform(0.02, 0.98, size=m)).astype(np.float32)
    return logp, parent, np.arange(m, dtype=np.int32) + 100


@pytest.mark.parametrize("seed", range(6))
def test_top_n_maximises_survival_mass_over_prefix_closed_sets(seed):
    rng = np.random.default_rng(seed)
    m = 9
    logp, parent, token = random_candidates(rng, m)
    score, depth = eagle_scores_ref(logp, parent)
    mass = np.exp(score.astype(np.float64))
    for n in (1, 3, 5, 9):
        st, par, tok, kept = eagle_rerank_ref(logp, parent, token, n)
        assert st == 0
        best = max(sum(mass[list(sub)])
                   for sub in itertools.combinations(range(m), n)
                   if all(parent[c] < 0 or parent[c] in sub for c in sub))
        assert abs(mass[kept].sum() - best) < 1e-9
        # breadth-first packing: parents before children, depths non-decreasing
        d = np.zeros(n + 1, int)
        for i in range(1, n + 1):
            assert 0 <= par[i] < i
            d[i] = d[par[i]] + 1
        assert np.all(np.diff(d) >= 0)


def test_deep_for_easy_contexts_wide_for_divergent_ones():
    layers, k, n = 6, 4, 12
    rng = np.random.default_rng(0)
    shapes = {}
    for name, top in (("easy", 0.97), ("divergent", 0.26)):
        # every node: the best child has probability `top`, the rest share 1 - top
        logp, parent, token = [], [], []
        frontier = [-1]
        for lay in range(layers):
            nxt = []
            for p in frontier[:k]:
                probs = [top] + [(1 - top) / (k - 1)] * (k - 1)
                for r in range(k):
                    nxt.append(len(logp))
                    logp.append(np.log(probs[r] * (1 - 1e-3 * rng.random())))
                    parent.append(p)
                    token.append(r)
            frontier = nxt
        st, par, tok, kept = eagle_rerank_ref(np.array(logp, np.float32), np.array(parent),
                                              np.array(token), n)
        d = np.zeros(n + 1, int)
        for i in range(1, n + 1):
            d[i] = d[par[i]] + 1
        shapes[name] = (d.max(), np.bincount(d)[1])
    # easy: the whole depth is used; divergent: every root child is kept and
    # the tree stops at depth 2
    assert shapes["easy"][0] == layers and shapes["divergent"][0] <= 2
    assert shapes["divergent"][1] == k


def test_expand_select_and_worked_rerank():
    # root children A .6, B .3, C .1; A's children .55 / .4; B's child .9
    logp = np.log(np.array([0.6, 0.3, 0.1, 0.55, 0.4, 0.9], np.float64)).astype(np.float32)
    parent = np.array([-1, -1, -1, 0, 0, 1], np.int32)
    token = np.array([1, 2, 3, 4, 5, 6], np.int32)
    assert eagle_expand_select_ref(logp, parent, 1, 2).tolist() == [0, 1]
    assert eagle_expand_select_ref(logp, parent, 2, 2).tolist() == [3, 5]   # .33, .27 (.24 left)
    st, par, tok, kept = eagle_rerank_ref(logp, parent, token, 4, root_token=0)
    # scores: A .6, A-child(4) .33, B .3, B-child(6) .27, A-child(5) .24, C .1
    assert kept.tolist() == [0, 1, 3, 5]
    assert tok.tolist() == [0, 1, 2, 4, 6] and par.tolist() == [-1, 0, 0, 1, 2]


def test_agrees_with_the_tree_generator():
    rng = np.random.default_rng(5)
    for _ in range(10):
        p, t, sc, (lp, par, tok) = wl.eagle_tree(rng, 6, 8, 64, 32000, 2.0, return_candidates=True)
        st, rp, rt, kept = eagle_rerank_ref(lp, par, tok, 64, 0)
        assert st == 0 and np.array_equal(rp, p) and np.array_equal(rt, t)


def test_not_enough_candidates_or_positive_logprob():
    logp = np.array([-0.1, -0.2], np.float32)
    parent = np.array([-1, -1], np.int32)
    assert eagle_rerank_ref(logp, parent, np.array([1, 2]), 3)[0] == 1
    # a positive log-probability puts a child above its parent
    st, *_ = eagle_rerank_ref(np.array([-0.5, -0.9, 0.3], np.float32), np.array([-1, -1, 1]),
                              np.array([1, 2, 3]), 2)
    assert st == 1
