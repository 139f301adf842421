"""Pins of the DDTree construction oracle (oracle/ddtree_ref.py) to what
"Accelerating Speculative Decoding with Block Diffusion Draft Trees" fixes:
the §6 worked example's flattened tree, Proposition 2 (the top-B prefixes are
prefix-closed and optimal) and Lemma 1 (per-depth top-K suffices) by brute
force over every prefix, Proposition 3 (pops come out in score order, each
tuple once), and log-probabilities against scipy's log_softmax."""

import itertools

import numpy as np
import pytest
from scipy.special import log_softmax

from oracle.ddtree_ref import ddtree_build_ref, ddtree_from_logits_ref, topk_logprobs_ref


def prefixes_of(parents, tokens):
    """Token prefix (tuple) of every non-root node."""
    out = []
    for i in range(1, len(parents)):
        seq, j = [], i
        while j > 0:
            seq.append(int(tokens[j]))
            j = int(parents[j])
        out.append(tuple(reversed(seq)))
    return out


def test_worked_example_flattening():
    # §6 prints the flattened tree [b, A, B, B, A, B, C] with position ids
    # [0, 1, 1, 2, 2, 2, 3] for vocabulary {A, B, C, D}, L = 3, B = 6, but not
    # the marginals; these marginals give that tree (by hand: the six largest
    # prefixes are A .6, AB .30, B .28, ABC .21, AA .18, BB .14; next AAC .126)
    q = np.array([[0.60, 0.28, 0.07, 0.05],
                  [0.30, 0.50, 0.10, 0.10],
                  [0.10, 0.10, 0.70, 0.10]])
    parents, toks, depths, scores, pops = ddtree_from_logits_ref(np.log(q).astype(np.float32), 6,
                                                                 root_token=9)
    A, B, C = 0, 1, 2
    assert toks.tolist() == [9, A, B, B, A, B, C]
    assert depths.tolist() == [0, 1, 1, 2, 2, 2, 3]
    assert parents.tolist() == [-1, 0, 0, 1, 1, 2, 3]
    np.testing.assert_allclose(np.exp(scores[1:]), [0.6, 0.28, 0.30, 0.18, 0.14, 0.21], rtol=1e-6)
    # pop order: A, AB, B, ABC, AA, BB
    assert pops == [(1,), (1, 1), (2,), (1, 1, 1), (1, 2), (2, 1)]


@pytest.mark.parametrize("seed,L,V,B", [(0, 3, 5, 7), (1, 3, 5, 30), (2, 4, 3, 40), (3, 2, 6, 4),
                                        (4, 3, 4, 1), (5, 1, 7, 7), (6, 3, 6, 3)])
def test_top_b_equals_brute_force(seed, L, V, B):
    """Top-B over every prefix of every token (no top-K cut) equals the heap's
    tree: Proposition 2 (prefix-closed, optimal) and Lemma 1 (K = min(B, V)
    loses nothing)."""
    rng = np.random.default_rng(seed)
    logits = rng.normal(0, 2.0, size=(L, V)).astype(np.float32)
    lq = log_softmax(logits.astype(np.float64), axis=1)
    allp = []
    for d in range(1, L + 1):
        for seq in itertools.product(range(V), repeat=d):
            s = 0.0
            for i, t in enumerate(seq):
                s += lq[i, t]
            allp.append((s, seq))
    allp.sort(key=lambda z: -z[0])
    want = {seq for _, seq in allp[:B]}
    parents, toks, depths, scores, pops = ddtree_from_logits_ref(logits, B)
    got = prefixes_of(parents, toks)
    assert len(got) == min(B, len(allp)) and set(got) == want
    for p in got:                                   # prefix-closed
        assert len(p) == 1 or p[:-1] in want
    # Proposition 3: non-increasing pop scores, no tuple popped twice
    assert len(set(pops)) == len(pops)
    lq_k = topk_logprobs_ref(logits, B)[1]
    seq_scores = []
    for rho in pops:
        s = 0.0
        for i, r in enumerate(rho):
            s += lq_k[i, r - 1]
        seq_scores.append(s)
    assert all(seq_scores[i] >= seq_scores[i + 1] - 1e-12 for i in range(len(seq_scores) - 1))
    # depth-major flattening: depths non-decreasing, parents earlier
    assert np.all(np.diff(depths) >= 0) and np.all(parents[1:] < np.arange(1, len(parents)))
    assert np.all(depths[1:] == depths[parents[1:]] + 1)


def test_equal_scores_break_by_depth_then_parent_then_rank():
    # uniform marginals: every prefix of one depth has the same score
    logq = np.full((2, 3), -np.log(3.0))
    toks = np.array([[5, 6, 7], [8, 9, 10]])
    parents, t, depths, scores, pops = ddtree_build_ref(logq, toks, 5)
    assert pops == [(1,), (2,), (3,), (1, 1), (1, 2)]
    assert t.tolist() == [-1, 5, 6, 7, 8, 9] and parents.tolist() == [-1, 0, 0, 0, 1, 1]


def test_budget_larger_than_all_prefixes():
    logq = np.log(np.array([[0.7, 0.3], [0.6, 0.4]]))
    toks = np.array([[0, 1], [0, 1]])
    parents, t, depths, scores, pops = ddtree_build_ref(logq, toks, 100)
    assert len(pops) == 2 + 4 and len(set(pops)) == 6


def test_topk_logprobs_against_scipy_and_ties():
    rng = np.random.default_rng(11)
    h = rng.normal(0, 3.0, size=(4, 1000)).astype(np.float32)
    h[1, [10, 20, 30]] = 50.0                       # exact ties at the top
    h[2, :500] = -np.inf                            # masked half
    toks, lq = topk_logprobs_ref(h, 64)
    ref = log_softmax(h.astype(np.float64), axis=1)
    for r in range(4):
        assert np.allclose(lq[r], ref[r, toks[r]], rtol=0, atol=1e-12)
        vals = h[r, toks[r]]
        assert np.all(np.diff(vals.astype(np.float64)) <= 0)
        brk = np.diff(vals.astype(np.float64)) == 0
        assert np.all(np.diff(toks[r])[brk] > 0)    # equal logits: token ascending
        assert set(toks[r]) == set(np.argsort(-h[r].astype(np.float64), kind="stable")[:64])
    assert toks[1, :3].tolist() == [10, 20, 30]
    assert np.all(toks[2] >= 500)
    full_t, full_lq = topk_logprobs_ref(h[:1], 1000)
    assert abs(np.exp(full_lq[0]).sum() - 1.0) < 1e-12
    dead = np.full((1, 8), -np.inf, np.float32)
    t, l = topk_logprobs_ref(dead, 4)
    assert t.tolist() == [[0, 1, 2, 3]] and np.all(l == -np.inf)
