"""Pins of the rejection-sampling oracle (oracle/rejection_ref.py): the
speculative-sampling rule the page refers to is lossless when the draft tokens
are drawn from q - every emitted token follows the target's conditional
distribution (Monte Carlo against the exact target, 6 sigma); at T = 0 the
walk is the greedy walk along the chosen path; the path is the leaf with the
largest cumulative draft log-probability."""

import numpy as np

from oracle.accept_ref import greedy_accept_ref
from oracle.rejection_ref import chosen_path_ref, rejection_walk_ref


def gumbel(rng, shape):
    u = np.clip(rng.random(shape), 1e-12, 1 - 1e-12)
    return -np.log(-np.log(u))


def softmax(x):
    e = np.exp(x - x.max())
    return e / e.sum()


def test_emitted_tokens_follow_the_target():
    rng = np.random.default_rng(5)
    V = 3
    tgt = {(): rng.normal(0, 1.5, V)}
    drf = {(): rng.normal(0, 1.5, V)}
    for a in range(V):
        tgt[(a,)] = rng.normal(0, 1.5, V)
        drf[(a,)] = rng.normal(0, 1.5, V)
        for b in range(V):
            tgt[(a, b)] = rng.normal(0, 1.5, V)
    n = 60_000
    first = np.zeros(V)
    second = np.zeros((V, V))
    for _ in range(n):
        x1 = rng.choice(V, p=softmax(drf[()]))
        x2 = rng.choice(V, p=softmax(drf[(x1,)]))
        parents = [-1, 0, 1]
        toks = [7, x1, x2]
        tl = np.stack([tgt[()], tgt[(x1,)], tgt[(x1, x2)]])
        dl = np.stack([drf[()], drf[(x1,)], drf[(x1,)]])
        st, acc, bonus, _ = rejection_walk_ref(parents, toks, [0.0, -1.0, -1.0], tl, dl,
                                               rng.random(3), gumbel(rng, (3, V)), 1.0, 4)
        emitted = [toks[i] for i in acc[1:]] + [bonus]
        first[emitted[0]] += 1
        if len(emitted) >= 2:
            second[emitted[0], emitted[1]] += 1
    p1 = softmax(tgt[()])
    assert np.all(np.abs(first / n - p1) < 6 * np.sqrt(p1 * (1 - p1) / n))
    for a in range(V):
        m = second[a].sum()
        pa = softmax(tgt[(a,)])
        assert np.all(np.abs(second[a] / m - pa) < 6 * np.sqrt(pa * (1 - pa) / m) + 1e-12)


def test_greedy_limit_is_the_greedy_walk_on_the_path():
    rng = np.random.default_rng(1)
    V = 50
    parents = [-1, 0, 1, 2, 3]                      # a chain
    toks = [9, 4, 7, 1, 3]
    tl = rng.normal(0, 1, (5, V))
    tl[0, 4] = tl[1, 7] = 9.0                      # the target agrees twice, then not
    dl = rng.normal(0, 1, (5, V))
    st, acc, bonus, _ = rejection_walk_ref(parents, toks, [0, -1, -1, -1, -1], tl, dl,
                                           rng.random(5), gumbel(rng, (5, V)), 0.0, 8)
    targets = np.argmax(tl, axis=1)
    gst, gpath, gbonus = greedy_accept_ref(parents, toks, targets, 8)
    assert st == gst == 0 and acc == gpath and bonus == gbonus == int(np.argmax(tl[2]))


def test_chosen_path_by_cumulative_draft_logprob():
    #        0
    #      /   \
    #     1     2        logp: 1 -> -0.1, 2 -> -0.5
    #    / \     \
    #   3   4     5      3 -> -2.0, 4 -> -1.0, 5 -> -0.6  (leaf scores -2.1, -1.1, -1.1)
    parents = [-1, 0, 0, 1, 1, 2]
    logp = [0.0, -0.1, -0.5, -2.0, -1.0, -0.6]
    assert chosen_path_ref(parents, logp) == [0, 1, 4]     # tie -1.1: smaller index 4
    assert chosen_path_ref([-1], [0.0]) == [0]


def test_zero_mass_tokens():
    """A token the target gives no mass is rejected even when the drafter
    gives it none either (0/0 counts as 0); a token only the drafter rules
    out is accepted whatever the uniform."""
    g = np.zeros((2, 3))
    tl = np.array([[1.0, 0.5, -np.inf], [0.0, 0.0, 0.0]])
    dl = np.array([[0.0, -np.inf, -np.inf], [0.0, 0.0, 0.0]])
    st, acc, bonus, det = rejection_walk_ref([-1, 0], [0, 2], [0, -1], tl, dl, [0.5, 0.0], g,
                                             1.0, 4)
    assert st == 0 and acc == [0] and det["ratios"][0][1] == 0.0
    assert bonus == 1                      # residual max(0, p - q) has mass on token 1 only
    st, acc, bonus, det = rejection_walk_ref([-1, 0], [0, 1], [0, -1], tl, dl, [0.5, 0.999],
                                             g, 1.0, 4)
    assert st == 0 and acc == [0, 1] and det["ratios"][0][1] == np.inf
    # greedy: a token other than the argmax is rejected even with q(x) = 0
    st, acc, bonus, _ = rejection_walk_ref([-1, 0], [0, 1], [0, -1], tl, dl, [0.5, 0.0], g,
                                           0.0, 4)
    assert acc == [0] and bonus == 0
