"""Pins of the sampling-acceptance oracle (oracle/sample_ref.py) to facts that
do not come from the oracle: the Gumbel-max theorem ("解码：采样、束搜索和推测性
解码", "Gumbel Max技巧"), the greedy limit, and the lossless verifier walk of
"Accelerating Speculative Decoding with Block Diffusion Draft Trees" §7.3
(checked by exhaustive enumeration of the target's autoregressive
distribution on a toy tree against Monte Carlo runs of the walk)."""

import itertools

import numpy as np

from oracle.sample_ref import sample_tokens_ref, sampled_walk_ref


def gumbel(rng, shape):
    u = rng.random(shape)
    u = np.clip(u, 1e-12, 1.0 - 1e-12)
    return (-np.log(-np.log(u))).astype(np.float32)


def softmax(h):
    e = np.exp(h - h.max())
    return e / e.sum()


def test_gumbel_argmax_follows_softmax():
    rng = np.random.default_rng(7)
    h = np.array([0.3, -1.2, 2.0, 0.0, 1.1], dtype=np.float32)
    n = 200_000
    for temp in (1.0, 0.5, 2.0):
        picks = sample_tokens_ref(np.broadcast_to(h, (n, h.size)), gumbel(rng, (n, h.size)), temp)
        freq = np.bincount(picks, minlength=h.size) / n
        want = softmax(h.astype(np.float64) / temp)
        sigma = np.sqrt(want * (1 - want) / n)
        assert np.all(np.abs(freq - want) < 6 * sigma + 1e-12), (temp, freq, want)


def test_zero_temperature_is_argmax_with_first_index_ties():
    h = np.array([[1.0, 3.0, 3.0, -2.0], [0.0, 0.0, 0.0, 0.0], [-5.0, -1.0, -3.0, -1.0]], dtype=np.float32)
    g = np.full(h.shape, 100.0, dtype=np.float32)        # ignored at T = 0
    assert sample_tokens_ref(h, g, 0.0).tolist() == [1, 0, 1]


def test_sampling_is_float32_scale_then_add():
    # the decision is x = fl(fl(h * fl(1/T)) + g); a case where an fp64
    # evaluation would pick the other entry pins the precision and order
    h = np.array([[16777216.0, 16777217.0]], dtype=np.float32)   # 2^24: the second rounds to 2^24
    g = np.array([[1.0, 0.0]], dtype=np.float32)
    # float32: h = [2^24, 2^24]; x = [2^24 + 1 -> 2^24, 2^24] -> tie -> index 0
    assert sample_tokens_ref(h, g, 1.0).tolist() == [0]


def toy_target(vocab, depth, seed):
    """A target's next-token logits for every prefix of length <= depth."""
    rng = np.random.default_rng(seed)
    table = {}
    for k in range(depth + 1):
        for prefix in itertools.product(range(vocab), repeat=k):
            table[prefix] = rng.normal(0.0, 1.5, vocab).astype(np.float32)
    return table


def test_walk_is_lossless_against_autoregressive_sampling():
    vocab, temp = 3, 1.0
    # tree (root = node 0, its token is the previous bonus and not part of the
    # output): node 1 token 0, node 2 token 1 (children of the root); node 3
    # token 2 and node 4 token 0 under node 1
    parents = [-1, 0, 0, 1, 1]
    tokens = [9, 0, 1, 2, 0]
    paths = {0: (), 1: (0,), 2: (1,), 3: (0, 2), 4: (0, 0)}
    target = toy_target(vocab, 2, seed=3)
    logits = np.stack([target[paths[i]] for i in range(5)])
    children = {0: {0: 1, 1: 2}, 1: {2: 3, 0: 4}, 2: {}, 3: {}, 4: {}}

    # exact: sample from the target's conditionals until the first token that
    # is not a child of the current node; output = accepted tokens + that token
    exact = {}

    def expand(node, prefix, prob):
        p = softmax(target[prefix].astype(np.float64) / temp)
        for t in range(vocab):
            if t in children[node]:
                expand(children[node][t], prefix + (t,), prob * p[t])
            else:
                exact[prefix + (t,)] = exact.get(prefix + (t,), 0.0) + prob * p[t]

    expand(0, (), 1.0)
    assert abs(sum(exact.values()) - 1.0) < 1e-12

    rng = np.random.default_rng(11)
    n = 60_000
    counts = {}
    for _ in range(n):
        st, path, bonus = sampled_walk_ref(parents, tokens, logits, gumbel(rng, logits.shape), temp, 4)
        out = tuple(tokens[i] for i in path[1:]) + (bonus,)
        counts[out] = counts.get(out, 0) + 1
    assert set(counts) <= set(exact)
    for seq, p in exact.items():
        f = counts.get(seq, 0) / n
        assert abs(f - p) < 6 * np.sqrt(p * (1 - p) / n) + 1e-9, (seq, f, p)
