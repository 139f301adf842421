"""Rejection-sampling verification oracle (test infrastructure only: imported
by tests/, never by the product path).

Definitions followed, "02 · Token Tree 与 Tree Attention" §4: the target's
one forward gives logits p at every tree node; acceptance runs from the root
edge by edge with the min(1, p/q) rule (greedy compares token ids); in
practice one best path is chosen first (for example by path log-probability)
and accepted left to right, since the output keeps one chain; when an edge is
rejected a correction token is sampled at the current node, and when the
whole path is accepted the bonus token is sampled at the last node's next
position. "解码：采样、束搜索和推测性解码" ("Gumbel Max技巧") gives the
sampler: argmax_v (log w_v + g_v) draws from w / sum(w).

Readings where the pages leave a step open:
  * the path goes from the root to the leaf with the largest cumulative draft
    log-probability (sum of the draft log-probabilities of its tokens), the
    smallest node index on ties, a NaN sum counting as -inf;
  * the target distribution at node u is p_u = softmax(h_u / T) (T == 0:
    all mass on the first argmax), the draft distribution q_u = softmax(d_u)
    over the drafter's logits at u (the distribution u's children were
    drawn from);
  * edge u -> c is accepted when r_c < p_u(x_c) / q_u(x_c) (r_c ~ U(0, 1), one
    per node, given as input); a token the target gives no mass is never
    accepted (0/0 counts as 0), one the drafter gives none but the target
    some always is;
  * the correction after a rejection at u is drawn from the residual
    max(0, p_u - q_u) (the lossless choice of the speculative-sampling rule
    the page refers to; when the residual is zero everywhere, from p_u), with
    the node's Gumbel noise row; the bonus after a fully accepted path is
    drawn from p at the last node the same way;
  * arithmetic in float64 here; the CUDA kernel works in float32, so a
    decision can differ only when the oracle's margin is within float32
    rounding (the tests check any difference is such a near tie).
"""

import numpy as np


def chosen_path_ref(parents, draft_logp):
    """Root-to-leaf path with the largest cumulative draft log-probability."""
    n = len(parents)
    score = np.zeros(n)
    has_child = np.zeros(n, bool)
    for i in range(1, n):
        score[i] = score[parents[i]] + float(draft_logp[i])
        has_child[parents[i]] = True
    leaves = [i for i in range(n) if not has_child[i]]
    key = np.where(np.isnan(score), -np.inf, score)
    best = max(leaves, key=lambda i: (key[i], -i))
    path = [best]
    while path[-1] != 0:
        path.append(int(parents[path[-1]]))
    return path[::-1]


def _target_probs(h, temperature):
    h = np.asarray(h, np.float64)
    if temperature == 0:
        p = np.zeros_like(h)
        p[int(np.argmax(h))] = 1.0
        return p
    x = h / temperature
    e = np.exp(x - x.max())
    return e / e.sum()


def _softmax(d):
    d = np.asarray(d, np.float64)
    e = np.exp(d - d.max())
    return e / e.sum()


def _gumbel_draw(w, g):
    """argmax_v log w_v + g_v over w_v > 0 (first index on ties)."""
    w = np.asarray(w, np.float64)
    with np.errstate(divide="ignore"):
        key = np.where(w > 0, np.log(w) + np.asarray(g, np.float64), -np.inf)
    return int(np.argmax(key)), key


def rejection_walk_ref(parents, draft_tokens, draft_logp, target_logits, draft_logits,
                       uniforms, gumbel, temperature, max_depth):
    """Returns (status, accepted path as local node indices from the root,
    bonus token, details) for one request; status 16 when the accepted path
    is longer than max_depth."""
    path = chosen_path_ref(parents, draft_logp)
    details = {"path": path, "ratios": [], "stop": None}
    accepted = [0]
    for k in range(1, len(path)):
        u, c = path[k - 1], path[k]
        p = _target_probs(target_logits[u], temperature)
        q = _softmax(draft_logits[u])
        x = int(draft_tokens[c])
        if p[x] == 0:
            ratio = 0.0
        elif q[x] == 0:
            ratio = np.inf
        else:
            ratio = p[x] / q[x]
        details["ratios"].append((float(uniforms[c]), float(ratio)))
        if float(uniforms[c]) < ratio:
            accepted.append(c)
            continue
        res = np.maximum(p - q, 0.0)
        w = res if res.sum() > 0 else p
        tok, key = _gumbel_draw(w, gumbel[u])
        details["stop"] = (u, key)
        break
    else:
        last = path[-1]
        tok, key = _gumbel_draw(_target_probs(target_logits[last], temperature), gumbel[last])
        details["stop"] = (last, key)
    if len(accepted) - 1 > max_depth:
        return 16, accepted, tok, details
    return 0, accepted, tok, details
