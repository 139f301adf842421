"""DDTree draft-tree construction oracle (test infrastructure only: imported
by tests/, never by the product path).

Definitions followed, "Accelerating Speculative Decoding with Block Diffusion
Draft Trees":
  * §3-§4.1: the drafter gives one factorised distribution per position,
    q_i = softmax of that position's logits; a prefix u = (u_1..u_d) has
    q(u) = prod_i q_i(u_i), so its log-score is the sum of the per-position
    log-probabilities.
  * §4.2 (Proposition 2): the B prefixes of largest q are prefix-closed and
    form the optimal tree.
  * §4.3 (Lemma 1): only each depth's top-K tokens, K = min(B, |V|), matter.
  * §5 (Algorithm 1): best-first enumeration over rank tuples with a max-heap
    that starts from (1,), pops the best tuple, and pushes its next sibling
    (last rank + 1, while <= K) and its first child (append rank 1, while the
    depth is below L); B pops give the tree.
  * §6-§7.1: the tree is flattened depth by depth after the root b (position
    id = depth), e.g. [b, A, B, B, A, B, C] with positions [0, 1, 1, 2, 2, 2, 3].

Readings where the pages leave a step open:
  * ranks order a position's tokens by logit descending, equal logits by
    token id ascending;
  * log q_i(v) = h_i(v) - logsumexp(h_i), in float64 here; a position whose
    logits are all -inf gives -inf for every token;
  * a pushed tuple's score is its parent prefix's score plus its own last
    log-probability (the page's sibling update sigma - log q(r) + log q(r+1)
    is the same quantity), summed in float64 from the per-position values
    (the page fixes no precision; float64 is the plain reading of "the sum
    of the log-probabilities");
  * equal scores pop the shallower tuple first, then the one whose parent
    popped earlier, then the smaller last rank;
  * output order: the root, then depth by depth, pop order within a depth;
    parents are indices into that order.
"""

import heapq

import numpy as np


def topk_logprobs_ref(logits, k):
    """Per row: the k top tokens (logit descending, token ascending on ties)
    and their log-probabilities log softmax(h)[token]. logits [rows][V]."""
    h = np.asarray(logits, dtype=np.float32)
    rows, vocab = h.shape
    k = min(k, vocab)
    toks = np.zeros((rows, k), np.int32)
    logq = np.zeros((rows, k), np.float64)
    idx = np.arange(vocab)
    for r in range(rows):
        x = h[r].astype(np.float64)
        order = np.lexsort((idx, -x))[:k]            # primary: -x ascending
        toks[r] = order
        m = np.max(x)
        if not np.isfinite(m):
            logq[r] = -np.inf
            continue
        lse = m + np.log(np.sum(np.exp(x - m)))
        logq[r] = x[order] - lse
    return toks, logq


def ddtree_build_ref(logq, tokens, budget, root_token=-1):
    """Algorithm 1 over rank tuples.

    logq [L][K] per-depth log-probabilities in rank order (any float type; used
    as float64), tokens [L][K] the matching token ids. Returns (parents,
    node_tokens, depths, scores, pops) with node 0 the root; ``pops`` lists the
    popped rank tuples (1-based ranks) in pop order."""
    lq = np.asarray(logq, dtype=np.float64)
    L, K = lq.shape
    # heap entries: (-score, depth, parent pop index, last rank, tuple)
    heap = [(-lq[0, 0], 1, 0, 1, (1,))]
    pop_index = {(): 0}                  # root counts as popped first
    pops, scores = [], []
    while heap and len(pops) < budget:
        neg, d, _, r, rho = heapq.heappop(heap)
        sigma = -neg
        pops.append(rho)
        scores.append(sigma)
        pop_index[rho] = len(pops)
        parent = rho[:-1]
        parent_score = 0.0 if d == 1 else scores[pop_index[parent] - 1]
        if r + 1 <= K:                                   # next sibling
            heapq.heappush(heap, (-(parent_score + lq[d - 1, r]), d, pop_index[parent], r + 1,
                                  parent + (r + 1,)))
        if d < L:                                        # first child
            heapq.heappush(heap, (-(sigma + lq[d, 0]), d + 1, pop_index[rho], 1, rho + (1,)))
    # flatten: root, then by depth, pop order within a depth
    order = sorted(range(len(pops)), key=lambda j: (len(pops[j]), j))
    slot = {(): 0}
    for new, j in enumerate(order, start=1):
        slot[pops[j]] = new
    n = len(pops) + 1
    parents = np.full(n, -1, np.int32)
    node_tokens = np.full(n, root_token, np.int32)
    depths = np.zeros(n, np.int32)
    node_scores = np.zeros(n, np.float64)
    for j in order:
        rho = pops[j]
        s = slot[rho]
        parents[s] = slot[rho[:-1]]
        node_tokens[s] = tokens[len(rho) - 1][rho[-1] - 1]
        depths[s] = len(rho)
        node_scores[s] = scores[j]
    return parents, node_tokens, depths, node_scores, pops


def ddtree_from_logits_ref(logits, budget, root_token=-1):
    """The whole construction for one request: logits [L][V] -> tree."""
    toks, logq = topk_logprobs_ref(logits, budget)
    return ddtree_build_ref(logq, toks, budget, root_token)
