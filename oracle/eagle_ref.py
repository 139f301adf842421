"""EAGLE-2 dynamic-tree selection oracle (test infrastructure only: imported
by tests/, never by the product path).

Definitions followed, "02 · Token Tree 与 Tree Attention":
  * §3: EAGLE grows the tree layer by layer, each step expanding the top-k of
    the current layer ("layer x topk");
  * §5: EAGLE-2 scores every node by its prefix survival probability (the
    product of the drafter's probabilities along its path) and keeps the
    N_tree most promising nodes globally; easy contexts give deep trees,
    divergent ones wide trees.

Candidates are given in generation order (a candidate's parent comes before
it): per candidate the drafter's log-probability of its token under its
parent, its parent candidate (-1 for the root's children) and its token.

Readings where the pages leave a step open:
  * the score of a candidate is its parent's score plus its own
    log-probability (log of the survival product), evaluated in float32 in
    that order - the precision the CUDA kernel decides in, so equal inputs give
    equal selections;
  * ties: larger score first, then the shallower candidate, then the earlier
    generated one (layer expansion: score, then generation order);
  * the kept nodes are packed breadth first: by depth, then the parent's
    packed index, then generation order (the order of the children's ranks);
    node 0 is the root.
"""

import numpy as np


def eagle_scores_ref(logp, parent):
    """Cumulative float32 scores and depths (root's children have depth 1)."""
    logp = np.asarray(logp, dtype=np.float32)
    n = len(logp)
    score = np.zeros(n, np.float32)
    depth = np.zeros(n, np.int32)
    for c in range(n):
        p = int(parent[c])
        if p < 0:
            score[c] = logp[c]
            depth[c] = 1
        else:
            assert p < c, "a parent must be generated before its children"
            score[c] = np.float32(score[p] + logp[c])
            depth[c] = depth[p] + 1
    return score, depth


def eagle_expand_select_ref(logp, parent, layer, k):
    """The k candidates of depth ``layer`` to expand next: best score first,
    earlier generated on ties. Returns their indices in that order."""
    score, depth = eagle_scores_ref(logp, parent)
    idx = [c for c in range(len(score)) if depth[c] == layer]
    idx.sort(key=lambda c: (-float(score[c]), c))
    return np.array(idx[:k], np.int32)


def eagle_rerank_ref(logp, parent, token, n_keep, root_token=-1):
    """Global top-``n_keep`` candidates packed breadth first.

    Returns (status, parents, tokens, kept) where parents/tokens have
    n_keep + 1 entries (root first), ``kept`` the selected candidate indices
    in packed order, status 0 or 1 when fewer than n_keep candidates exist or
    the selection is not prefix-closed (a positive log-probability)."""
    score, depth = eagle_scores_ref(logp, parent)
    n = len(score)
    if n < n_keep:
        return 1, None, None, None
    order = sorted(range(n), key=lambda c: (-float(score[c]), int(depth[c]), c))
    kept = set(order[:n_keep])
    for c in kept:
        if int(parent[c]) >= 0 and int(parent[c]) not in kept:
            return 1, None, None, None
    packed = {-1: 0}
    seq = []
    for d in range(1, (max(int(depth[c]) for c in kept) if kept else 0) + 1):
        level = [c for c in kept if depth[c] == d]
        level.sort(key=lambda c: (packed[int(parent[c])], c))
        for c in level:
            packed[c] = len(seq) + 1
            seq.append(c)
    parents = np.array([-1] + [packed[int(parent[c])] for c in seq], np.int32)
    tokens = np.array([root_token] + [int(token[c]) for c in seq], np.int32)
    return 0, parents, tokens, np.array(seq, np.int32)
