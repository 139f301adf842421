"""Greedy tree acceptance oracle (test infrastructure only).

Definitions followed:
  * "Beam Search、约束解码与 Tree/Self Speculation", runnable three-part
    semantics experiment, ``verify_tree``: walking depth by depth, keep the
    branches whose next token equals the target's choice; stop at the first
    depth where none does. The committed cache gains the accepted tokens and
    every other tentative node is released.
  * "02 · Token Tree 与 Tree Attention", §4: from the root, accept the child
    whose token equals the target's (greedy) choice and continue from it; when
    no child matches, the target's own token at that node is the correction
    (the next round's bonus/root token).
  * "Accelerating Speculative Decoding with Block Diffusion Draft Trees",
    §6 (worked walk) and §7.2 (verifier walk): the first mismatching target
    token becomes the next bonus token.

Reading where the pages are silent: if several children of the current node
carry the matching token (possible only when a parent list has duplicate
sibling tokens), the smallest packed index is taken.
"""

from .tree_ref import ST_OK, ST_PATH_OVERFLOW


def greedy_accept_ref(parents, draft_tokens, target_ids, max_depth):
    """Walk one request's tree against per-node target ids.

    parents[i] (parent[0] = -1), draft_tokens[i] (token of node i; node 0 is
    the root, whose token is the previous bonus) and target_ids[i] (the
    target's greedy token after node i's prefix).

    Returns (status, path, bonus): ``path`` lists packed node indices from the
    root (path[0] = 0); the number of accepted draft nodes is len(path) - 1.
    A path with more than max_depth accepted nodes gives ST_PATH_OVERFLOW.
    """
    n = len(parents)
    children = [[] for _ in range(n)]
    for j in range(1, n):
        children[int(parents[j])].append(j)        # ascending packed index
    path = [0]
    cur = 0
    while True:
        want = int(target_ids[cur])
        nxt = None
        for c in children[cur]:
            if int(draft_tokens[c]) == want:
                nxt = c
                break
        if nxt is None:
            bonus = want
            break
        path.append(nxt)
        cur = nxt
    if len(path) - 1 > max_depth:
        return ST_PATH_OVERFLOW, path, bonus
    return ST_OK, path, bonus


def verify_branches_ref(base_cache, branches, target_next):
    """The glossary experiment's branch-list semantics.

    ``branches`` are root-to-leaf token lists; ``target_next`` the target's
    token at each depth. Returns (committed_cache, accepted_tokens,
    released_tentative_count) where the tentative set is every distinct
    non-empty branch prefix.
    """
    tentative = {tuple(b[:d]) for b in branches for d in range(1, len(b) + 1)}
    accepted = []
    alive = list(branches)
    for depth, tok in enumerate(target_next):
        alive = [b for b in alive
                 if len(b) > depth and list(b[:depth]) == accepted and b[depth] == tok]
        if not alive:
            break
        accepted.append(tok)
    kept = {tuple(accepted[:d]) for d in range(1, len(accepted) + 1)}
    return list(base_cache) + accepted, accepted, len(tentative - kept)
