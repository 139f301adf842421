"""Tree metadata oracle: ancestor mask, depths, positions, child/sibling links
(test infrastructure only).

Definitions followed:
  * "Beam Search、约束解码与 Tree/Self Speculation", section "Packed tree
    attention": unique nodes are packed in topological order with a parent per
    node; each node sees the whole committed prefix plus its own ancestor
    chain, never siblings or cousins; the runnable packed-vs-branch experiment
    builds the chain by following parent pointers up to the root.
  * "02 · Token Tree 与 Tree Attention", §2 (the root is the previous round's
    bonus token) and §3 (mask rule; RoPE position = prompt length + tree depth,
    e.g. depths [0,1,1,2] with prompt length 7 give positions [7,8,8,9]; the
    builder's outputs are a tree mask, positions and retrieve_index /
    retrieve_next_token / retrieve_next_sibling).

Readings where the pages are silent:
  * node 0 is the root (depth 0); parent[0] = -1 and parent[i] < i for i >= 1;
  * the mask is stored tree-only and bit-packed: bit (j % 32) of word j // 32
    of row i is set iff node j is an ancestor of node i or i itself;
  * retrieve_next_token[i] = smallest-index child of i (or -1);
    retrieve_next_sibling[i] = smallest-index node j > i with the same parent
    (or -1); retrieve_index[i] = index of node i in the flattened batch.
"""

import numpy as np

# Per-request status flags (bit values are part of the library's interface).
ST_OK = 0
ST_BAD_SIZE = 1        # node count outside [1, max_nodes] or negative prompt length
ST_BAD_ROOT = 2        # parent[0] != -1
ST_BAD_PARENT = 4      # some parent[i] (i >= 1) outside [0, i-1]
ST_BAD_BLOCK = 8       # a block-table entry that is needed is missing or out of range
ST_PATH_OVERFLOW = 16  # accepted path does not fit the caller's path buffer


def ancestor_path(parents, node):
    """Root-to-node chain (inclusive), following parent pointers.

    Same walk as ``ancestor_path`` in the packed-vs-branch experiment of
    "Beam Search、约束解码与 Tree/Self Speculation".
    """
    chain = []
    while node != -1:
        chain.append(int(node))
        node = int(parents[node])
    return chain[::-1]


def validate_tree_ref(parents, prompt_len, max_nodes):
    """Status flags for one request's parent list (see module docstring)."""
    n = len(parents)
    if n < 1 or n > max_nodes or prompt_len < 0:
        return ST_BAD_SIZE
    st = ST_OK
    if int(parents[0]) != -1:
        st |= ST_BAD_ROOT
    for i in range(1, n):
        p = int(parents[i])
        if p < 0 or p >= i:
            st |= ST_BAD_PARENT
    return st


def tree_build_ref(parents, prompt_len, max_nodes):
    """Tree metadata for one request.

    Returns a dict with ``status`` and, when the status is 0,
      mask      uint32 [N, W], W = ceil(max_nodes / 32)
      depth     int32 [N]   (root depth 0)
      positions int32 [N]   (prompt_len + depth)
      next_token, next_sibling int32 [N]
    """
    parents = [int(p) for p in parents]
    n = len(parents)
    st = validate_tree_ref(parents, prompt_len, max_nodes)
    out = {"status": st}
    if st != ST_OK:
        return out
    words = (max_nodes + 31) // 32
    mask = np.zeros((n, words), dtype=np.uint32)
    depth = np.zeros(n, dtype=np.int32)
    for i in range(n):
        chain = ancestor_path(parents, i)
        depth[i] = len(chain) - 1
        for j in chain:
            mask[i, j // 32] |= np.uint32(1 << (j % 32))
    positions = (prompt_len + depth).astype(np.int32)
    next_token = np.full(n, -1, dtype=np.int32)
    next_sibling = np.full(n, -1, dtype=np.int32)
    for i in range(n):
        children = [j for j in range(n) if j != 0 and parents[j] == i]
        if children:
            next_token[i] = min(children)
        if i != 0:
            later = [j for j in range(i + 1, n) if parents[j] == parents[i]]
            if later:
                next_sibling[i] = min(later)
    out.update(mask=mask, depth=depth, positions=positions,
               next_token=next_token, next_sibling=next_sibling)
    return out
