"""KV commit / rollback oracle (test infrastructure only).

Definitions followed:
  * "Beam Search、约束解码与 Tree/Self Speculation", section "Tree/Self
    Speculation" and the three-part semantics experiment: the accepted path's
    tentative KV joins the committed cache ([10,11] -> [10,11,4,7]); the other
    tentative nodes are rolled back / released.
  * "02 · Token Tree 与 Tree Attention", §4: the chosen path's KV is committed
    and becomes the next round's prompt; siblings and nodes past the rejection
    point are discarded; pages are allocated per tree and reclaimed.
  * "投机解码的树状注意力验证…", section "实现中的 KV Cache 与批处理约束": the tree owns a
    contiguous region in node order; with a paged cache, reclaiming means
    freeing or reusing pages.

Readings where the pages are silent:
  * tentative node i of a request with prompt length P sits in slot P + i;
    the root (node 0) is always committed (it is the confirmed bonus token);
  * accepted node path[k] (k = 1..a) moves to slot P + k, so the committed
    length becomes P + 1 + a; the KV bytes are moved unchanged (their RoPE
    position P + depth = P + k already matches the new slot);
  * blocks whose logical index is >= ceil(new_len / block_size), among those
    the request held, are released in ascending logical order and their
    block-table entries set to -1.
"""

import numpy as np

from .tree_ref import ST_BAD_BLOCK, ST_OK


def kv_commit_ref(k_cache_bits, v_cache_bits, block_table_row, n_blocks,
                  prompt_len, path, block_size=16):
    """Commit one request's accepted path.

    k_cache_bits/v_cache_bits: bf16 bit arrays [num_blocks, Hkv, bs, D]
    (modified in place). block_table_row: int32 [max_blocks] (modified in
    place). Returns (status, new_len, new_n_blocks, released_blocks).
    """
    num_blocks = k_cache_bits.shape[0]
    a = len(path) - 1
    # Every slot that is read or written must lie in a held, in-range block.
    touched = [prompt_len + int(path[k]) for k in range(1, a + 1)]
    touched += [prompt_len + k for k in range(1, a + 1)]
    for slot in touched:
        lb = slot // block_size
        if lb >= n_blocks or not (0 <= int(block_table_row[lb]) < num_blocks):
            return ST_BAD_BLOCK, None, None, None

    def loc(slot):
        return int(block_table_row[slot // block_size]), slot % block_size

    # Read every source row first, then write (a destination slot can be the
    # source of an earlier accepted node).
    moved = []
    for k in range(1, a + 1):
        b, r = loc(prompt_len + int(path[k]))
        moved.append((k_cache_bits[b, :, r, :].copy(), v_cache_bits[b, :, r, :].copy()))
    for k in range(1, a + 1):
        b, r = loc(prompt_len + k)
        k_cache_bits[b, :, r, :] = moved[k - 1][0]
        v_cache_bits[b, :, r, :] = moved[k - 1][1]

    new_len = prompt_len + 1 + a
    keep = -(-new_len // block_size)
    released = []
    for lb in range(keep, n_blocks):
        released.append(int(block_table_row[lb]))
        block_table_row[lb] = -1
    return ST_OK, new_len, min(keep, n_blocks), released
