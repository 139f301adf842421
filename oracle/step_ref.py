"""One whole verification step over a batch of requests (oracle, test
infrastructure only): tree metadata -> depth-RoPE + tentative KV write ->
packed tree attention -> greedy accept -> KV commit.

The step order is the verify flow of "02 · Token Tree 与 Tree Attention"
(§3 mask/positions, §4 accept then commit) and of "Accelerating Speculative
Decoding with Block Diffusion Draft Trees" §7 (one target forward over the
flattened tree, then the verifier walk).

Batching (several requests, each with its own tree, concatenated) follows
"投机解码的树状注意力验证…", section "实现中的 KV Cache 与批处理约束".

Per-request status handling (a reading of the library's interface): tree
errors skip the rest of the step for that request; a missing block skips the
attention, accept and commit of that request; an accepted path that does not
fit max_depth skips the commit.
"""

import numpy as np

from .accept_ref import greedy_accept_ref
from .attention_ref import tree_attention_verify_ref
from .bf16_ref import bf16_bits_to_f64, f64_to_bf16_bits
from .commit_ref import kv_commit_ref
from .rope_ref import rope_ref
from .tree_ref import ST_BAD_BLOCK, ST_OK, tree_build_ref


def _blocks_ok(block_table_row, n_blocks, num_blocks, first_slot, end_slot, bs):
    """True when every slot in [first_slot, end_slot) lies in a held,
    in-range block."""
    if end_slot <= first_slot:
        return True
    for lb in range(first_slot // bs, (end_slot - 1) // bs + 1):
        if lb >= n_blocks or not (0 <= int(block_table_row[lb]) < num_blocks):
            return False
    return True


def verify_step_ref(w, attention=True, sample=None, commit=True):
    """Run one verification step on a workload ``w``.

    ``w`` is a mapping with the batch arrays (see the workload generators):
    geometry (num_q_heads, num_kv_heads, head_dim, block_size, rope_base,
    rope_style, max_nodes, max_depth), cu_nodes, parents (local parent indices,
    concatenated), prompt_len, q/k_new/v_new (bf16 bits), draft_tokens,
    target_ids, block_table, n_blocks, k_cache/v_cache (bf16 bits, copied, not
    modified).

    ``sample`` optionally maps request -> list of (node, q_head) pairs whose
    attention outputs are computed (others stay NaN).

    Returns a dict of per-request results and the post-step caches.
    """
    hq, hkv, d = w["num_q_heads"], w["num_kv_heads"], w["head_dim"]
    bs = w["block_size"]
    max_nodes, max_depth = w["max_nodes"], w["max_depth"]
    cu = np.asarray(w["cu_nodes"])
    batch = len(cu) - 1
    total = int(cu[-1])
    k_cache = np.array(w["k_cache"], copy=True)
    v_cache = np.array(w["v_cache"], copy=True)
    block_table = np.array(w["block_table"], copy=True)
    n_blocks = np.array(w["n_blocks"], copy=True)
    num_blocks = k_cache.shape[0]

    words = (max_nodes + 31) // 32
    res = {
        "status": np.zeros(batch, np.int32),
        "mask": np.zeros((total, words), np.uint32),
        "depth": np.zeros(total, np.int32),
        "positions": np.zeros(total, np.int32),
        "retrieve_index": np.zeros(total, np.int32),
        "next_token": np.zeros(total, np.int32),
        "next_sibling": np.zeros(total, np.int32),
        "out": np.full((total, hq, d), np.nan),
        "k_rot_bits": np.zeros((total, hkv, d), np.uint16),
        "paths": [None] * batch,
        "accept_len": np.zeros(batch, np.int32),
        "bonus": np.zeros(batch, np.int32),
        "new_len": np.zeros(batch, np.int32),
        "released": [[] for _ in range(batch)],
    }
    for b in range(batch):
        t0, t1 = int(cu[b]), int(cu[b + 1])
        n = t1 - t0
        plen = int(w["prompt_len"][b])
        parents = [int(p) for p in w["parents"][t0:t1]]
        tb = tree_build_ref(parents, plen, max_nodes)
        res["status"][b] = tb["status"]
        if tb["status"] != ST_OK:
            continue
        res["mask"][t0:t1] = tb["mask"]
        res["depth"][t0:t1] = tb["depth"]
        res["positions"][t0:t1] = tb["positions"]
        res["retrieve_index"][t0:t1] = np.arange(t0, t1, dtype=np.int32)
        res["next_token"][t0:t1] = tb["next_token"]
        res["next_sibling"][t0:t1] = tb["next_sibling"]

        row = block_table[b]
        if not _blocks_ok(row, int(n_blocks[b]), num_blocks, 0, plen + n, bs):
            res["status"][b] |= ST_BAD_BLOCK
            continue
        q_rot = rope_ref(bf16_bits_to_f64(w["q"][t0:t1]), tb["positions"],
                         w["rope_base"], w["rope_style"])
        k_rot = rope_ref(bf16_bits_to_f64(w["k_new"][t0:t1]), tb["positions"],
                         w["rope_base"], w["rope_style"])
        v_new = bf16_bits_to_f64(w["v_new"][t0:t1])
        res["k_rot_bits"][t0:t1] = f64_to_bf16_bits(k_rot)
        if attention:
            pairs = None if sample is None else sample.get(b, [])
            if pairs is None or pairs:
                res["out"][t0:t1] = tree_attention_verify_ref(
                    q_rot, k_rot, v_new, parents, k_cache, v_cache, row, plen, bs,
                    pairs=pairs)
        # Tentative write of the rotated K and raw V into slots P + i.
        for i in range(n):
            s = plen + i
            blk, r = int(row[s // bs]), s % bs
            k_cache[blk, :, r, :] = res["k_rot_bits"][t0 + i]
            v_cache[blk, :, r, :] = w["v_new"][t0 + i]

        st, path, bonus = greedy_accept_ref(parents, w["draft_tokens"][t0:t1],
                                            w["target_ids"][t0:t1], max_depth)
        if st != ST_OK:
            res["status"][b] |= st
            continue
        res["paths"][b] = path
        res["accept_len"][b] = len(path) - 1
        res["bonus"][b] = bonus
        if not commit:
            continue
        st, new_len, nb, released = kv_commit_ref(k_cache, v_cache, row,
                                                  int(n_blocks[b]), plen, path, bs)
        if st != ST_OK:
            res["status"][b] |= st
            continue
        res["new_len"][b] = new_len
        n_blocks[b] = nb
        res["released"][b] = released
    res["k_cache"] = k_cache
    res["v_cache"] = v_cache
    res["block_table"] = block_table
    res["n_blocks"] = n_blocks
    return res
