"""Packed tree attention oracle (test infrastructure only).

Definitions followed:
  * "Beam Search、约束解码与 Tree/Self Speculation", section "Packed tree
    attention" and its runnable packed-vs-branch experiment: a node's query
    attends to every committed prefix key plus the keys of its own root-to-node
    chain; ``branch_reference`` gathers exactly those keys per node and runs
    ordinary softmax(q k^T / sqrt(d)) v, which the experiment shows equal to
    the packed form with an [N, P+N] ancestry mask (``packed_attention``).
  * "02 · Token Tree 与 Tree Attention", §3: visible = prompt ∪ ancestors of
    the node; invisible = siblings, cousins and any non-ancestor draft token.
  * "投机解码的树状注意力验证…", section "实现中的 KV Cache 与批处理约束": the tree's
    tentative K/V occupy a contiguous cache region in node order.

Grouped-query attention (not discussed by the pages; the geometry is given by
the workloads): query head h reads KV head h // (Hq / Hkv).

The per-node gather (``branch_attention_ref``) is the oracle; the dense masked
form is kept only so the tests can show the two agree, as the page's
experiment does.
"""

import math

import numpy as np

from .bf16_ref import bf16_bits_to_f64
from .tree_ref import ancestor_path


def _softmax(s):
    s = s - np.max(s, axis=-1, keepdims=True)
    e = np.exp(s)
    return e / np.sum(e, axis=-1, keepdims=True)


def branch_attention_ref(q, k_prompt, v_prompt, k_tree, v_tree, parents, scale=None):
    """Per-node gather attention.

    q [N, Hq, D]; k_prompt, v_prompt [P, Hkv, D]; k_tree, v_tree [N, Hkv, D];
    all float64. Returns float64 [N, Hq, D].
    """
    q = np.asarray(q, np.float64)
    n, hq, d = q.shape
    hkv = k_tree.shape[1]
    group = hq // hkv
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    out = np.zeros((n, hq, d), dtype=np.float64)
    for i in range(n):
        chain = ancestor_path(parents, i)
        for h in range(hq):
            g = h // group
            keys = np.concatenate([k_prompt[:, g, :], k_tree[chain, g, :]], axis=0)
            vals = np.concatenate([v_prompt[:, g, :], v_tree[chain, g, :]], axis=0)
            p = _softmax((keys @ q[i, h]) * scale)
            out[i, h] = p @ vals
    return out


def dense_tree_mask_ref(parents, prompt_len):
    """[N, P+N] bool mask: all prompt columns visible, tree columns visible on
    the node's ancestor chain (the experiment's ``tree_mask``)."""
    n = len(parents)
    mask = np.zeros((n, prompt_len + n), dtype=bool)
    mask[:, :prompt_len] = True
    for i in range(n):
        for j in ancestor_path(parents, i):
            mask[i, prompt_len + j] = True
    return mask


def packed_attention_ref(q, k_prompt, v_prompt, k_tree, v_tree, mask, scale=None):
    """Dense masked softmax over [prompt ‖ tree] keys (the experiment's
    ``packed_attention``), with GQA head sharing. float64 in and out."""
    n, hq, d = q.shape
    hkv = k_tree.shape[1]
    group = hq // hkv
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    out = np.zeros((n, hq, d), dtype=np.float64)
    for h in range(hq):
        g = h // group
        keys = np.concatenate([k_prompt[:, g, :], k_tree[:, g, :]], axis=0)
        vals = np.concatenate([v_prompt[:, g, :], v_tree[:, g, :]], axis=0)
        s = (q[:, h, :] @ keys.T) * scale
        s = np.where(mask, s, -np.inf)
        out[:, h, :] = _softmax(s) @ vals
    return out


def gather_prompt_kv_ref(cache_bits, block_table_row, prompt_len, block_size=16):
    """Committed prompt rows 0..P-1 of one request from a paged pool.

    cache_bits: bf16 bit patterns [num_blocks, Hkv, block_size, D]. Slot s
    lives in block block_table_row[s // block_size] at row s % block_size.
    Returns float64 [P, Hkv, D].
    """
    slots = np.arange(prompt_len)
    blocks = np.asarray(block_table_row)[slots // block_size].astype(np.int64)
    rows = cache_bits[blocks, :, slots % block_size, :]          # [P, Hkv, D]
    return bf16_bits_to_f64(rows)


def tree_attention_verify_ref(q_rot, k_tree_rot, v_tree, parents, k_cache_bits,
                              v_cache_bits, block_table_row, prompt_len,
                              block_size=16, scale=None, pairs=None):
    """Attention outputs of one request (float64, not rounded).

    q_rot [N, Hq, D], k_tree_rot/v_tree [N, Hkv, D] are float64 (the rotated,
    bf16-rounded values); the prompt K/V are read from the paged pools.
    ``pairs`` optionally restricts the computed (node, q_head) outputs (the
    others are NaN), for sampled checks at large sizes.
    """
    kp = gather_prompt_kv_ref(k_cache_bits, block_table_row, prompt_len, block_size)
    vp = gather_prompt_kv_ref(v_cache_bits, block_table_row, prompt_len, block_size)
    n, hq, d = q_rot.shape
    hkv = k_tree_rot.shape[1]
    group = hq // hkv
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if pairs is None:
        pairs = [(i, h) for i in range(n) for h in range(hq)]
    out = np.full((n, hq, d), np.nan, dtype=np.float64)
    for i, h in pairs:
        chain = ancestor_path(parents, i)
        g = h // group
        keys = np.concatenate([kp[:, g, :], k_tree_rot[chain, g, :]], axis=0)
        vals = np.concatenate([vp[:, g, :], v_tree[chain, g, :]], axis=0)
        p = _softmax((keys @ q_rot[i, h]) * scale)
        out[i, h] = p @ vals
    return out
