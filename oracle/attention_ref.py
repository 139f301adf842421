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
    others are NaN), for checks of selected outputs at large sizes.

    Same visible set and softmax as ``branch_attention_ref``: query (i, h)
    attends to all P prompt keys of KV head g = h // G plus the keys of node
    i's root-to-node chain. The scores against the prompt keys of one KV head
    are taken for all its selected queries in one matrix product, and each
    output is sum_j exp(s_j - m) v_j / sum_j exp(s_j - m) over those keys, m
    the row's largest score (the softmax written out, normalised after the
    weighted sum).
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
    chains = {}
    for g in range(hkv):
        sel = [(i, h) for (i, h) in pairs if h // group == g]
        if not sel:
            continue
        kg = np.ascontiguousarray(kp[:, g, :])                 # [P, D]
        vg = np.ascontiguousarray(vp[:, g, :])
        qs = np.stack([q_rot[i, h] for (i, h) in sel])         # [m, D]
        s_prompt = (qs @ kg.T) * scale                         # [m, P]
        s_chain = []
        for r, (i, _) in enumerate(sel):
            if i not in chains:
                chains[i] = ancestor_path(parents, i)
            s_chain.append((k_tree_rot[chains[i], g, :] @ qs[r]) * scale)
        m = np.array([max(np.max(s_prompt[r], initial=-np.inf), np.max(s_chain[r]))
                      for r in range(len(sel))])
        e_prompt = np.exp(s_prompt - m[:, None])
        num = e_prompt @ vg                                    # [m, D]
        den = e_prompt.sum(axis=1)
        for r, (i, h) in enumerate(sel):
            e_chain = np.exp(s_chain[r] - m[r])
            out[i, h] = (num[r] + e_chain @ v_tree[chains[i], g, :]) / (den[r] + e_chain.sum())
    return out
