"""Pins of the CPU oracle to facts that do not come from the oracle itself:
values the pages print (tests/golden/), closed forms, textbook special cases,
library routines and brute force. A plausible slip in the oracle (dropped key,
wrong sign or pairing in RoPE, wrong GQA head, off-by-one position, wrong
walk or commit order) fails at least one test here."""

import numpy as np
import pytest
import torch

from oracle import (
    ST_BAD_BLOCK, ST_BAD_PARENT, ST_BAD_ROOT, ST_BAD_SIZE, ST_OK, ST_PATH_OVERFLOW,
    bf16_bits_to_f64, branch_attention_ref, dense_tree_mask_ref, f64_to_bf16_bits,
    gather_prompt_kv_ref, greedy_accept_ref, kv_commit_ref, packed_attention_ref,
    rope_inv_freq_f32, rope_ref, round_to_bf16, tree_attention_verify_ref, tree_build_ref,
    verify_branches_ref,
)

# --------------------------------------------------------------------------
# helpers independent of the oracle


def forward_sequences(parents, tokens):
    """Token sequence of every node built forward from the root (parents
    precede children), not by walking parent pointers upward."""
    seqs = []
    for i, p in enumerate(parents):
        seqs.append(() if p == -1 else seqs[p] + (int(tokens[i]),))
    return seqs


def forward_chains(parents):
    chains = []
    for i, p in enumerate(parents):
        chains.append([i] if p == -1 else chains[p] + [i])
    return chains


def random_tree(rng, n, distinct_sibling_tokens=True, vocab=50):
    parents = [-1] + [int(rng.integers(0, i)) for i in range(1, n)]
    tokens = [int(rng.integers(0, vocab))]
    used = {}
    for i in range(1, n):
        p = parents[i]
        s = used.setdefault(p, set())
        while True:
            t = int(rng.integers(0, vocab))
            if not distinct_sibling_tokens or t not in s:
                break
        s.add(t)
        tokens.append(t)
    return parents, tokens


# --------------------------------------------------------------------------
# bf16


def test_bf16_rounding_matches_torch_rne():
    rng = np.random.default_rng(0)
    vals = [rng.standard_normal(20000).astype(np.float32),
            (rng.standard_normal(2000) * 1e-39).astype(np.float32),   # subnormals
            np.clip(rng.standard_normal(2000) * 1e38, -3.39e38, 3.39e38).astype(np.float32),  # near overflow
            np.array([0.0, -0.0, 1.0, -1.0, np.inf, -np.inf], np.float32)]
    # exact ties: a bf16 value plus half of its quantum
    base = bf16_bits_to_f64(rng.integers(0x3000, 0x4F00, 3000).astype(np.uint16))
    _, e = np.frexp(base)
    vals.append((base + np.ldexp(1.0, e - 9)).astype(np.float32))
    vals.append((base - np.ldexp(1.0, e - 9)).astype(np.float32))
    x = np.concatenate(vals)
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = f64_to_bf16_bits(x.astype(np.float64))
    assert np.array_equal(got, want)
    assert np.array_equal(bf16_bits_to_f64(got), round_to_bf16(x.astype(np.float64)))


# --------------------------------------------------------------------------
# tree metadata


def test_positions_page_example(golden):
    g = golden("token_tree_positions.json")
    parents = [-1, 0, 0, 1]                       # depths [0, 1, 1, 2]
    tb = tree_build_ref(parents, g["prompt_length"], 8)
    assert tb["depth"].tolist() == g["depths"]
    assert tb["positions"].tolist() == g["positions"]


def _glossary_as_rooted(g):
    """The glossary table has no root; add the last committed token as node 0
    (prefix [10, 11] -> prompt [10] plus root 11, so P = prefix - 1)."""
    parents = [-1] + [p + 1 for p in g["parents"]]
    return parents, g["prefix_length"] - 1


def test_glossary_packed_table(golden):
    g = golden("glossary_packed_table.json")
    parents, plen = _glossary_as_rooted(g)
    tb = tree_build_ref(parents, plen, 64)
    assert tb["status"] == ST_OK
    assert tb["depth"][1:].tolist() == g["depths"]
    assert tb["positions"][1:].tolist() == g["position_ids"]
    for i, vis in enumerate(g["visible_ancestors"]):
        row = tb["mask"][i + 1, 0]
        bits = [j - 1 for j in range(1, 9) if (int(row) >> j) & 1]
        assert bits == vis
        assert (int(row) & 1) == 1                 # the root is always visible
    # visible keys = committed prefix (P + root) + the node's chain
    counts = [plen + bin(int(r)).count("1") for r in tb["mask"][1:, 0]]
    assert counts == g["mask_visible_counts"]
    assert sum(len(b) for b in [[4, 5, 6], [4, 7, 8], [9, 0, 1]]) == g["branch_expanded_positions"]
    assert len(g["tokens"]) == g["unique_tree_nodes"]


@pytest.mark.parametrize("seed", range(6))
def test_mask_matches_prefix_relation(seed):
    """Every node pair's visibility equals the prefix relation of their token
    sequences (mask-correctness rule of the tree-attention verification page)."""
    rng = np.random.default_rng(seed)
    n = int(rng.integers(1, 90))
    parents, tokens = random_tree(rng, n)
    tb = tree_build_ref(parents, 5, 96)
    seqs = forward_sequences(parents, tokens)
    for i in range(n):
        for j in range(n):
            bit = (int(tb["mask"][i, j // 32]) >> (j % 32)) & 1
            assert bit == int(seqs[i][:len(seqs[j])] == seqs[j])
        assert bin(sum(int(w) << (32 * k) for k, w in enumerate(tb["mask"][i]))).count("1") \
            == tb["depth"][i] + 1
        assert tb["depth"][i] == len(seqs[i])
        assert tb["positions"][i] == 5 + len(seqs[i])


@pytest.mark.parametrize("seed", range(4))
def test_child_sibling_links_enumerate_children(seed):
    rng = np.random.default_rng(100 + seed)
    n = int(rng.integers(1, 70))
    parents, _ = random_tree(rng, n)
    tb = tree_build_ref(parents, 0, 70)
    for i in range(n):
        want = [j for j in range(n) if parents[j] == i]
        got, c = [], int(tb["next_token"][i])
        while c != -1:
            got.append(c)
            c = int(tb["next_sibling"][c])
        assert got == want
    assert tb["next_sibling"][0] == -1


def test_tree_validation_flags():
    assert tree_build_ref([], 3, 8)["status"] == ST_BAD_SIZE
    assert tree_build_ref([-1] * 9, 3, 8)["status"] == ST_BAD_SIZE
    assert tree_build_ref([-1, 0], -1, 8)["status"] == ST_BAD_SIZE
    assert tree_build_ref([0, 0], 3, 8)["status"] == ST_BAD_ROOT
    assert tree_build_ref([0, 1], 3, 8)["status"] == ST_BAD_ROOT | ST_BAD_PARENT
    assert tree_build_ref([-1, 1], 3, 8)["status"] == ST_BAD_PARENT
    assert tree_build_ref([-1, 0, -1], 3, 8)["status"] == ST_BAD_PARENT
    assert tree_build_ref([-1, 0, 5], 3, 8)["status"] == ST_BAD_PARENT
    assert tree_build_ref([-1], 0, 1)["status"] == ST_OK


# --------------------------------------------------------------------------
# RoPE


def test_rope_identity_at_position_zero():
    rng = np.random.default_rng(1)
    x = round_to_bf16(rng.standard_normal((5, 3, 64)))
    assert np.array_equal(rope_ref(x, np.zeros(5, int)), x)


def test_rope_is_complex_rotation_per_pair():
    """Pair i of an interleaved head rotates like the complex number
    x[2i] + 1j*x[2i+1] multiplied by exp(1j * angle)."""
    rng = np.random.default_rng(2)
    d = 16
    x = rng.standard_normal((4, 2, d))
    pos = np.array([0, 3, 17, 2000])
    got = rope_ref(x, pos, round_bf16=False)
    inv = rope_inv_freq_f32(d, 10000.0)
    assert inv[0] == 1.0 and np.all(np.diff(inv) < 0)
    assert np.isclose(inv[-1], 10000.0 ** (-(d - 2) / d), rtol=1e-7)
    for i in range(d // 2):
        ang = (pos.astype(np.float64) * np.float64(inv[i])).astype(np.float32).astype(np.float64)
        z = (x[..., 2 * i] + 1j * x[..., 2 * i + 1]) * np.exp(1j * ang)[:, None]
        assert np.allclose(got[..., 2 * i], z.real, atol=1e-13)
        assert np.allclose(got[..., 2 * i + 1], z.imag, atol=1e-13)


def test_rope_relative_position_and_norm():
    rng = np.random.default_rng(3)
    q = rng.standard_normal((1, 1, 64))
    k = rng.standard_normal((1, 1, 64))
    def dot(m, n):
        return float(np.sum(rope_ref(q, [m], round_bf16=False) * rope_ref(k, [n], round_bf16=False)))
    for (m, n, s) in [(5, 2, 7), (9, 9, 100), (40, 3, 11)]:
        assert abs(dot(m, n) - dot(m + s, n + s)) < 1e-4
    r = rope_ref(q, [123], round_bf16=False)
    assert np.allclose(np.hypot(r[..., 0::2], r[..., 1::2]), np.hypot(q[..., 0::2], q[..., 1::2]))


def test_rope_half_split_is_permuted_interleaved():
    rng = np.random.default_rng(4)
    d = 32
    x = rng.standard_normal((6, 2, d))
    pos = rng.integers(0, 5000, 6)
    perm = np.empty(d, int)                 # half-split layout -> interleaved layout
    perm[0::2] = np.arange(d // 2)
    perm[1::2] = np.arange(d // 2) + d // 2
    half = rope_ref(x, pos, style=1, round_bf16=False)
    inter = rope_ref(x[..., perm], pos, style=0, round_bf16=False)
    assert np.array_equal(half[..., perm], inter)


# --------------------------------------------------------------------------
# attention


def _rand_qkv(rng, n, p, hq, hkv, d):
    return (rng.standard_normal((n, hq, d)), rng.standard_normal((p, hkv, d)),
            rng.standard_normal((p, hkv, d)), rng.standard_normal((n, hkv, d)),
            rng.standard_normal((n, hkv, d)))


def test_packed_equals_branch_and_wrong_mask_leaks(golden):
    """The glossary's experiment: packed masked attention equals per-node
    gather attention, and a lower-triangular tree mask leaks siblings."""
    g = golden("glossary_packed_table.json")
    rng = np.random.default_rng(233)
    parents, p, n, d = g["parents"], g["prefix_length"], len(g["parents"]), 8
    q, kp, vp, kt, vt = _rand_qkv(rng, n, p, 2, 2, d)
    pos = np.array(g["position_ids"])
    q = rope_ref(q, pos, round_bf16=False)
    kt = rope_ref(kt, pos, round_bf16=False)
    kp = rope_ref(kp, np.arange(p), round_bf16=False)
    mask = dense_tree_mask_ref(parents, p)
    assert mask.sum(-1).tolist() == g["mask_visible_counts"]
    ref = branch_attention_ref(q, kp, vp, kt, vt, parents)
    packed = packed_attention_ref(q, kp, vp, kt, vt, mask)
    assert np.max(np.abs(packed - ref)) < g["packed_vs_branch_tolerance"]
    wrong = np.concatenate([np.ones((n, p), bool), np.tril(np.ones((n, n), bool))], 1)
    leak = np.max(np.abs(packed_attention_ref(q, kp, vp, kt, vt, wrong) - ref))
    assert leak > g["sibling_leak_threshold"]


@pytest.mark.parametrize("seed", range(3))
def test_packed_equals_branch_random_rooted_gqa(seed):
    rng = np.random.default_rng(10 + seed)
    n, p = int(rng.integers(1, 40)), int(rng.integers(0, 30))
    parents, _ = random_tree(rng, n)
    q, kp, vp, kt, vt = _rand_qkv(rng, n, p, 8, 2, 16)
    ref = branch_attention_ref(q, kp, vp, kt, vt, parents)
    packed = packed_attention_ref(q, kp, vp, kt, vt, dense_tree_mask_ref(parents, p))
    assert np.max(np.abs(packed - ref)) < 1e-12


def test_chain_tree_is_causal_attention():
    """A tree that is a single path is ordinary causal attention over
    prompt + draft (checked against torch's scaled_dot_product_attention)."""
    rng = np.random.default_rng(5)
    n, p, h, d = 12, 9, 3, 32
    parents = [-1] + list(range(n - 1))
    q, kp, vp, kt, vt = _rand_qkv(rng, n, p, h, h, d)
    ref = branch_attention_ref(q, kp, vp, kt, vt, parents)
    keys = np.concatenate([kp, kt], 0)
    vals = np.concatenate([vp, vt], 0)
    allowed = np.arange(p + n)[None, :] <= (p + np.arange(n))[:, None]
    sdpa = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q.transpose(1, 0, 2)), torch.from_numpy(keys.transpose(1, 0, 2)),
        torch.from_numpy(vals.transpose(1, 0, 2)), attn_mask=torch.from_numpy(allowed))
    assert np.max(np.abs(sdpa.numpy().transpose(1, 0, 2) - ref)) < 1e-12


def test_attention_closed_forms():
    rng = np.random.default_rng(6)
    # a lone root with no prompt returns its own value
    q, kp, vp, kt, vt = _rand_qkv(rng, 1, 0, 2, 1, 8)
    assert np.allclose(branch_attention_ref(q, kp, vp, kt, vt, [-1])[0, 1], vt[0, 0], atol=1e-15)
    # zero keys: uniform weights = mean of exactly the prompt + chain values;
    # value = kv-head index + 1 pins the GQA head map h -> h // (Hq/Hkv)
    n, p, hq, hkv, d = 7, 5, 6, 3, 4
    parents = [-1, 0, 0, 1, 3, 2, 5]
    q = rng.standard_normal((n, hq, d))
    kp, kt = np.zeros((p, hkv, d)), np.zeros((n, hkv, d))
    vp = np.zeros((p, hkv, d)) + np.arange(hkv)[None, :, None] + 1.0
    vt = rng.standard_normal((n, hkv, d))
    out = branch_attention_ref(q, kp, vp, kt, vt, parents)
    chains = forward_chains(parents)
    for i in range(n):
        for h in range(hq):
            g = h // (hq // hkv)
            want = (vp[:, g].sum(0) + vt[chains[i], g].sum(0)) / (p + len(chains[i]))
            assert np.allclose(out[i, h], want, atol=1e-14)


@pytest.mark.parametrize("seed", range(4))
def test_paged_step_attention_equals_branch_gather(seed):
    """The step oracle's attention (prompt scores per KV head in one matrix
    product, softmax normalised after the weighted sum) equals the per-node
    gather on the same keys, for all outputs and for a selected subset; the
    unselected outputs stay NaN. Covers an empty prompt and GQA groups."""
    rng = np.random.default_rng(40 + seed)
    bs, hq, hkv, d = 4, 8, 2, 16
    n = int(rng.integers(1, 30))
    plen = [0, 1, 17, 45][seed]
    parents, _ = random_tree(rng, n)
    nblk = -(-(plen + n) // bs) + 3
    table = rng.permutation(nblk)[: -(-(plen + n) // bs)]
    kpool = f64_to_bf16_bits(rng.standard_normal((nblk, hkv, bs, d)))
    vpool = f64_to_bf16_bits(rng.standard_normal((nblk, hkv, bs, d)))
    q = rng.standard_normal((n, hq, d)) * 2.0
    kt, vt = rng.standard_normal((n, hkv, d)), rng.standard_normal((n, hkv, d))
    kp = gather_prompt_kv_ref(kpool, table, plen, bs)
    vp = gather_prompt_kv_ref(vpool, table, plen, bs)
    want = branch_attention_ref(q, kp, vp, kt, vt, parents)
    got = tree_attention_verify_ref(q, kt, vt, parents, kpool, vpool, table, plen, bs)
    assert np.max(np.abs(got - want)) < 1e-13
    pairs = sorted({(int(rng.integers(0, n)), int(rng.integers(0, hq))) for _ in range(7)})
    part = tree_attention_verify_ref(q, kt, vt, parents, kpool, vpool, table, plen, bs, pairs=pairs)
    sel = np.zeros((n, hq), bool)
    for i, h in pairs:
        sel[i, h] = True
    assert np.max(np.abs(part[sel] - want[sel])) < 1e-13
    assert np.all(np.isnan(part[~sel]))


def test_paged_gather_follows_block_table():
    rng = np.random.default_rng(7)
    bs, nb, hkv, d, plen = 4, 11, 2, 3, 29
    table = rng.permutation(nb)[: -(-plen // bs)]
    pool = np.zeros((nb, hkv, bs, d), np.uint16)
    for s in range(plen):                       # slot id encoded as a bf16 value
        pool[table[s // bs], :, s % bs, :] = f64_to_bf16_bits(np.float64(s))
    got = gather_prompt_kv_ref(pool, table, plen, bs)
    assert np.array_equal(got[:, 0, 0], np.arange(plen, dtype=np.float64))


# --------------------------------------------------------------------------
# acceptance


def test_glossary_verify_example(golden):
    g = golden("glossary_verify_example.json")
    committed, accepted, released = verify_branches_ref(g["base_cache"], g["branches"], g["target_next"])
    assert committed == g["committed"] and accepted == g["accepted"]
    assert released == g["released_tentative"]


def _glossary_tree_rooted(golden):
    t = golden("glossary_packed_table.json")
    parents, plen = _glossary_as_rooted(t)
    tokens = [11] + t["tokens"]
    return parents, tokens, plen


def test_greedy_walk_on_glossary_tree(golden):
    g = golden("glossary_verify_example.json")
    parents, tokens, _ = _glossary_tree_rooted(golden)
    seqs = forward_sequences(parents, tokens)
    tgt = [99] * len(parents)
    # the target's next token after each accepted prefix
    for depth, tok in enumerate(g["target_next"]):
        node = seqs.index(tuple(g["target_next"][:depth]))
        tgt[node] = tok
    st, path, bonus = greedy_accept_ref(parents, tokens, tgt, 8)
    assert st == ST_OK
    assert [tokens[i] for i in path[1:]] == g["accepted"]
    assert bonus == g["target_next"][len(g["accepted"])]


def test_ddtree_walk_example(golden):
    g = golden("ddtree_walk.json")
    names = g["flattened"]
    ids = {c: k for k, c in enumerate("bABCD")}
    tokens = [ids[c] for c in names]
    parents = g["reconstructed_parents"]
    tb = tree_build_ref(parents, 0, 8)
    assert tb["positions"].tolist() == g["position_ids"]
    seqs = forward_sequences(parents, tokens)
    tgt = [ids["D"]] * len(parents)
    for pre, nxt in g["target_walk"].items():
        key = tuple(ids[c] for c in pre) if pre != "b" else ()
        tgt[seqs.index(key)] = ids[nxt]
    st, path, bonus = greedy_accept_ref(parents, tokens, tgt, 8)
    assert [names[i] for i in path[1:]] == g["accepted"]
    assert bonus == ids[g["bonus"]]
    assert len(path) == g["tokens_per_round"]       # bonus/root + accepted


@pytest.mark.parametrize("seed", range(8))
def test_greedy_walk_brute_force(seed):
    """With distinct sibling tokens the accepted path is the deepest node
    whose every edge matches the target id at its parent."""
    rng = np.random.default_rng(200 + seed)
    n = int(rng.integers(1, 80))
    parents, tokens = random_tree(rng, n, vocab=6)
    tgt = [int(rng.integers(0, 6)) for _ in range(n)]
    chains = forward_chains(parents)
    ok = [all(tokens[c[k]] == tgt[c[k - 1]] for k in range(1, len(c))) for c in chains]
    deepest = max((len(chains[i]), -i) for i in range(n) if ok[i])
    best = -deepest[1]
    st, path, bonus = greedy_accept_ref(parents, tokens, tgt, n)
    assert path == chains[best] and bonus == tgt[best] and st == ST_OK


def test_greedy_walk_tie_takes_smallest_index_and_overflow():
    parents = [-1, 0, 0, 2]
    tokens = [0, 5, 5, 7]
    tgt = [5, 1, 7, 3]
    st, path, bonus = greedy_accept_ref(parents, tokens, tgt, 4)
    assert path == [0, 1] and bonus == 1
    chain = [-1, 0, 1, 2]
    st, path, _ = greedy_accept_ref(chain, [0, 1, 2, 3], [1, 2, 3, 4], 2)
    assert st == ST_PATH_OVERFLOW


# --------------------------------------------------------------------------
# commit


def test_glossary_commit_example(golden):
    """Slots carry token ids; after the commit the cache reads [10,11,4,7]
    and the other 6 tentative slots fall past the committed length."""
    g = golden("glossary_verify_example.json")
    parents, tokens, plen = _glossary_tree_rooted(golden)
    bs, hkv, d = 2, 1, 2
    n = len(parents)
    nb = -(-(plen + n) // bs)
    table = np.array([3, 0, 4, 1, 2, -1, -1], np.int32)
    k = np.zeros((8, hkv, bs, d), np.uint16)
    v = np.zeros_like(k)
    seq = [10] + tokens                                  # slot s holds token seq[s]
    for s, tok in enumerate(seq):
        k[table[s // bs], :, s % bs, :] = f64_to_bf16_bits(np.float64(tok))
        v[table[s // bs], :, s % bs, :] = f64_to_bf16_bits(np.float64(-tok))
    path = [0, 1, 4]                                     # tokens 11 -> 4 -> 7
    held = table[:nb].tolist()
    st, new_len, new_nb, released = kv_commit_ref(k, v, table, nb, plen, path, bs)
    assert st == ST_OK
    got = [int(bf16_bits_to_f64(k[table[s // bs], 0, s % bs, 0])) for s in range(new_len)]
    assert got == g["committed"]
    assert (plen + n) - new_len == g["released_tentative"]
    assert new_len == plen + 1 + 2 and new_nb == 2
    assert released == held[2:] and sorted(released + table[:new_nb].tolist()) == sorted(held)
    assert np.all(table[new_nb:] == -1)


@pytest.mark.parametrize("seed", range(6))
def test_commit_moves_path_rows_unchanged(seed):
    rng = np.random.default_rng(300 + seed)
    bs, hkv, d = 16, 2, 8
    n = int(rng.integers(1, 60))
    parents, _ = random_tree(rng, n)
    chains = forward_chains(parents)
    path = chains[int(rng.integers(0, n))]
    plen = int(rng.integers(0, 50))
    nb_need = -(-(plen + n) // bs)
    nb = nb_need + int(rng.integers(0, 3))
    num_blocks = nb + 4
    table = np.full(nb + 2, -1, np.int32)
    table[:nb] = rng.permutation(num_blocks)[:nb]
    k = rng.integers(0, 65535, (num_blocks, hkv, bs, d)).astype(np.uint16)
    v = rng.integers(0, 65535, (num_blocks, hkv, bs, d)).astype(np.uint16)
    k0, v0, t0 = k.copy(), v.copy(), table.copy()
    st, new_len, new_nb, released = kv_commit_ref(k, v, table, nb, plen, path, bs)
    assert st == ST_OK
    a = len(path) - 1
    assert new_len == plen + 1 + a
    def row(arr, tab, s):
        return arr[tab[s // bs], :, s % bs, :]
    for s in range(plen + 1):                         # prompt and root untouched
        assert np.array_equal(row(k, table, s), row(k0, t0, s))
    for kk in range(1, a + 1):
        assert np.array_equal(row(k, table, plen + kk), row(k0, t0, plen + path[kk]))
        assert np.array_equal(row(v, table, plen + kk), row(v0, t0, plen + path[kk]))
    keep = -(-new_len // bs)
    assert released == t0[keep:nb].tolist() and new_nb == min(keep, nb)
    assert np.all(table[keep:] == -1) and np.array_equal(table[:keep], t0[:keep])


def test_commit_overlapping_slots_and_bad_block():
    bs = 4
    table = np.array([0, 1], np.int32)
    k = np.zeros((2, 1, bs, 1), np.uint16)
    for s in range(8):
        k[s // bs, 0, s % bs, 0] = s
    v = k.copy()
    # path [0,2,3]: slot 2 -> 1, then slot 3 -> 2 (slot 2 is read before written)
    st, new_len, _, _ = kv_commit_ref(k, v, table, 2, 0, [0, 2, 3], bs)
    assert st == ST_OK and new_len == 3
    assert [int(k[s // bs, 0, s % bs, 0]) for s in range(4)] == [0, 2, 3, 3]
    bad = np.array([0, 9], np.int32)
    k2 = np.zeros((2, 1, bs, 1), np.uint16)
    st, *_ = kv_commit_ref(k2, k2.copy(), bad, 2, 2, [0, 1, 3], bs)
    assert st == ST_BAD_BLOCK and bad.tolist() == [0, 9]
