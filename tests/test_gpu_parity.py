"""GPU parity: every library call against the CPU oracle on the same seeded
inputs. Integer outputs (mask, positions, links, paths, block tables, moved KV
bytes) must match bit for bit; attention outputs within max-abs 2e-2 and
relative Frobenius 5e-3; rotated keys within one bf16 ulp of the exact
rotation plus the float32 rotation's absolute error (the GPU rotates in
float32, the oracle exactly)."""

import numpy as np
import pytest
import torch

from oracle import kv_commit_ref
from gen import workloads as wl
from speculative_decoding_tree_build_gb300.build import build
from speculative_decoding_tree_build_gb300.step import DeviceBatch

from parity import (bf16_bits_to_f64, bf16_ulp_diff, check_accept_outputs, check_tree_outputs,
                    compare_out, oracle_step, rope_close, run_gpu, sample_pairs, split_unit_pairs,
                    tentative_rows)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build()
    assert torch.cuda.is_available()


SMALL = {1: {}, 2: dict(batch=3, prompt_scale=0.25), 3: dict(batch=2, prompt_scale=0.1),
         4: dict(batch=1, prompt_scale=0.05), 5: dict(batch=4, prompt_scale=0.02)}


def _check_step(w, db_pre_k, db_pre_v, db, ref, pairs=None):
    """Compare a whole step: tree metadata, attention, tentative writes,
    accept and commit."""
    check_tree_outputs(db, ref, w)
    compare_out(db.out_f32(), ref["out"], w, pairs)
    cu = w["cu_nodes"]
    k_diff = k_total = 0
    for b in range(w["batch"]):
        if ref["status"][b]:
            continue
        n = int(cu[b + 1] - cu[b])
        got_k = tentative_rows(db_pre_k, w, b, n)
        got_v = tentative_rows(db_pre_v, w, b, n)
        want_k = ref["k_rot_bits"][cu[b]:cu[b + 1]]
        assert np.array_equal(got_v, w["v_new"][cu[b]:cu[b + 1]])
        rope_close(got_k, bf16_bits_to_f64(w["k_new"][cu[b]:cu[b + 1]]),
                   ref["positions"][cu[b]:cu[b + 1]], w)
        d = bf16_ulp_diff(got_k, want_k)
        k_diff += int(np.count_nonzero(d))
        k_total += d.size
    # last-bit differences (float32 rotation vs exact) are rare rounding
    # boundaries: counted over the batch, since a one-node request has too
    # few elements for a per-request rate
    assert k_total == 0 or k_diff / k_total < 1e-3
    check_accept_outputs(db, ref, w)
    # commit: the GPU's own pre-commit pool with the oracle's path applied
    k_exp, v_exp = db_pre_k.copy(), db_pre_v.copy()
    table = np.array(w["block_table"], copy=True)
    nb = np.array(w["n_blocks"], copy=True)
    for b in range(w["batch"]):
        if ref["paths"][b] is None:
            continue
        st, new_len, new_nb, released = kv_commit_ref(k_exp, v_exp, table[b], int(nb[b]),
                                                      int(w["prompt_len"][b]), ref["paths"][b])
        assert st == 0
        nb[b] = new_nb
        assert new_len == ref["new_len"][b] and released == ref["released"][b]
    k_post, v_post = db.cache_bits()
    assert np.array_equal(k_post, k_exp) and np.array_equal(v_post, v_exp)
    assert np.array_equal(db.block_table.cpu().numpy(), ref["block_table"])
    assert np.array_equal(db.n_blocks.cpu().numpy(), ref["n_blocks"])
    assert np.array_equal(db.new_len.cpu().numpy(), ref["new_len"])
    rel = db.released.cpu().numpy()
    cnt = db.released_count.cpu().numpy()
    for b in range(w["batch"]):
        assert cnt[b] == len(ref["released"][b])
        assert rel[b][:cnt[b]].tolist() == ref["released"][b]
        assert np.all(rel[b][cnt[b]:] == -1)


def _run_and_check(w, pairs=None, fused=False):
    db = run_gpu(w, ("build", "attn"))
    pre_k, pre_v = db.cache_bits()
    run_gpu(w, ("accept_commit",) if fused else ("accept", "commit"), db)
    ref = oracle_step(w, sample=pairs)
    _check_step(w, pre_k, pre_v, db, ref, pairs)
    return db, ref


@pytest.mark.parametrize("cfg", [1, 2, 3, 4, 5])
def test_step_small_all_outputs(cfg):
    w = wl.make_config(cfg, **SMALL[cfg])
    _run_and_check(w)


@pytest.mark.parametrize("cfg", [1, 2, 3, 5])
def test_step_small_fused_accept_commit(cfg):
    """tv_accept_commit against the same oracle step as the two calls."""
    w = wl.make_config(cfg, **SMALL[cfg])
    _run_and_check(w, fused=True)


@pytest.mark.parametrize("cfg", [2, 3, 4, 5])
def test_step_full_size_sampled(cfg):
    """Full workload sizes, in the bench's launch configuration; attention
    checked on every (node, head) of each unit whose key range is split
    between CTAs (merged partials) and on sampled outputs of the rest;
    everything else exhaustively."""
    w = wl.make_config(cfg)
    pairs = sample_pairs(w, per_request=3, seed=cfg)
    split, n_split = split_unit_pairs(w, torch.cuda.get_device_properties(0).multi_processor_count)
    assert n_split > 0
    for b, extra in split.items():
        pairs[b] = sorted(set(pairs.get(b, [])) | set(extra))
    _run_and_check(w, pairs)


def test_multistep_ragged_eight_steps():
    """Config-5 style loop: verify -> accept -> commit with block release and
    host re-allocation, 8 steps, both sides evolving their own caches."""
    rng = np.random.default_rng(55)
    w_gpu = wl.make_config(5, batch=6, prompt_scale=0.03)
    w_ref = dict(w_gpu)
    db = DeviceBatch(w_gpu)
    for step in range(8):
        db.tree_build()
        db.attention()
        torch.cuda.synchronize()
        pre_k, pre_v = db.cache_bits()
        db.accept()
        db.commit()
        torch.cuda.synchronize()
        w_ref_step = dict(w_ref)
        ref = oracle_step(w_ref_step)
        w_view = dict(w_ref_step)
        _check_step(w_view, pre_k, pre_v, db, ref)
        # next step: released blocks go back to the free list (host allocator)
        free = list(w_ref["free_blocks"])
        for b in range(w_ref["batch"]):
            free.extend(ref["released"][b])
        state = dict(w_ref, k_cache=ref["k_cache"], v_cache=ref["v_cache"],
                     block_table=ref["block_table"], n_blocks=ref["n_blocks"], free_blocks=free)
        trees = []
        for b in range(w_ref["batch"]):
            n_tree = int(rng.choice([16, 32, 64, 128]))
            trees.append(wl.eagle_tree(rng, 0, int(rng.integers(4, 11)), n_tree, wl.VOCAB_LLAMA,
                                       2.0, until_count=True)[:2])
        w_ref = wl.next_step_inputs(rng, state, ref["new_len"], ref["bonus"], trees)
        db.load_step_inputs(w_ref)
        db.block_table.copy_(torch.from_numpy(w_ref["block_table"]))
        db.n_blocks.copy_(torch.from_numpy(w_ref["n_blocks"]))
        db.w = w_ref


def _custom(geom, trees, plens, seed=0, vocab=100, p_match=0.7, max_nodes=None):
    rng = np.random.default_rng(seed)
    tr = [(np.asarray(p, np.int32), np.asarray(t, np.int32)) for p, t in trees]
    return wl.assemble(rng, geom, plens, tr, vocab, p_match, max_nodes=max_nodes)


def _chain(n):
    return list(range(-1, n - 1)), list(range(n))


def _star(n):
    return [-1] + [0] * (n - 1), list(range(n))


@pytest.mark.parametrize("case", ["empty_prompt", "root_only", "chain_1024", "star_300",
                                  "block_edges", "group16_d64_halfsplit", "tail_g1_16_nodes",
                                  "tail_g16_d64_one_node", "tail_g8_halfsplit", "batch_4096_roots",
                                  "many_tiny_trees", "mixed_unit_shapes"])
def test_attention_edge_cases(case):
    """Degenerate and boundary shapes. The tail_* cases end a KV head's query
    rows with a unit of at most 16 rows after full 256-row units: 16 nodes of
    one head, one node of 16 heads, and 8-head groups of one and two nodes,
    with prompts long enough that those units are also split between CTAs
    and merged. batch_4096_roots is the largest batch the library takes (one
    root node each, prompts of 0-16 tokens: the work plan's prefix over the
    batch at its largest); many_tiny_trees gives every CTA dozens of
    one-tile units in a row. mixed_unit_shapes gives every CTA a run of
    units whose row counts alternate between one and two 128-row tiles (and
    256-row units followed by short remainders), so the CTA's two MMA
    issuers and two softmax groups hand the score buffers back and forth
    between segments."""
    if case == "empty_prompt":
        w = _custom(wl.GEOM_8B, [wl.medusa_tree(np.random.default_rng(1), (4, 3), 100)] * 2, [0, 0])
    elif case == "root_only":
        w = _custom(wl.GEOM_8B, [([-1], [5]), ([-1], [6]), ([-1], [7])], [0, 1, 77])
    elif case == "chain_1024":
        w = _custom(wl.Geometry(2, 2, 128), [_chain(1024)], [37], max_nodes=1024)
    elif case == "star_300":
        w = _custom(wl.Geometry(8, 2, 128), [_star(300), _star(17)], [64, 15])
    elif case == "block_edges":
        rng = np.random.default_rng(3)
        trees = [wl.eagle_tree(rng, 4, 3, 20, 1000)[:2] for _ in range(5)]
        w = _custom(wl.GEOM_8B, trees, [15, 16, 63, 64, 65])
    elif case == "tail_g1_16_nodes":
        w = _custom(wl.Geometry(2, 2, 128), [_star(272), _chain(272)], [3, 700], max_nodes=272)
    elif case == "tail_g16_d64_one_node":
        w = _custom(wl.Geometry(16, 1, 64), [_star(17), _chain(17), _star(17)], [0, 40, 1333])
    elif case == "batch_4096_roots":
        rng = np.random.default_rng(11)
        w = _custom(wl.Geometry(4, 2, 64), [([-1], [int(x)]) for x in rng.integers(0, 100, 4096)],
                    list(rng.integers(0, 17, 4096)))
    elif case == "many_tiny_trees":
        rng = np.random.default_rng(12)
        trees = [wl.eagle_tree(rng, 2, 3, int(rng.integers(1, 6)), 1000)[:2] for _ in range(1500)]
        w = _custom(wl.Geometry(8, 2, 128), trees, list(rng.integers(0, 200, 1500)))
    elif case == "mixed_unit_shapes":
        rng = np.random.default_rng(13)
        sizes = [1, 40, 9, 65, 33, 2, 64, 20, 70, 5] * 6
        trees = [wl.eagle_tree(rng, 0, int(rng.integers(3, 9)), n - 1, 1000, until_count=True)[:2]
                 if n > 1 else ([-1], [1]) for n in sizes]
        w = _custom(wl.GEOM_8B, trees, list(rng.integers(100, 700, len(sizes))))
    elif case == "tail_g8_halfsplit":
        rng = np.random.default_rng(5)
        trees = [wl.eagle_tree(rng, 4, 4, 32, 1000)[:2], _star(34), _chain(33)]
        w = _custom(wl.Geometry(64, 8, 128, rope_style=1), trees, [500, 1000, 77])
    else:
        geom = wl.Geometry(16, 1, 64, rope_style=1)
        rng = np.random.default_rng(4)
        w = _custom(geom, [wl.eagle_tree(rng, 5, 4, 40, 1000)[:2] for _ in range(3)], [5, 300, 129])
    _run_and_check(w)


def test_invalid_tree_and_block_leave_outputs_untouched():
    rng = np.random.default_rng(9)
    trees = [wl.medusa_tree(rng, (3, 2), 100) for _ in range(3)]
    w = _custom(wl.GEOM_8B, trees, [40, 50, 60])
    w["parents"][w["cu_nodes"][1] + 4] = 7            # request 1: forward parent
    w["block_table"][2, 2] = -1                       # request 2: a missing block
    w["n_blocks"][2] = max(w["n_blocks"][2], 3)
    db = DeviceBatch(w)
    sentinel = torch.full_like(db.out, 3.0)
    db.out.copy_(sentinel)
    k0, v0 = db.cache_bits()
    db.tree_build()
    db.attention()
    torch.cuda.synchronize()
    st = db.status.cpu().numpy()
    assert st[0] == 0 and st[1] == 4 and st[2] == 8
    cu = w["cu_nodes"]
    out = db.out.float().cpu().numpy()
    assert np.all(out[cu[1]:cu[3]] == 3.0)
    assert not np.any(out[cu[0]:cu[1]] == 3.0)
    k1, v1 = db.cache_bits()
    for b in (1, 2):
        n = int(cu[b + 1] - cu[b])
        blocks = [int(x) for x in w["block_table"][b][:w["n_blocks"][b]] if x >= 0]
        assert np.array_equal(k1[blocks], k0[blocks]) and np.array_equal(v1[blocks], v0[blocks])
    db.accept()
    db.commit()
    torch.cuda.synchronize()
    assert np.array_equal(db.block_table.cpu().numpy()[1:], w["block_table"][1:])


def test_workspace_reuse_is_deterministic():
    """Repeated calls on one workspace (whose arrival counters each call must
    leave at zero) give identical outputs, including split units."""
    w = wl.make_config(2, batch=4, prompt_scale=0.5)
    db = run_gpu(w, ("build", "attn"))
    out1 = db.out.clone()
    for _ in range(3):
        db.attention()
    torch.cuda.synchronize()
    assert torch.equal(out1, db.out)
