"""GPU parity of the sampling-acceptance calls (tv_sample_tokens,
tv_sampled_accept) against the oracle on the same seeded logits and Gumbel
noise. Token ids, accepted paths and bonus tokens must match bit for bit: the
kernel takes the oracle's decision in the oracle's precision (float32,
product rounded before the sum, first maximum)."""


import numpy as np
import pytest
import torch

import speculative_decoding_tree_build_gb300 as tv
from oracle import sample_tokens_ref, sampled_walk_ref
from gen import workloads as wl
from speculative_decoding_tree_build_gb300.build import build

pytestmark = pytest.mark.gpu

BAD_TEMPERATURE = tv.TV_ST["BAD_TEMPERATURE"]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build()
    assert torch.cuda.is_available()


def _dev(a, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a))
    return t.to("cuda", dtype=dtype) if dtype is not None else t.cuda()


def _tree_workload(cfg, batch, vocab=None):
    w = wl.make_config(cfg, batch=batch, prompt_scale=0.01, cache_fill="zeros")
    if vocab is not None and vocab != w["vocab"]:
        w = dict(w)
        w["draft_tokens"] = (w["draft_tokens"] % vocab).astype(np.int32)
        w["vocab"] = vocab
    return w


def _run_sample(w, logits, gumbel, temps, vocab, status=None, with_noise=True):
    cu = _dev(w["cu_nodes"].astype(np.int32))
    total = int(w["cu_nodes"][-1])
    lg = _dev(logits)[:, :vocab]
    gb = _dev(gumbel)[:, :vocab] if with_noise else None
    tok = torch.full((total,), -7, dtype=torch.int32, device="cuda")
    st = torch.zeros(w["batch"], dtype=torch.int32, device="cuda") if status is None else \
        _dev(np.asarray(status, np.int32))
    tv.sample_tokens(lg, gb, cu, _dev(np.asarray(temps, np.float32)), w["max_nodes"], tok, st)
    torch.cuda.synchronize()
    return tok.cpu().numpy(), st.cpu().numpy()


def _run_walk(w, logits, gumbel, temps, vocab, max_depth=None, status=None, with_noise=True):
    cu = _dev(w["cu_nodes"].astype(np.int32))
    md = w["max_depth"] if max_depth is None else max_depth
    bsz = w["batch"]
    path = torch.full((bsz, md + 1), -9, dtype=torch.int32, device="cuda")
    alen = torch.full((bsz,), -9, dtype=torch.int32, device="cuda")
    bonus = torch.full((bsz,), -9, dtype=torch.int32, device="cuda")
    st = torch.zeros(bsz, dtype=torch.int32, device="cuda") if status is None else \
        _dev(np.asarray(status, np.int32))
    tv.sampled_accept(_dev(logits)[:, :vocab], _dev(gumbel)[:, :vocab] if with_noise else None,
                      cu, _dev(np.asarray(temps, np.float32)), _dev(w["parents"]),
                      _dev(w["draft_tokens"]), w["max_nodes"], path, alen, bonus, st)
    torch.cuda.synchronize()
    return path.cpu().numpy(), alen.cpu().numpy(), bonus.cpu().numpy(), st.cpu().numpy()


def _check_tokens(w, logits, gumbel, temps, vocab, got):
    cu = w["cu_nodes"]
    for b in range(w["batch"]):
        t0, t1 = int(cu[b]), int(cu[b + 1])
        want = sample_tokens_ref(logits[t0:t1, :vocab], gumbel[t0:t1, :vocab], float(temps[b]))
        assert np.array_equal(got[t0:t1], want), f"request {b}"


def _check_walk(w, logits, gumbel, temps, vocab, path, alen, bonus, st, max_depth=None):
    cu = w["cu_nodes"]
    md = w["max_depth"] if max_depth is None else max_depth
    depths = []
    for b in range(w["batch"]):
        t0, t1 = int(cu[b]), int(cu[b + 1])
        rst, rpath, rbonus = sampled_walk_ref(w["parents"][t0:t1], w["draft_tokens"][t0:t1],
                                              logits[t0:t1, :vocab], gumbel[t0:t1, :vocab],
                                              float(temps[b]), md)
        if rst != 0:
            assert st[b] == tv.TV_ST["PATH_OVERFLOW"] and alen[b] == -9, f"request {b}"
            continue
        assert st[b] == 0 and alen[b] == len(rpath) - 1 and bonus[b] == rbonus, f"request {b}"
        want = np.full(md + 1, -1)
        want[:len(rpath)] = rpath
        assert np.array_equal(path[b], want), f"request {b}"
        depths.append(len(rpath) - 1)
    return depths


TEMPS = [0.0, 1.0, 0.7, 1.6, 1.0, 0.0, 0.35, 1.0]


@pytest.mark.parametrize("cfg,batch", [(1, 1), (2, 3), (3, 2), (4, 1), (5, 6)])
def test_sample_tokens_and_walk_match_oracle(cfg, batch):
    w = _tree_workload(cfg, batch)
    rng = np.random.default_rng(500 + cfg)
    vocab = w["vocab"]
    logits, gumbel = wl.sampling_inputs(rng, w)
    temps = [TEMPS[b % len(TEMPS)] for b in range(batch)]
    tok, st = _run_sample(w, logits, gumbel, temps, vocab)
    assert np.all(st == 0)
    _check_tokens(w, logits, gumbel, temps, vocab, tok)
    path, alen, bonus, st = _run_walk(w, logits, gumbel, temps, vocab)
    _check_walk(w, logits, gumbel, temps, vocab, path, alen, bonus, st)


@pytest.mark.parametrize("vocab,ld", [(1, 4), (3, 8), (5, 8), (1001, 1004), (4099, 4100),
                                      (32000, 32768), (151936, 151936)])
def test_ragged_vocab_and_row_stride(vocab, ld):
    """Vocabularies that are not a multiple of 4 or of the cluster slice, and
    rows padded past the vocabulary with NaN (which would win if read)."""
    w = _tree_workload(2, 2, vocab=vocab)
    rng = np.random.default_rng(vocab)
    logits, gumbel = wl.sampling_inputs(rng, w, vocab=vocab, ld=ld)
    temps = [1.0, 0.0]
    tok, st = _run_sample(w, logits, gumbel, temps, vocab)
    assert np.all(st == 0) and np.all((tok >= 0) & (tok < vocab))
    _check_tokens(w, logits, gumbel, temps, vocab, tok)
    path, alen, bonus, st = _run_walk(w, logits, gumbel, temps, vocab)
    _check_walk(w, logits, gumbel, temps, vocab, path, alen, bonus, st)


def _single_rows(rows, vocab, temps):
    """A batch of one-node requests with the given logits rows."""
    n = len(rows)
    w = {"batch": n, "max_nodes": 1, "max_depth": 0, "vocab": vocab,
         "cu_nodes": np.arange(n + 1, dtype=np.int32), "parents": np.full(n, -1, np.int32),
         "draft_tokens": np.zeros(n, np.int32)}
    return w, np.stack(rows).astype(np.float32), temps


def test_ties_nan_signed_zero_and_infinities():
    vocab = 32000
    z = np.zeros(vocab, np.float32)
    rows, noise_rows, temps = [], [], []

    def add(row, noise, t):
        rows.append(np.asarray(row, np.float32))
        noise_rows.append(np.asarray(noise, np.float32))
        temps.append(t)

    add(z, z, 0.0)                                           # all equal -> 0
    add(z, z, 1.0)
    r = np.full(vocab, -np.inf, np.float32)
    add(r, z, 0.0)                                           # all -inf -> 0
    add(r, z, 1.0)
    r = z.copy(); r[[3999, 4000, 28000]] = 5.0               # across cluster slices
    add(r, z, 0.0)
    add(r, z, 2.0)
    r = z.copy(); r[31999] = 1.0                             # maximum at the last entry
    add(r, z, 0.0)
    r = np.full(vocab, -1.0, np.float32); r[10] = -0.0; r[5] = 0.0
    add(r, z, 0.0)                                           # +0 and -0 tie -> 5
    r = np.full(vocab, -1.0, np.float32); r[10] = 0.0; r[5] = -0.0
    add(r, z, 0.0)
    r = z.copy(); r[[20000, 7]] = np.nan; r[100] = np.inf
    add(r, z, 0.0)                                           # NaN beats +inf, first NaN
    add(r, z, 1.0)
    r = z.copy(); r[[17, 25000]] = np.inf
    add(r, z, 1.0)
    g = z.copy(); g[[12, 31000]] = 3.0                       # noise alone decides
    add(z, g, 1.0)
    rng = np.random.default_rng(3)
    r = rng.integers(-3, 4, size=vocab).astype(np.float32)   # many exact ties
    add(r, np.zeros(vocab, np.float32), 0.5)
    g = (rng.integers(-2, 3, size=vocab) * 0.25).astype(np.float32)
    add(r, g, 1.0)
    # rounding: h * (1/T) is rounded before the noise is added
    r = np.full(vocab, -10.0, np.float32); r[1] = np.float32(16777216.0); r[2] = np.float32(16777218.0)
    g = z.copy(); g[1] = 1.0
    add(r, g, 1.0)
    w, logits, temps = _single_rows(rows, vocab, temps)
    gumbel = np.stack(noise_rows)
    with np.errstate(invalid="ignore", over="ignore"):
        tok, st = _run_sample(w, logits, gumbel, temps, vocab)
        assert np.all(st == 0)
        for i in range(len(rows)):
            want = sample_tokens_ref(logits[i:i + 1], gumbel[i:i + 1], temps[i])[0]
            assert tok[i] == want, (i, tok[i], want)
    assert tok[0] == 0 and tok[2] == 0 and tok[4] == 3999 and tok[6] == 31999
    assert tok[7] == 5 and tok[8] == 5 and tok[9] == 7 and tok[12] == 12
    # the one-node walk returns the sampled token as the bonus
    path, alen, bonus, st = _run_walk(w, logits, gumbel, temps, vocab)
    assert np.all(st == 0) and np.all(alen == 0) and np.array_equal(bonus, tok)


def test_walk_follows_forced_children_to_a_leaf_and_overflows():
    """Targets that always pick a child (huge boost) drive the walk to a leaf;
    a max_depth below that depth reports PATH_OVERFLOW and leaves the outputs
    untouched."""
    w = _tree_workload(3, 4)
    rng = np.random.default_rng(9)
    w = dict(w, p_match=1.0)
    logits, gumbel = wl.sampling_inputs(rng, w, boost=(1e4, 2e4))
    temps = [1.0, 0.0, 0.8, 1.0]
    path, alen, bonus, st = _run_walk(w, logits, gumbel, temps, w["vocab"])
    depths = _check_walk(w, logits, gumbel, temps, w["vocab"], path, alen, bonus, st)
    cu = w["cu_nodes"]
    for b in range(w["batch"]):
        last = path[b][alen[b]]
        assert last not in w["parents"][cu[b]:cu[b + 1]]          # ended at a leaf
    assert min(depths) >= 2
    path, alen, bonus, st = _run_walk(w, logits, gumbel, temps, w["vocab"],
                                      max_depth=min(depths) - 1)
    assert np.all(st == tv.TV_ST["PATH_OVERFLOW"]) and np.all(alen == -9)
    assert np.all(path == -9)


def test_status_flags_and_skips():
    w = _tree_workload(2, 5)
    rng = np.random.default_rng(4)
    vocab = w["vocab"]
    logits, gumbel = wl.sampling_inputs(rng, w)
    temps = [1.0, -1.0, float("nan"), 0.0, 1.0]
    pre = [0, 0, 0, 0, tv.TV_ST["BAD_PARENT"]]
    tok, st = _run_sample(w, logits, gumbel, temps, vocab, status=pre)
    assert st.tolist() == [0, BAD_TEMPERATURE, BAD_TEMPERATURE, 0, tv.TV_ST["BAD_PARENT"]]
    cu = w["cu_nodes"]
    for b in (1, 2, 4):
        assert np.all(tok[cu[b]:cu[b + 1]] == -7)
    for b in (0, 3):
        want = sample_tokens_ref(logits[cu[b]:cu[b + 1]], gumbel[cu[b]:cu[b + 1]], temps[b])
        assert np.array_equal(tok[cu[b]:cu[b + 1]], want)
    path, alen, bonus, st = _run_walk(w, logits, gumbel, temps, vocab, status=pre)
    assert st.tolist() == [0, BAD_TEMPERATURE, BAD_TEMPERATURE, 0, tv.TV_ST["BAD_PARENT"]]
    assert np.all(alen[[1, 2, 4]] == -9) and np.all(bonus[[1, 2, 4]] == -9)
    # no noise array: greedy requests run, sampled ones are flagged
    temps = [0.0, 1.0, 0.0, 0.5, 0.0]
    tok, st = _run_sample(w, logits, gumbel, temps, vocab, with_noise=False)
    assert st.tolist() == [0, BAD_TEMPERATURE, 0, BAD_TEMPERATURE, 0]
    for b in (0, 2, 4):
        want = sample_tokens_ref(logits[cu[b]:cu[b + 1]], gumbel[cu[b]:cu[b + 1]], 0.0)
        assert np.array_equal(tok[cu[b]:cu[b + 1]], want)
    path, alen, bonus, st = _run_walk(w, logits, gumbel, temps, vocab, with_noise=False)
    assert st.tolist() == [0, BAD_TEMPERATURE, 0, BAD_TEMPERATURE, 0]
    _check_walk({**w, "batch": 1, "cu_nodes": cu[:2]}, logits, gumbel, temps, vocab,
                path[:1], alen[:1], bonus[:1], st[:1])


def test_walk_equals_sample_then_greedy_accept_full_size():
    """At the bench's size (32 requests, EAGLE-2 trees of 65 nodes, vocab
    32000, mixed temperatures): every node's token against the oracle, the
    fused walk against the oracle walk, and the fused walk against
    tv_sample_tokens followed by tv_greedy_accept on the device."""
    w = _tree_workload(3, 32)
    rng = np.random.default_rng(77)
    vocab = w["vocab"]
    logits, gumbel = wl.sampling_inputs(rng, w)
    temps = [TEMPS[b % len(TEMPS)] for b in range(32)]
    tok, st = _run_sample(w, logits, gumbel, temps, vocab)
    assert np.all(st == 0)
    _check_tokens(w, logits, gumbel, temps, vocab, tok)
    path, alen, bonus, st = _run_walk(w, logits, gumbel, temps, vocab)
    depths = _check_walk(w, logits, gumbel, temps, vocab, path, alen, bonus, st)
    assert max(depths) >= 2
    # device chain: tree_build links -> greedy_accept on the sampled tokens
    total = int(w["cu_nodes"][-1])
    mn = w["max_nodes"]
    words = (mn + 31) // 32
    cu = _dev(w["cu_nodes"].astype(np.int32))
    i32 = dict(dtype=torch.int32, device="cuda")
    mask = torch.empty(total * words, **i32)
    depth, pos, ridx, nxt, sib = (torch.empty(total, **i32) for _ in range(5))
    st2 = torch.empty(32, **i32)
    tv.tree_build(_dev(w["parents"]), cu, _dev(w["prompt_len"].astype(np.int32)), mn, mask, depth,
                  pos, ridx, nxt, sib, st2)
    p2 = torch.empty((32, w["max_depth"] + 1), **i32)
    l2, b2 = torch.empty(32, **i32), torch.empty(32, **i32)
    tv.greedy_accept(_dev(tok), _dev(w["draft_tokens"]), cu, nxt, sib, mn, p2, l2, b2, st2)
    torch.cuda.synchronize()
    assert np.all(st2.cpu().numpy() == 0)
    assert np.array_equal(p2.cpu().numpy(), path)
    assert np.array_equal(l2.cpu().numpy(), alen) and np.array_equal(b2.cpu().numpy(), bonus)


def test_ddtree_vocab_walk_sampled_rows():
    """Vocabulary 151936 with DDTree trees of 257 nodes (4 requests): the
    walk against the oracle walk, and per-node tokens on every node."""
    w = _tree_workload(4, 4)
    rng = np.random.default_rng(151936)
    vocab = w["vocab"]
    logits, gumbel = wl.sampling_inputs(rng, w, boost=(12.0, 20.0))
    temps = [1.0, 0.6, 0.0, 1.4]
    path, alen, bonus, st = _run_walk(w, logits, gumbel, temps, vocab)
    _check_walk(w, logits, gumbel, temps, vocab, path, alen, bonus, st)
    tok, st = _run_sample(w, logits, gumbel, temps, vocab)
    assert np.all(st == 0)
    _check_tokens(w, logits, gumbel, temps, vocab, tok)
