"""GPU parity of tv_rejection_accept against the oracle (rejection_walk_ref)
on the same seeded target logits, draft logits, uniforms and Gumbel noise.

The chosen path is exact (float64 sums in both). The kernel reduces the
log-sum-exps in float32, so an acceptance decision or a draw may differ from
the oracle's float64 one only where the oracle's own margin is within float32
rounding: a ratio within 5e-4 (relative) of its uniform, or a draw whose key
at the kernel's token is within 1e-3 of the oracle's best key. Each such case
ends the comparison of that request and is counted; every test allows at most
a couple. Greedy requests (T = 0) must match exactly."""

import numpy as np
import pytest
import torch

import speculative_decoding_tree_build_gb300 as tv
from oracle import chosen_path_ref, rejection_walk_ref
from gen import workloads as wl
from speculative_decoding_tree_build_gb300.build import build

pytestmark = pytest.mark.gpu

RATIO_TOL = 5e-4
KEY_TOL = 1e-3
TEMPS = [0.0, 1.0, 0.7, 1.6, 1.0, 0.0, 0.35, 1.0]


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


def _run(w, inputs, temps, vocab, max_depth=None, status=None, with_noise=True, max_nodes=None):
    logits, draft, gumbel, uniforms, draft_logp = inputs
    cu = _dev(w["cu_nodes"].astype(np.int32))
    md = w["max_depth"] if max_depth is None else max_depth
    bsz = w["batch"]
    path = torch.full((bsz, md + 1), -9, dtype=torch.int32, device="cuda")
    alen = torch.full((bsz,), -9, dtype=torch.int32, device="cuda")
    bonus = torch.full((bsz,), -9, dtype=torch.int32, device="cuda")
    st = torch.zeros(bsz, dtype=torch.int32, device="cuda") if status is None else \
        _dev(np.asarray(status, np.int32))
    tv.rejection_accept(_dev(logits)[:, :vocab], _dev(draft)[:, :vocab],
                        _dev(gumbel)[:, :vocab] if with_noise else None, _dev(uniforms),
                        cu, _dev(np.asarray(temps, np.float32)), _dev(w["parents"]),
                        _dev(w["draft_tokens"]), _dev(draft_logp),
                        w["max_nodes"] if max_nodes is None else max_nodes,
                        path, alen, bonus, st)
    torch.cuda.synchronize()
    return path.cpu().numpy(), alen.cpu().numpy(), bonus.cpu().numpy(), st.cpu().numpy()


def _near_tie_decision(details, k):
    r, ratio = details["ratios"][k]
    return np.isfinite(ratio) and abs(r - ratio) <= RATIO_TOL * max(ratio, 1e-30)


def _near_tie_draw(details, tok):
    key = details["stop"][1]
    return 0 <= tok < len(key) and np.isfinite(key[tok]) and key[tok] >= key.max() - KEY_TOL


def _check(w, inputs, temps, vocab, out, max_depth=None, skip=()):
    """Compares every request with the oracle; returns (accepted depths,
    near-tie count)."""
    logits, draft, gumbel, uniforms, draft_logp = inputs
    path, alen, bonus, st = out
    cu = w["cu_nodes"]
    md = w["max_depth"] if max_depth is None else max_depth
    depths, ties = [], 0
    for b in range(w["batch"]):
        if b in skip:
            continue
        t0, t1 = int(cu[b]), int(cu[b + 1])
        sl = slice(t0, t1)
        with np.errstate(over="ignore", invalid="ignore"):
            rst, racc, rbonus, det = rejection_walk_ref(
                w["parents"][sl], w["draft_tokens"][sl], draft_logp[sl], logits[sl, :vocab],
                draft[sl, :vocab], uniforms[sl], gumbel[sl, :vocab], float(temps[b]), md)
        greedy = float(temps[b]) == 0.0
        if rst != 0:
            if st[b] == tv.TV_ST["PATH_OVERFLOW"] and alen[b] == -9:
                continue
            assert not greedy, f"request {b}"
        else:
            assert st[b] in (0, tv.TV_ST["PATH_OVERFLOW"]), f"request {b}: status {st[b]}"
        if st[b] != 0:
            # overflow on the kernel side only: a decision near a tie made it longer
            ties += 1
            continue
        got = [int(x) for x in path[b, :alen[b] + 1]]
        assert np.all(path[b, alen[b] + 1:] == -1), f"request {b}"
        chosen = det["path"]
        assert got == chosen[:len(got)], f"request {b}: not a prefix of the chosen path"
        if got != racc:
            k = min(len(got), len(racc)) - 1          # first edge decided differently
            assert not greedy and _near_tie_decision(det, k), \
                f"request {b}: accepted {got} vs {racc}"
            ties += 1
            continue
        if bonus[b] != rbonus:
            assert not greedy and _near_tie_draw(det, int(bonus[b])), \
                f"request {b}: bonus {bonus[b]} vs {rbonus}"
            ties += 1
            continue
        depths.append(len(got) - 1)
    return depths, ties


@pytest.mark.parametrize("cfg,batch", [(1, 1), (2, 3), (3, 4), (4, 2), (5, 6)])
def test_rejection_walk_matches_oracle(cfg, batch):
    w = _tree_workload(cfg, batch)
    rng = np.random.default_rng(900 + cfg)
    vocab = w["vocab"]
    inputs = wl.rejection_inputs(rng, w)
    temps = [TEMPS[b % len(TEMPS)] for b in range(batch)]
    out = _run(w, inputs, temps, vocab)
    depths, ties = _check(w, inputs, temps, vocab, out)
    assert ties <= 1 and len(depths) >= batch - 1


@pytest.mark.parametrize("vocab,ld", [(1, 4), (3, 8), (5, 8), (1001, 1004), (4099, 4100),
                                      (32000, 32768), (151936, 151936)])
def test_ragged_vocab_and_row_stride(vocab, ld):
    """Vocabularies that are not a multiple of the cluster slice, rows padded
    past the vocabulary with NaN (which would win a maximum if read)."""
    w = _tree_workload(2, 3, vocab=vocab)
    rng = np.random.default_rng(vocab + 11)
    inputs = wl.rejection_inputs(rng, w, vocab=vocab, ld=ld)
    temps = [1.0, 0.0, 0.8]
    out = _run(w, inputs, temps, vocab)
    assert np.all((out[2] >= 0) & (out[2] < vocab))
    _, ties = _check(w, inputs, temps, vocab, out)
    assert ties <= 1


def _chain(n, vocab):
    return {"batch": 1, "max_nodes": n, "max_depth": n - 1, "vocab": vocab,
            "cu_nodes": np.array([0, n], np.int32),
            "parents": np.arange(-1, n - 1, dtype=np.int32),
            "draft_tokens": np.arange(n, dtype=np.int32) % vocab}


def test_long_chain_spans_several_passes():
    """A 300-node chain whose target and draft rows are equal up to node 150:
    p/q is exactly 1 there, so every one of those edges is accepted and the
    walk crosses several passes of path rows before its first real decision."""
    vocab = 4096
    w = _chain(300, vocab)
    rng = np.random.default_rng(21)
    inputs = wl.rejection_inputs(rng, w, vocab=vocab)
    logits, draft, gumbel, uniforms, draft_logp = inputs
    logits[:150] = draft[:150]
    for t in (1.0, 0.0):
        if t == 0.0:
            # greedy: draft tokens follow the target's argmax for 150 edges
            w["draft_tokens"][1:151] = np.argmax(logits[:150], axis=1)
        out = _run(w, inputs, [t], vocab)
        depths, ties = _check(w, inputs, [t], vocab, out)
        assert ties == 0 and depths[0] >= 150
    # all equal: the whole chain is accepted, and max_depth 200 overflows
    logits[:] = draft
    w["draft_tokens"][1:] = np.arange(1, 300) % vocab
    out = _run(w, inputs, [1.0], vocab)
    assert out[3][0] == 0 and out[1][0] == 299
    assert np.array_equal(out[0][0], np.arange(300))
    _, ties = _check(w, inputs, [1.0], vocab, out)
    assert ties == 0
    out = _run(w, inputs, [1.0], vocab, max_depth=200)
    assert out[3][0] == tv.TV_ST["PATH_OVERFLOW"] and out[1][0] == -9 and out[2][0] == -9


def test_path_choice_and_out_of_vocabulary_token():
    """The walk follows the leaf with the largest cumulative draft
    log-probability (smallest index on ties); a draft token outside the
    vocabulary is rejected."""
    vocab = 1000
    parents = np.array([-1, 0, 0, 1, 1, 2], np.int32)
    logp = np.array([0.0, -0.1, -0.5, -2.0, -1.0, -0.6], np.float32)
    w = {"batch": 1, "max_nodes": 6, "max_depth": 5, "vocab": vocab,
         "cu_nodes": np.array([0, 6], np.int32), "parents": parents,
         "draft_tokens": np.array([0, 10, 20, 30, 40, 50], np.int32)}
    rng = np.random.default_rng(4)
    logits, draft, gumbel, uniforms, _ = wl.rejection_inputs(rng, w, vocab=vocab)
    logits[0, 10] = logits[1, 40] = 50.0                 # greedy accepts 0 -> 1 -> 4
    inputs = (logits, draft, gumbel, uniforms, logp)
    assert chosen_path_ref(parents, logp) == [0, 1, 4]
    path, alen, bonus, st = _run(w, inputs, [0.0], vocab)
    assert st[0] == 0 and alen[0] == 2 and list(path[0, :3]) == [0, 1, 4]
    assert bonus[0] == int(np.argmax(logits[4]))
    _check(w, inputs, [0.0], vocab, (path, alen, bonus, st))
    w["draft_tokens"][4] = vocab + 3                     # now rejected at node 1
    path, alen, bonus, st = _run(w, inputs, [0.0], vocab)
    assert st[0] == 0 and alen[0] == 1 and bonus[0] == int(np.argmax(logits[1]))
    w["draft_tokens"][1] = -1                            # rejected at the root, sampling
    path, alen, bonus, st = _run(w, inputs, [1.0], vocab)
    assert st[0] == 0 and alen[0] == 0 and 0 <= bonus[0] < vocab


def test_status_flags_and_skips():
    w = _tree_workload(2, 7)
    rng = np.random.default_rng(8)
    vocab = w["vocab"]
    inputs = wl.rejection_inputs(rng, w)
    cu = w["cu_nodes"]
    w = dict(w)
    w["parents"] = w["parents"].copy()
    w["parents"][cu[1]] = 0                              # request 1: bad root
    w["parents"][cu[2] + 3] = 5                          # request 2: parent >= own index
    temps = [1.0, 1.0, 1.0, -0.5, float("nan"), 1.0, 0.0]
    status = [0, 0, 0, 0, 0, 64 | 1, 0]                  # request 5 arrives flagged
    out = _run(w, inputs, temps, vocab, status=status)
    path, alen, bonus, st = out
    want = [0, tv.TV_ST["BAD_ROOT"], tv.TV_ST["BAD_PARENT"], tv.TV_ST["BAD_TEMPERATURE"],
            tv.TV_ST["BAD_TEMPERATURE"], 65, 0]
    assert list(st) == want
    for b in (1, 2, 3, 4, 5):
        assert alen[b] == -9 and bonus[b] == -9 and np.all(path[b] == -9)
    _, ties = _check(w, inputs, temps, vocab, out, skip=(1, 2, 3, 4, 5))
    assert ties <= 1
    # sampling without noise: flagged; greedy without noise: fine
    out = _run(w, inputs, [0.0, 0.0, 0.0, 0.0, 0.0, 1.0, 0.0], vocab, with_noise=False)
    assert out[3][5] == tv.TV_ST["BAD_TEMPERATURE"] and out[3][0] == 0 and out[3][6] == 0
    # a request larger than max_nodes
    n0 = int(cu[1] - cu[0])
    out = _run(w, inputs, [0.0] * 7, vocab, max_nodes=n0 - 1)
    assert out[3][0] & tv.TV_ST["BAD_SIZE"]


def test_full_size_eagle_batch():
    """At the bench's size (32 requests, EAGLE-2 trees of 65 nodes, vocab
    32000, mixed temperatures): every request against the oracle."""
    w = _tree_workload(3, 32)
    rng = np.random.default_rng(78)
    vocab = w["vocab"]
    inputs = wl.rejection_inputs(rng, w)
    temps = [TEMPS[b % len(TEMPS)] for b in range(32)]
    out = _run(w, inputs, temps, vocab)
    depths, ties = _check(w, inputs, temps, vocab, out)
    assert ties <= 2 and max(depths) >= 2


def test_ddtree_vocab():
    """Vocabulary 151936 with DDTree trees of 257 nodes (3 requests)."""
    w = _tree_workload(4, 3)
    rng = np.random.default_rng(151937)
    vocab = w["vocab"]
    inputs = wl.rejection_inputs(rng, w)
    temps = [1.0, 0.0, 0.6]
    out = _run(w, inputs, temps, vocab)
    _, ties = _check(w, inputs, temps, vocab, out)
    assert ties <= 1


def test_zero_mass_tokens_and_infinite_logits():
    """-inf logits: a token the target rules out is rejected, one only the
    drafter rules out is accepted; the residual draw skips -inf entries."""
    vocab = 3
    w = {"batch": 3, "max_nodes": 2, "max_depth": 1, "vocab": vocab,
         "cu_nodes": np.array([0, 2, 4, 6], np.int32),
         "parents": np.array([-1, 0, -1, 0, -1, 0], np.int32),
         "draft_tokens": np.array([0, 2, 0, 1, 0, 1], np.int32)}
    tl = np.array([[1.0, 0.5, -np.inf], [0.0, 0.0, 0.0]] * 3, np.float32)
    dl = np.array([[0.0, -np.inf, -np.inf], [0.0, 0.0, 0.0]] * 3, np.float32)
    g = np.zeros((6, vocab), np.float32)
    g[1] = [0.0, 2.0, 0.0]
    g[3] = [3.0, 0.0, 0.0]
    unif = np.array([0.5, 0.5, 0.5, 0.999, 0.5, 0.0], np.float32)
    logp = np.array([0, -1, 0, -1, 0, -1], np.float32)
    inputs = (tl, dl, g, unif, logp)
    temps = [1.0, 1.0, 0.0]
    with np.errstate(divide="ignore", invalid="ignore"):
        out = _run(w, inputs, temps, vocab)
        depths, ties = _check(w, inputs, temps, vocab, out)
    path, alen, bonus, st = out
    assert ties == 0 and list(alen) == [0, 1, 0] and list(bonus) == [1, 0, 0]
