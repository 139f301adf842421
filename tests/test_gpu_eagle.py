"""GPU parity of the EAGLE-2 selection calls (tv_eagle_expand_select,
tv_eagle_rerank) against the oracle, bit for bit: both derive the scores in
float32 in the same order and rank with the same keys."""

import numpy as np
import pytest
import torch

import speculative_decoding_tree_build_gb300 as tv
from oracle import eagle_expand_select_ref, eagle_rerank_ref, eagle_scores_ref, tree_build_ref
from gen import workloads as wl
from speculative_decoding_tree_build_gb300.build import build

pytestmark = pytest.mark.gpu
I32 = dict(dtype=torch.int32, device="cuda")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build()
    assert torch.cuda.is_available()


def pack(requests, max_cands):
    """[(logp, parent, token)] -> padded device arrays + counts."""
    b = len(requests)
    lp = np.zeros((b, max_cands), np.float32)
    par = np.full((b, max_cands), -1, np.int32)
    tok = np.zeros((b, max_cands), np.int32)
    cnt = np.zeros(b, np.int32)
    for i, (l, p, t) in enumerate(requests):
        n = len(l)
        lp[i, :n], par[i, :n], tok[i, :n], cnt[i] = l, p, t, n
    return (torch.from_numpy(lp).cuda(), torch.from_numpy(par).cuda(), torch.from_numpy(tok).cuda(),
            torch.from_numpy(cnt).cuda())


def gpu_select(requests, max_cands, layer, k, status=None):
    lp, par, tok, cnt = pack(requests, max_cands)
    sel = torch.full((len(requests), k), -9, **I32)
    st = torch.zeros(len(requests), **I32) if status is None else \
        torch.tensor(status, **I32)
    tv.eagle_expand_select(lp, par, cnt, layer, k, sel, st)
    torch.cuda.synchronize()
    return sel.cpu().numpy(), st.cpu().numpy()


def gpu_rerank(requests, max_cands, n_keep, roots=None, status=None):
    lp, par, tok, cnt = pack(requests, max_cands)
    b = len(requests)
    parents = torch.full((b * (n_keep + 1),), -9, **I32)
    tokens = torch.full((b * (n_keep + 1),), -9, **I32)
    cu = torch.full((b + 1,), -9, **I32)
    st = torch.zeros(b, **I32) if status is None else torch.tensor(status, **I32)
    rt = None if roots is None else torch.tensor(roots, **I32)
    tv.eagle_rerank(lp, par, tok, cnt, n_keep, parents, tokens, cu, st, root_tokens=rt)
    torch.cuda.synchronize()
    return (parents.cpu().numpy().reshape(b, -1), tokens.cpu().numpy().reshape(b, -1),
            cu.cpu().numpy(), st.cpu().numpy())


def check_rerank(requests, max_cands, n_keep, roots):
    par, tok, cu, st = gpu_rerank(requests, max_cands, n_keep, roots)
    assert cu.tolist() == [i * (n_keep + 1) for i in range(len(requests) + 1)]
    for i, (l, p, t) in enumerate(requests):
        rst, rp, rt, kept = eagle_rerank_ref(l, p, t, n_keep, roots[i])
        if rst:
            assert st[i] == tv.TV_ST["BAD_SIZE"] and np.all(par[i] == -9), i
            continue
        assert st[i] == 0 and np.array_equal(par[i], rp) and np.array_equal(tok[i], rt), i
    return par, tok, cu, st


@pytest.mark.parametrize("batch,layers,topk,keep", [(32, 6, 8, 64), (4, 10, 4, 100),
                                                    (3, 3, 10, 1), (2, 16, 8, 1023)])
def test_expansion_layers_and_rerank_match_oracle(batch, layers, topk, keep):
    """EAGLE-2 expansion driven by the oracle's layer choice (the recipe of
    the EAGLE-2 workload), then every layer's device selection and the rerank
    against the oracle."""
    rng = np.random.default_rng(batch * 100 + layers)
    chooser = lambda lp, par, lay: eagle_expand_select_ref(lp, par, lay, topk)
    reqs = [wl.eagle_candidates(rng, layers, topk, 32000, 2.0, chooser) for _ in range(batch)]
    max_cands = max(len(r[0]) for r in reqs)
    assert max_cands <= 4096
    for layer in range(1, layers + 1):
        sel, st = gpu_select(reqs, max_cands, layer, topk)
        assert np.all(st == 0)
        for i, (l, p, t) in enumerate(reqs):
            want = eagle_expand_select_ref(l, p, layer, topk)
            got = sel[i][sel[i] >= 0]
            assert np.array_equal(got, want) and np.all(sel[i][len(want):] == -1), (layer, i)
    if keep <= min(len(r[0]) for r in reqs):
        check_rerank(reqs, max_cands, keep, list(range(batch)))


def test_random_forests_ties_and_chains():
    rng = np.random.default_rng(7)
    reqs = []
    for m in (5, 64, 700, 4096):
        parent = np.full(m, -1, np.int32)
        for c in range(1, m):
            parent[c] = rng.integers(-1, c)
        reqs.append((np.log(rng.uniform(0.05, 0.95, m)).astype(np.float32), parent,
                     rng.integers(0, 32000, m).astype(np.int32)))
    # exact ties everywhere: equal log-probabilities
    m = 300
    parent = np.array([-1] * 10 + [int(rng.integers(0, c)) for c in range(10, m)], np.int32)
    reqs.append((np.full(m, np.log(0.5), np.float32), parent, np.arange(m, dtype=np.int32)))
    # a chain of 1100 candidates
    m = 1100
    reqs.append((np.full(m, -0.01, np.float32), np.arange(-1, m - 1, dtype=np.int32),
                 np.arange(m, dtype=np.int32)))
    for keep in (1, 5, 300, 1023):
        ok = [r if len(r[0]) >= keep else None for r in reqs]
        sub = [r for r in ok if r is not None]
        check_rerank(sub, 4096, keep, list(range(len(sub))))
    for layer in (1, 2, 3, 7):
        sel, st = gpu_select(reqs, 4096, layer, 16)
        for i, (l, p, t) in enumerate(reqs):
            want = eagle_expand_select_ref(l, p, layer, 16)
            assert np.array_equal(sel[i][:len(want)], want) and np.all(sel[i][len(want):] == -1)


def test_status_cases():
    good = (np.log(np.array([0.6, 0.3, 0.5, 0.4], np.float32)), np.array([-1, -1, 0, 0], np.int32),
            np.array([1, 2, 3, 4], np.int32))
    short = (good[0][:2], good[1][:2], good[2][:2])
    positive = (np.array([-0.5, -0.9, 0.3], np.float32), np.array([-1, -1, 1], np.int32),
                np.array([1, 2, 3], np.int32))
    bad_parent = (good[0], np.array([-1, 2, 0, 0], np.int32), good[2])
    par, tok, cu, st = gpu_rerank([good, short, positive, bad_parent, good], 8, 3,
                                  status=[0, 0, 0, 0, tv.TV_ST["BAD_ROOT"]])
    BS, BP = tv.TV_ST["BAD_SIZE"], tv.TV_ST["BAD_PARENT"]
    assert st.tolist() == [0, BS, 0, BP, tv.TV_ST["BAD_ROOT"]]
    assert np.all(par[[1, 3, 4]] == -9) and np.all(tok[[1, 3, 4]] == -9)
    assert par[0, 0] == -1 and par[2, 0] == -1
    # with n_keep = 2 the positive log-probability breaks prefix closure
    par, tok, cu, st = gpu_rerank([positive], 8, 2)
    assert st.tolist() == [BS]
    sel, st = gpu_select([good, bad_parent], 8, 1, 2)
    assert st.tolist() == [0, BP] and sel[0].tolist() == [0, 1]


def test_rerank_output_feeds_tree_build():
    rng = np.random.default_rng(3)
    batch, keep = 8, 64
    reqs = [wl.eagle_candidates(rng, 6, 8, 32000, 2.0,
                                lambda lp, par, lay: eagle_expand_select_ref(lp, par, lay, 8))
            for _ in range(batch)]
    par, tok, cu, st = gpu_rerank(reqs, 400, keep, list(range(batch)))
    n = keep + 1
    words = (n + 31) // 32
    outs = [torch.empty(batch * n * words, **I32)] + [torch.empty(batch * n, **I32) for _ in range(5)]
    st2 = torch.empty(batch, **I32)
    tv.tree_build(torch.from_numpy(par.reshape(-1)).cuda(), torch.from_numpy(cu).cuda(),
                  torch.zeros(batch, **I32), n, *outs, st2)
    torch.cuda.synchronize()
    assert np.all(st2.cpu().numpy() == 0)
    depth = outs[1].cpu().numpy().reshape(batch, n)
    for b in range(batch):
        assert np.array_equal(depth[b], tree_build_ref(par[b], 0, n)["depth"])
        assert np.all(np.diff(depth[b]) >= 0)
