"""GPU parity of the DDTree construction calls against the oracle.

tv_ddtree_topk: token ranks bit for bit (they are decided by comparisons of
the input logits), log-probabilities within 1e-5 (the row's log-sum-exp is
accumulated in float32). tv_ddtree_build: fed the same float32
log-probabilities as the oracle, it must give the oracle's tree, except where
the kernel's float32 prefix sums decide between prefixes whose float64 scores
(the oracle's) lie within float32 rounding of each other: such a tree is
checked to be a valid top-B within that rounding bound, and the cases are
counted and bounded. The two chained (logits -> tree) may differ from the
oracle only where two prefix scores are within the log-sum-exp error; such a
tree is checked the same way."""

import numpy as np
import pytest
import torch

import speculative_decoding_tree_build_gb300 as tv
from oracle import ddtree_build_ref, tree_build_ref, topk_logprobs_ref
from speculative_decoding_tree_build_gb300.build import build

pytestmark = pytest.mark.gpu
LOGQ_ATOL = 1e-5


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build()
    assert torch.cuda.is_available()


def gpu_topk(logits, k, ld=None):
    rows, vocab = logits.shape
    ld = -(-vocab // 4) * 4 if ld is None else ld            # rows 16-byte aligned
    full = np.full((rows, ld), np.nan, np.float32)
    full[:, :vocab] = logits
    lg = torch.from_numpy(full).cuda()[:, :vocab]
    tt = torch.full((rows, k), -5, dtype=torch.int32, device="cuda")
    tq = torch.full((rows, k), 7.0, dtype=torch.float32, device="cuda")
    tv.ddtree_topk(lg, k, tt, tq)
    torch.cuda.synchronize()
    return tt.cpu().numpy(), tq.cpu().numpy()


def check_topk(logits, k, ld=None):
    toks, lq = gpu_topk(logits, k, ld)
    rt, rq = topk_logprobs_ref(logits, k)
    assert np.array_equal(toks, rt)
    fin = np.isfinite(rq)
    assert np.array_equal(fin, np.isfinite(lq))
    assert np.all(lq[~fin] == -np.inf)
    if fin.any():
        assert np.max(np.abs(lq[fin].astype(np.float64) - rq[fin])) < LOGQ_ATOL


@pytest.mark.parametrize("rows,vocab,k,sigma", [(4, 151936, 256, 3.0), (16, 32000, 64, 1.0),
                                                (3, 4097, 1024, 2.0), (5, 1001, 1, 3.0),
                                                (2, 300, 300, 1.0), (3, 8192, 7, 0.01)])
def test_topk_matches_oracle(rows, vocab, k, sigma):
    rng = np.random.default_rng(rows * 1000 + k)
    logits = rng.normal(0, sigma, size=(rows, vocab)).astype(np.float32)
    check_topk(logits, k)


def test_topk_ties_masks_and_orderings():
    rng = np.random.default_rng(2)
    v = 20000
    rows = [
        rng.integers(-3, 4, size=v).astype(np.float32),           # massive exact ties
        np.zeros(v, np.float32),                                  # all equal
        np.arange(v, dtype=np.float32) * 1e-3,                    # ascending: every logit enters
        -np.arange(v, dtype=np.float32) * 1e-3,                   # descending
        np.where(rng.random(v) < 0.9, -np.inf, rng.normal(0, 2, v)).astype(np.float32),
        np.full(v, -np.inf, np.float32),                          # nothing finite
        np.concatenate([np.full(v - 3, -np.inf), [1.0, 1.0, -2.0]]).astype(np.float32),
    ]
    check_topk(np.stack(rows), 256, ld=20004)
    check_topk(np.stack(rows)[:, :9999], 1000, ld=10000)


def gpu_build(logq, toks, budget, roots=None):
    batch, L, k = logq.shape
    n = tv.ddtree_nodes(L, k, budget)
    par = torch.full((batch * n,), -7, dtype=torch.int32, device="cuda")
    tok = torch.full((batch * n,), -7, dtype=torch.int32, device="cuda")
    cu = torch.full((batch + 1,), -7, dtype=torch.int32, device="cuda")
    rt = None if roots is None else torch.from_numpy(np.asarray(roots, np.int32)).cuda()
    tv.ddtree_build(torch.from_numpy(np.ascontiguousarray(logq, np.float32)).cuda(),
                    torch.from_numpy(np.ascontiguousarray(toks, np.int32)).cuda(), budget, par,
                    tok, cu, rt)
    torch.cuda.synchronize()
    return n, par.cpu().numpy().reshape(batch, n), tok.cpu().numpy().reshape(batch, n), cu.cpu().numpy()


def _gpu_tuples(par, tok, toks_ranked):
    """Rank tuples (1-based ranks per depth) of a flattened tree's nodes."""
    n = len(par)
    depth = np.zeros(n, int)
    tup = [()] * n
    for i in range(1, n):
        depth[i] = depth[par[i]] + 1
        r = int(np.nonzero(toks_ranked[depth[i] - 1] == tok[i])[0][0]) + 1
        tup[i] = tup[par[i]] + (r,)
    return depth, tup


def check_top_b_within(par, tok, logq, toks_ranked, tol):
    """A tree that differs from the oracle's: it must still be a top-B under
    the float64 prefix scores within ``tol`` (prefix-closed and flattened
    depth by depth, no prefix outside it better than one inside by more than
    tol, and pop order within a depth non-increasing up to tol)."""
    L, K = logq.shape
    n = len(par)
    assert par[0] == -1 and np.all(par[1:] < np.arange(1, n))

    def score(rho):
        return float(sum(float(logq[i, r - 1]) for i, r in enumerate(rho)))
    depth, tup = _gpu_tuples(par, tok, toks_ranked)
    assert np.all(np.diff(depth) >= 0)
    inside = set(tup[1:])
    assert len(inside) == n - 1
    sc = [score(t) for t in tup[1:]]
    worst_in = min(sc)
    frontier = []
    for t in list(inside) + [()]:
        if len(t) < L and t + (1,) not in inside:
            frontier.append(t + (1,))
        if t and t[-1] < K and t[:-1] + (t[-1] + 1,) not in inside:
            frontier.append(t[:-1] + (t[-1] + 1,))
    if frontier:
        assert max(score(t) for t in frontier) <= worst_in + tol
    for i in range(1, n - 1):
        if depth[i] == depth[i + 1]:
            assert sc[i - 1] >= sc[i] - tol


def f32_sum_tol(logq):
    """Bound on the difference between a float32 and a float64 sum of up to
    L of the given values: L roundings of a partial sum no larger than the
    largest possible prefix magnitude."""
    L = logq.shape[0]
    mag = np.where(np.isfinite(logq), np.abs(logq.astype(np.float64)), 0.0)
    big = float(np.sum(np.max(mag, axis=1)))
    return 2.0 * L * 2.0 ** -24 * (1.0 + big)


@pytest.mark.parametrize("batch,L,V,budget,sigma", [(16, 16, 151936, 256, 3.0), (4, 3, 4, 6, 1.0),
                                                    (3, 16, 2000, 1023, 3.0), (2, 1, 500, 40, 1.0),
                                                    (5, 64, 50, 300, 0.5), (2, 4, 2, 100, 1.0),
                                                    (3, 16, 1000, 1, 3.0)])
def test_build_matches_oracle_on_oracle_logq(batch, L, V, budget, sigma):
    rng = np.random.default_rng(batch * 7 + L)
    k = min(budget, V)
    logits = rng.normal(0, sigma, size=(batch, L, V)).astype(np.float32)
    logq = np.zeros((batch, L, k), np.float32)
    toks = np.zeros((batch, L, k), np.int32)
    for b in range(batch):
        t, q = topk_logprobs_ref(logits[b], k)
        toks[b], logq[b] = t, q.astype(np.float32)
    roots = rng.integers(0, V, size=batch)
    n, par, tok, cu = gpu_build(logq, toks, budget, roots)
    assert cu.tolist() == [b * n for b in range(batch + 1)]
    near_ties = 0
    for b in range(batch):
        rp, rt, rd, rs, pops = ddtree_build_ref(logq[b], toks[b], budget, int(roots[b]))
        assert len(rp) == n
        if np.array_equal(par[b], rp) and np.array_equal(tok[b], rt):
            continue
        near_ties += 1                 # float32 vs float64 prefix sums at a near-tie
        assert tok[b][0] == roots[b]
        check_top_b_within(par[b], tok[b], logq[b], toks[b], f32_sum_tol(logq[b]))
    assert near_ties <= 2, f"{near_ties} of {batch} trees differ"


def test_build_ties_and_dead_positions():
    # uniform positions (all scores of a depth equal) and a position with no
    # finite logit (log q = -inf): the tie rules decide everything
    L, k = 4, 8
    logq = np.full((2, L, k), -np.log(8.0), np.float32)
    logq[1, 2] = -np.inf
    toks = np.tile(np.arange(k, dtype=np.int32), (2, L, 1)) + 100
    n, par, tok, cu = gpu_build(logq, toks, 200)
    for b in range(2):
        # equal float32 values sum to the same score in float32 and float64
        # alike here, so the tie rules alone decide: exact agreement
        rp, rt, *_ = ddtree_build_ref(logq[b], toks[b], 200)
        assert np.array_equal(par[b], rp) and np.array_equal(tok[b], rt)


def _scores_by_prefix(logq):
    """float64 score of a rank tuple under the given per-depth values."""
    def score(rho):
        return float(sum(float(logq[i, r - 1]) for i, r in enumerate(rho)))
    return score


def test_chained_topk_and_build_from_logits():
    """The DDTree workload's recipe: 16 requests, L = 16, vocabulary 151936, N(0, 3)
    logits, budget 256; the chained GPU result against the oracle from the
    same logits, then fed to tv_tree_build."""
    rng = np.random.default_rng(44)
    batch, L, V, B = 16, 16, 151936, 256
    logits = rng.normal(0, 3.0, size=(batch * L, V)).astype(np.float32)
    toks_g, lq_g = gpu_topk(logits, B)
    n, par, tok, cu = gpu_build(lq_g.reshape(batch, L, B), toks_g.reshape(batch, L, B), B)
    rt, rq = topk_logprobs_ref(logits, B)
    assert np.array_equal(toks_g, rt)
    mismatches = 0
    for b in range(batch):
        rows = slice(b * L, (b + 1) * L)
        rp, rtk, rd, rs, pops = ddtree_build_ref(rq[rows], rt[rows], B)
        if np.array_equal(par[b], rp) and np.array_equal(tok[b], rtk):
            continue
        mismatches += 1
        # a near-tie: the GPU tree must still be a top-B under exact scores
        # within the log-sum-exp error (prefix-closed, no outside prefix
        # better than an inside one by more than the tolerance)
        score = _scores_by_prefix(rq[rows])
        rank_of = {int(t): i + 1 for i, t in enumerate(rt[rows][0])}
        assert par[b][0] == -1 and np.all(par[b][1:] < np.arange(1, n))
        depth = np.zeros(n, int)
        tup = [()] * n
        for i in range(1, n):
            depth[i] = depth[par[b][i]] + 1
            pos = depth[i] - 1
            r = int(np.nonzero(rt[rows][pos] == tok[b][i])[0][0]) + 1
            tup[i] = tup[par[b][i]] + (r,)
        inside = set(tup[1:])
        worst_in = min(score(t) for t in inside)
        frontier = []
        for t in list(inside) + [()]:
            if len(t) < L and t + (1,) not in inside:
                frontier.append(t + (1,))
            if t and t[-1] < B and t[:-1] + (t[-1] + 1,) not in inside:
                frontier.append(t[:-1] + (t[-1] + 1,))
        best_out = max(score(t) for t in frontier)
        assert best_out <= worst_in + 2 * LOGQ_ATOL * L
    assert mismatches <= 2
    # the trees feed the verification step directly
    total = batch * n
    i32 = dict(dtype=torch.int32, device="cuda")
    mn = n
    words = (mn + 31) // 32
    outs = [torch.empty(total * words, **i32)] + [torch.empty(total, **i32) for _ in range(5)]
    st = torch.empty(batch, **i32)
    tv.tree_build(torch.from_numpy(par.reshape(-1)).cuda(), torch.from_numpy(cu).cuda(),
                  torch.zeros(batch, **i32), mn, *outs, st)
    torch.cuda.synchronize()
    assert np.all(st.cpu().numpy() == 0)
    depth_gpu = outs[1].cpu().numpy().reshape(batch, n)
    for b in range(batch):
        ref = tree_build_ref(par[b], 0, mn)
        assert np.array_equal(depth_gpu[b], ref["depth"])
        assert np.all(np.diff(depth_gpu[b]) >= 0)            # flattened depth by depth
