"""GPU parity of tv_tree_mask_dense against the oracle's dense mask
([N, P+N] bool; QLEN_ONLY = its tree columns; additive = 0 / -inf), bit for
bit, on the verification workloads and at odd output alignments."""

import numpy as np
import pytest
import torch

import speculative_decoding_tree_build_gb300 as tv
from oracle import dense_tree_mask_ref
from gen import workloads as wl
from speculative_decoding_tree_build_gb300.build import build

pytestmark = pytest.mark.gpu
I32 = dict(dtype=torch.int32, device="cuda")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build()
    assert torch.cuda.is_available()


def device_tree(w, status=None):
    cu = torch.from_numpy(w["cu_nodes"].astype(np.int32)).cuda()
    plen = torch.from_numpy(np.asarray(w["prompt_len"], np.int32)).cuda()
    total, mn = int(w["cu_nodes"][-1]), w["max_nodes"]
    words = (mn + 31) // 32
    mask = torch.empty(total * words, **I32)
    outs = [torch.empty(total, **I32) for _ in range(5)]
    st = torch.empty(w["batch"], **I32)
    tv.tree_build(torch.from_numpy(w["parents"]).cuda(), cu, plen, mn, mask, *outs, st)
    if status is not None:
        st.copy_(torch.tensor(status, **I32))
    return cu, plen, mask, st


def expected(w, mode, dtype, skip=()):
    blocks = []
    cu = w["cu_nodes"]
    for b in range(w["batch"]):
        par = w["parents"][cu[b]:cu[b + 1]]
        p = int(w["prompt_len"][b])
        m = dense_tree_mask_ref(par, p)
        if mode == tv.MASK_QLEN_ONLY:
            m = m[:, p:]
        blocks.append((b in skip, m))
    return blocks


def run_dense(w, mode, dtype, offset=0, status=None):
    cu, plen, mask, st = device_tree(w, status)
    n_el = tv.dense_mask_elements(w["cu_nodes"], w["prompt_len"], mode)
    tdt = torch.uint8 if dtype == tv.MASK_BOOL else torch.float32
    sentinel = 7 if dtype == tv.MASK_BOOL else 3.5
    buf = torch.full((n_el + offset,), sentinel, dtype=tdt, device="cuda")
    out = buf[offset:]
    tv.tree_mask_dense(mask, cu, plen, st, w["max_nodes"], out, mode, dtype)
    torch.cuda.synchronize()
    assert torch.all(buf[:offset] == sentinel)
    return out.cpu().numpy(), sentinel


def check(w, mode, dtype, offset=0, status=None):
    got, sentinel = run_dense(w, mode, dtype, offset, status)
    skip = {b for b, s in enumerate(status or []) if s}
    pos = 0
    for b, (skipped, m) in enumerate(expected(w, mode, dtype, skip)):
        blk = got[pos:pos + m.size].reshape(m.shape)
        pos += m.size
        if skipped:
            assert np.all(blk == sentinel)
            continue
        want = m.astype(np.uint8) if dtype == tv.MASK_BOOL else np.where(m, 0.0, -np.inf)
        assert np.array_equal(blk, want), b
    assert pos == got.size


@pytest.mark.parametrize("cfg,batch", [(1, 1), (2, 3), (3, 2), (5, 6)])
@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("dtype", [0, 1])
def test_dense_mask_matches_oracle(cfg, batch, mode, dtype):
    w = wl.make_config(cfg, batch=batch, prompt_scale=0.05, cache_fill="zeros")
    check(w, mode, dtype)


@pytest.mark.parametrize("offset", [1, 3, 4, 13])
def test_unaligned_outputs_and_skipped_requests(offset):
    w = wl.make_config(5, batch=5, prompt_scale=0.01, cache_fill="zeros")
    dtype = tv.MASK_BOOL if offset % 4 else tv.MASK_ADDITIVE_F32
    check(w, tv.MASK_FULL, dtype, offset=offset if dtype == tv.MASK_BOOL else offset // 4,
          status=[0, tv.TV_ST["BAD_BLOCK"], 0, 0, tv.TV_ST["BAD_PARENT"]])


def test_dense_mask_bench_workload_full_size():
    w = wl.make_config(2, cache_fill="zeros")
    check(w, tv.MASK_FULL, tv.MASK_BOOL)
    check(w, tv.MASK_FULL, tv.MASK_ADDITIVE_F32)
