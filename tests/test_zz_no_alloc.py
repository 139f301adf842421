"""The allocation-free attention entry point (tv_tree_attention_verify_noalloc).

It serves callers that cannot allocate device memory (a plugin that only gets
a stream and tensors from its host framework, code running while another
component owns the device memory pool, a loop that must not call cudaMalloc).
Its scratch lives in a fixed array inside the library, so these tests check
that it gives the same outputs as the workspace entry point, bit for bit, call
after call on the shared array, and that oversized work is refused up front.

This file is collected last on purpose: if it fails, a run that stops at the
first failure has already run every other test.
"""

import ctypes

import numpy as np
import pytest
import torch

import speculative_decoding_tree_build_gb300 as tv
from gen import workloads as wl
from speculative_decoding_tree_build_gb300.build import build
from speculative_decoding_tree_build_gb300.step import DeviceBatch

pytestmark = pytest.mark.gpu


def _noalloc_call(lib, db, out, status):
    """One call through the C ABI with raw device pointers."""
    return lib.tv_tree_attention_verify_noalloc(
        ctypes.byref(db.g), db.batch, db.max_nodes, db.q.data_ptr(), db.k_new.data_ptr(),
        db.v_new.data_ptr(), db.cu_nodes.data_ptr(), db.positions.data_ptr(),
        db.mask.data_ptr(), db.prompt_len.data_ptr(), db.block_table.data_ptr(),
        db.n_blocks.data_ptr(), db.block_table.shape[1], db.k_cache.data_ptr(),
        db.v_cache.data_ptr(), db.k_cache.shape[0], out.data_ptr(), status.data_ptr(),
        torch.cuda.current_stream().cuda_stream)


def _same(got, want):
    """Both entry points run the same kernels with the same work plan, so the
    outputs must agree bit for bit; any difference would point at scratch
    records left over from a previous call."""
    g = got.view(torch.int16).cpu().numpy()
    r = want.view(torch.int16).cpu().numpy()
    assert np.array_equal(g, r), f"{int(np.count_nonzero(g != r))} outputs differ"
    assert np.all(np.isfinite(got.float().cpu().numpy()))


@pytest.mark.parametrize("cfg", [2, 5])
def test_noalloc_matches_workspace_entry_point_twice(cfg):
    build()
    lib = tv.load()
    w = wl.make_config(cfg, batch=4, prompt_scale=0.25 if cfg == 2 else 0.03)
    db = DeviceBatch(w)
    db.tree_build()
    db.attention()                                   # caller-provided workspace
    torch.cuda.synchronize()
    want = db.out.clone()
    assert int(db.status.abs().sum()) == 0
    for _ in range(2):                               # the static scratch is reused
        out = torch.full_like(db.out, 7.0)
        status = torch.zeros_like(db.status)
        assert _noalloc_call(lib, db, out, status) == 0
        torch.cuda.synchronize()
        assert int(status.abs().sum()) == 0
        _same(out, want)


def test_noalloc_rejects_work_larger_than_its_scratch():
    build()
    lib = tv.load()
    w = wl.make_config(2, batch=2, prompt_scale=0.1)
    db = DeviceBatch(w)
    big = tv.geom(1024, 64, 128)          # 64 KV heads x 4096 requests x 1024-node trees
    need = tv.workspace_bytes(big, 4096, 1024)
    assert need > (64 << 20)
    out = torch.zeros_like(db.out)
    rc = lib.tv_tree_attention_verify_noalloc(
        ctypes.byref(big), 4096, 1024, db.q.data_ptr(), db.k_new.data_ptr(),
        db.v_new.data_ptr(), db.cu_nodes.data_ptr(), db.positions.data_ptr(),
        db.mask.data_ptr(), db.prompt_len.data_ptr(), db.block_table.data_ptr(),
        db.n_blocks.data_ptr(), db.block_table.shape[1], db.k_cache.data_ptr(),
        db.v_cache.data_ptr(), db.k_cache.shape[0], out.data_ptr(), db.status.data_ptr(),
        torch.cuda.current_stream().cuda_stream)
    assert rc == -4 and tv.status_string(rc) == "TV_ERR_WORKSPACE"
    # refused before any launch: nothing was written
    torch.cuda.synchronize()
    assert int(out.view(torch.int16).abs().sum()) == 0
    assert int(db.status.abs().sum()) == 0
