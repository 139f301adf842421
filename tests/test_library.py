"""The C-ABI library builds, loads without a GPU, exports every function that
include/treeverify.h declares, and rejects bad arguments on the host before
touching the device."""

import ctypes
import os
import re

import pytest

import speculative_decoding_tree_build_gb300 as tv
from speculative_decoding_tree_build_gb300.build import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build()
    return tv.load()


def header_functions():
    names = []
    for f in os.listdir(os.path.join(ROOT, "include")):
        if f.endswith(".h"):
            with open(os.path.join(ROOT, "include", f), encoding="utf-8") as fh:
                text = fh.read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(tv_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_step_calls():
    names = header_functions()
    for want in ("tv_tree_build", "tv_tree_attention_verify", "tv_greedy_accept", "tv_kv_commit",
                 "tv_sample_tokens", "tv_sampled_accept", "tv_rejection_accept", "tv_ddtree_topk", "tv_ddtree_build",
                 "tv_ddtree_nodes", "tv_eagle_expand_select", "tv_eagle_rerank",
                 "tv_tree_mask_dense", "tv_accept_commit",
                 "tv_workspace_bytes",
                 "tv_status_string", "tv_version"):
        assert want in names


def test_library_exports_every_declared_symbol(lib):
    raw = ctypes.CDLL(tv.lib_path)
    for name in header_functions():
        assert hasattr(raw, name), name


def test_status_strings(lib):
    assert tv.status_string(0) == "TV_OK"
    assert tv.status_string(-1) == "TV_ERR_NULL_POINTER"
    assert tv.status_string(8) == "TV_ST_BAD_BLOCK"
    assert tv.status_string(64) == "TV_ST_BAD_TEMPERATURE"
    assert tv.version() >= 1


FAKE = 0x10000  # a non-null, 256-byte aligned value; never dereferenced


def test_host_validation_rejects_before_launch(lib):
    L = lib
    P = FAKE
    # tree build
    assert L.tv_tree_build(P, P, P, -1, 8, P, P, P, P, P, P, P, None) == -3
    assert L.tv_tree_build(P, P, P, 1, 0, P, P, P, P, P, P, P, None) == -3
    assert L.tv_tree_build(P, P, P, 1, 1025, P, P, P, P, P, P, P, None) == -3
    assert L.tv_tree_build(None, P, P, 1, 8, P, P, P, P, P, P, P, None) == -1
    assert L.tv_tree_build(None, None, None, 0, 8, None, None, None, None, None, None, None,
                           None) == 0
    # accept
    assert L.tv_greedy_accept(P, P, P, P, P, 1, 8, -1, P, P, P, P, None) == -3
    assert L.tv_greedy_accept(P, None, P, P, P, 1, 8, 4, P, P, P, P, None) == -1
    # geometry checks
    g = tv.geom(32, 8, 128)
    bad_d = tv.geom(32, 8, 96)
    bad_group = tv.geom(30, 8, 128)
    bad_block = tv.geom(32, 8, 128, block_size=32)
    bad_style = tv.geom(32, 8, 128, rope_style=2)
    for bg in (bad_d, bad_group, bad_block, bad_style):
        assert L.tv_kv_commit(ctypes.byref(bg), 1, P, P, 4, P, P, P, 8, P, P, 10, P, P, P, P,
                              None) == -2
    assert L.tv_kv_commit(ctypes.byref(g), 1, P, P, 4, P, None, P, 8, P, P, 10, P, P, P, P,
                          None) == -1
    # a K+V row of every KV head must fit the commit's 64 KiB staging buffer:
    # 256 KV heads x 128 x 2 x 2 bytes = 128 KiB does not (refused before any launch)
    wide = tv.geom(256, 256, 128)
    assert L.tv_kv_commit(ctypes.byref(wide), 1, P, P, 4, P, P, P, 8, P, P, 10, P, P, P, P,
                          None) == -2
    assert L.tv_accept_commit(ctypes.byref(wide), P, P, P, P, P, 1, 41, 4, P, P, P, P, P, P, 8,
                              P, P, 10, P, P, P, P, None) == -2
    fits = tv.geom(128, 128, 128)                         # exactly 64 KiB per row
    assert L.tv_kv_commit(ctypes.byref(fits), 0, None, None, 4, None, None, None, 8, None, None,
                          10, None, None, None, None, None) == 0
    assert L.tv_kv_commit(ctypes.byref(g), 0, None, None, 4, None, None, None, 8, None, None, 10,
                          None, None, None, None, None) == 0
    # attention
    args = [P, P, P, P, P, P, P, P, P, 8, P, P, 100, P, P, 1 << 20, P, None]
    assert L.tv_tree_attention_verify(ctypes.byref(bad_d), 1, 41, *args) == -2
    assert L.tv_tree_attention_verify(ctypes.byref(g), 1, 0, *args) == -3
    assert L.tv_tree_attention_verify(ctypes.byref(g), 0, 41, *args) == 0
    nul = list(args)
    nul[0] = None
    assert L.tv_tree_attention_verify(ctypes.byref(g), 1, 41, *nul) == -1
    mis = list(args)
    mis[0] = FAKE + 2
    assert L.tv_tree_attention_verify(ctypes.byref(g), 1, 41, *mis) == -5
    mis = list(args)
    mis[14] = FAKE + 16                                   # workspace needs 256-byte alignment
    assert L.tv_tree_attention_verify(ctypes.byref(g), 1, 41, *mis) == -5
    assert L.tv_workspace_bytes(ctypes.byref(bad_d), 1, 41, ctypes.byref(ctypes.c_size_t())) == -2
    assert L.tv_workspace_bytes(ctypes.byref(g), 1, 41, None) == -1
    # sampling: (logits, ld, gumbel, ld, cu, temperature, batch, max_nodes, vocab, tokens, status)
    S = L.tv_sample_tokens
    assert S(P, 32000, P, 32000, P, P, 0, 8, 32000, P, P, None) == 0
    assert S(P, 32000, P, 32000, P, P, -1, 8, 32000, P, P, None) == -3
    assert S(P, 32000, P, 32000, P, P, 1, 1025, 32000, P, P, None) == -3
    assert S(P, 32000, P, 32000, P, P, 1, 8, 0, P, P, None) == -3
    assert S(P, 100, P, 32000, P, P, 1, 8, 32000, P, P, None) == -3     # ld < vocab
    assert S(P, 32000, P, 100, P, P, 1, 8, 32000, P, P, None) == -3
    assert S(None, 32000, P, 32000, P, P, 1, 8, 32000, P, P, None) == -1
    assert S(P, 32000, P, 32000, P, None, 1, 8, 32000, P, P, None) == -1
    assert S(P + 4, 32000, P, 32000, P, P, 1, 8, 32000, P, P, None) == -5
    assert S(P, 32002, P, 32000, P, P, 1, 8, 32000, P, P, None) == -5   # row stride % 4
    assert S(P, 32000, P + 8, 32000, P, P, 1, 8, 32000, P, P, None) == -5
    A = L.tv_sampled_accept
    args = [P, 32000, P, 32000, P, P, P, P, 1, 8, 4, 32000, P, P, P, P, None]
    assert A(*args[:8], 0, *args[9:]) == 0
    assert A(*args[:10], -1, *args[11:]) == -3                          # max_depth
    assert A(*args[:6], None, *args[7:]) == -1                          # parents
    assert A(P + 4, *args[1:]) == -5
    # rejection-sampling acceptance
    Rj = L.tv_rejection_accept
    args = [P, 32000, P, 32000, P, 32000, P, P, P, P, P, P, 1, 8, 4, 32000, P, P, P, P, None]
    assert Rj(*args[:12], 0, *args[13:]) == 0                           # empty batch
    assert Rj(*args[:13], 1025, *args[14:]) == -3                       # max_nodes
    assert Rj(*args[:14], -1, *args[15:]) == -3                         # max_depth
    assert Rj(*args[:15], 0, *args[16:]) == -3                          # vocab
    assert Rj(P, 100, *args[2:]) == -3                                  # logits ld < vocab
    assert Rj(*args[:3], 100, *args[4:]) == -3                          # draft ld < vocab
    assert Rj(*args[:5], 100, *args[6:]) == -3                          # gumbel ld < vocab
    assert Rj(*args[:4], None, 0, *args[6:12], 0, *args[13:]) == 0      # noise optional
    assert Rj(*args[:2], None, *args[3:]) == -1                         # draft logits
    assert Rj(*args[:11], None, *args[12:]) == -1                       # draft_logp
    assert Rj(*args[:19], None, None) == -1                             # status
    # DDTree construction
    assert L.tv_ddtree_nodes(16, 256, 256) == 257
    assert L.tv_ddtree_nodes(3, 4, 6) == 7 and L.tv_ddtree_nodes(4, 2, 100) == 31
    assert L.tv_ddtree_nodes(0, 4, 6) == -3 and L.tv_ddtree_nodes(3, 4, 1024) == -3
    T = L.tv_ddtree_topk
    assert T(P, 1000, 0, 1000, 8, P, P, None) == 0
    assert T(P, 1000, 4, 1000, 1001, P, P, None) == -3      # k > vocab
    assert T(P, 2000, 4, 2000, 1025, P, P, None) == -3      # k > 1024
    assert T(P, 999, 4, 1000, 8, P, P, None) == -3          # ld < vocab
    assert T(None, 1000, 4, 1000, 8, P, P, None) == -1
    assert T(P + 4, 1000, 4, 1000, 8, P, P, None) == -5
    assert T(P, 1002, 4, 1000, 8, P, P, None) == -5
    Bd = L.tv_ddtree_build
    assert Bd(P, P, 0, 16, 256, 256, None, P, P, P, None) == 0
    assert Bd(P, P, 2, 16, 256, 1024, None, P, P, P, None) == -3
    assert Bd(P, P, 2, 64, 1023, 1023, None, P, P, P, None) == -3   # shared memory too large
    assert Bd(P, None, 2, 16, 256, 256, None, P, P, P, None) == -1
    # EAGLE-2 selection
    E = L.tv_eagle_expand_select
    assert E(P, P, P, 0, 400, 1, 8, P, P, None) == 0
    assert E(P, P, P, 2, 4097, 1, 8, P, P, None) == -3
    assert E(P, P, P, 2, 400, 0, 8, P, P, None) == -3
    assert E(P, None, P, 2, 400, 1, 8, P, P, None) == -1
    R = L.tv_eagle_rerank
    assert R(P, P, P, P, 0, 400, 64, None, P, P, P, P, None) == 0
    assert R(P, P, P, P, 2, 400, 1024, None, P, P, P, P, None) == -3
    assert R(P, P, P, P, 2, 40, 64, None, P, P, P, P, None) == -3     # n_keep > max_cands
    assert R(P, P, None, P, 2, 400, 64, None, P, P, P, P, None) == -1
    # fused accept + commit
    AC = L.tv_accept_commit
    assert AC(ctypes.byref(g), P, P, P, P, P, 0, 41, 4, P, P, P, P, P, P, 8, P, P, 10, P, P, P, P,
              None) == 0
    assert AC(ctypes.byref(bad_d), P, P, P, P, P, 1, 41, 4, P, P, P, P, P, P, 8, P, P, 10, P, P, P,
              P, None) == -2
    assert AC(ctypes.byref(g), P, P, P, P, P, 1, 41, -1, P, P, P, P, P, P, 8, P, P, 10, P, P, P, P,
              None) == -3
    assert AC(ctypes.byref(g), P, None, P, P, P, 1, 41, 4, P, P, P, P, P, P, 8, P, P, 10, P, P, P,
              P, None) == -1
    # dense mask export
    M = L.tv_tree_mask_dense
    assert M(P, P, P, P, 0, 41, 0, 0, P, None) == 0
    assert M(P, P, P, P, 2, 41, 2, 0, P, None) == -3        # mode
    assert M(P, P, P, P, 2, 41, 0, 2, P, None) == -3        # dtype
    assert M(P, P, P, P, 2, 0, 0, 0, P, None) == -3
    assert M(P, P, P, None, 2, 41, 0, 0, P, None) == -1
    assert M(P, P, P, P, 2, 41, 0, 1, P + 2, None) == -5    # float32 out not aligned


def test_missing_library_fails_loudly(tmp_path):
    """No CPU fallback: without the built library the binding raises."""
    with pytest.raises(FileNotFoundError):
        tv.load(str(tmp_path / "libtreeverify.so"))
