"""Python binding of libtreeverify (GB300 token-tree verification).

The functions below carry the names of the C entry points declared in
``include/treeverify.h`` and only marshal arguments: torch tensors are checked
for device, dtype and contiguity and passed as raw device pointers together
with the current CUDA stream. Every step of the verification runs in the
library's CUDA kernels; there is no CPU fallback. If the shared library has
not been built, ``load()`` raises.
"""

from __future__ import annotations

import ctypes
import os

import torch

__all__ = [
    "TV_OK", "TV_ST", "TvGeom", "TvError", "load", "lib_path", "geom", "workspace_bytes",
    "tree_build", "tree_attention_verify", "tree_attention_verify_noalloc", "greedy_accept", "kv_commit",
    "accept_commit",
    "sample_tokens", "sampled_accept", "rejection_accept", "ddtree_nodes", "ddtree_topk", "ddtree_build",
    "eagle_expand_select", "eagle_rerank", "tree_mask_dense", "dense_mask_elements",
    "status_string", "version",
]

_PKG = os.path.dirname(os.path.abspath(__file__))
lib_path = os.path.join(_PKG, "libtreeverify.so")

TV_OK = 0
TV_ST = {"BAD_SIZE": 1, "BAD_ROOT": 2, "BAD_PARENT": 4, "BAD_BLOCK": 8,
         "PATH_OVERFLOW": 16, "TIMEOUT": 32, "BAD_TEMPERATURE": 64}


class TvGeom(ctypes.Structure):
    _fields_ = [("num_q_heads", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("block_size", ctypes.c_int32),
                ("rope_base", ctypes.c_float), ("softmax_scale", ctypes.c_float),
                ("rope_style", ctypes.c_int32)]


class TvError(RuntimeError):
    def __init__(self, fn, code):
        super().__init__(f"{fn} failed: {status_string(code)} ({code})")
        self.code = code


_lib = None
_P = ctypes.c_void_p
_I = ctypes.c_int32
_SZ = ctypes.c_size_t
_I64 = ctypes.c_int64
_SIGS = {
    "tv_workspace_bytes": [ctypes.POINTER(TvGeom), _I, _I, ctypes.POINTER(_SZ)],
    "tv_tree_build": [_P, _P, _P, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P],
    "tv_tree_attention_verify": [ctypes.POINTER(TvGeom), _I, _I, _P, _P, _P, _P, _P, _P, _P,
                                 _P, _P, _I, _P, _P, _I, _P, _P, _SZ, _P, _P],
    "tv_tree_attention_verify_noalloc": [ctypes.POINTER(TvGeom), _I, _I, _P, _P, _P, _P, _P,
                                         _P, _P, _P, _P, _I, _P, _P, _I, _P, _P, _P],
    "tv_greedy_accept": [_P, _P, _P, _P, _P, _I, _I, _I, _P, _P, _P, _P, _P],
    "tv_kv_commit": [ctypes.POINTER(TvGeom), _I, _P, _P, _I, _P, _P, _P, _I, _P, _P, _I, _P,
                     _P, _P, _P, _P],
    "tv_sample_tokens": [_P, _I64, _P, _I64, _P, _P, _I, _I, _I, _P, _P, _P],
    "tv_sampled_accept": [_P, _I64, _P, _I64, _P, _P, _P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _P],
    "tv_rejection_accept": [_P, _I64, _P, _I64, _P, _I64, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I,
                            _P, _P, _P, _P, _P],
    "tv_ddtree_nodes": [_I, _I, _I],
    "tv_ddtree_topk": [_P, _I64, _I, _I, _I, _P, _P, _P],
    "tv_ddtree_build": [_P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _P],
    "tv_eagle_expand_select": [_P, _P, _P, _I, _I, _I, _I, _P, _P, _P],
    "tv_eagle_rerank": [_P, _P, _P, _P, _I, _I, _I, _P, _P, _P, _P, _P, _P],
    "tv_tree_mask_dense": [_P, _P, _P, _P, _I, _I, _I, _I, _P, _P],
    "tv_accept_commit": [ctypes.POINTER(TvGeom), _P, _P, _P, _P, _P, _I, _I, _I, _P, _P, _P, _P,
                         _P, _P, _I, _P, _P, _I, _P, _P, _P, _P, _P],
    "tv_status_string": [ctypes.c_int],
    "tv_version": [],
}


def load(path: str | None = None):
    """Load libtreeverify.so (raises if it has not been built)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or lib_path
    if not os.path.exists(p):
        raise FileNotFoundError(
            f"{p} is missing: build it with `python -m speculative_decoding_tree_build_gb300.build` "
            "(or __graft_entry__.build()); there is no fallback implementation")
    lib = ctypes.CDLL(p)
    for name, args in _SIGS.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = ctypes.c_char_p if name == "tv_status_string" else ctypes.c_int
    if path is None:
        _lib = lib
    return lib


def status_string(code: int) -> str:
    return load().tv_status_string(int(code)).decode()


def version() -> int:
    return load().tv_version()


def geom(num_q_heads, num_kv_heads, head_dim, block_size=16, rope_base=10000.0,
         softmax_scale=0.0, rope_style=0) -> TvGeom:
    return TvGeom(num_q_heads, num_kv_heads, head_dim, block_size, rope_base, softmax_scale,
                  rope_style)


def _ptr(t, dtype=None, name="tensor"):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(fn, rc):
    if rc != TV_OK:
        raise TvError(fn, rc)
    return rc


I32, U32, BF16 = torch.int32, torch.uint32 if hasattr(torch, "uint32") else torch.int32, torch.bfloat16


def workspace_bytes(g: TvGeom, batch: int, max_nodes: int) -> int:
    out = _SZ(0)
    _check("tv_workspace_bytes", load().tv_workspace_bytes(ctypes.byref(g), batch, max_nodes,
                                                           ctypes.byref(out)))
    return out.value


def tree_build(parents, cu_nodes, prompt_len, max_nodes, mask_bits, depth, positions,
               retrieve_index, next_token, next_sibling, status, stream=None):
    batch = cu_nodes.numel() - 1
    return _check("tv_tree_build", load().tv_tree_build(
        _ptr(parents, I32, "parents"), _ptr(cu_nodes, I32, "cu_nodes"),
        _ptr(prompt_len, I32, "prompt_len"), batch, max_nodes, _ptr(mask_bits, None, "mask_bits"),
        _ptr(depth, I32), _ptr(positions, I32), _ptr(retrieve_index, I32), _ptr(next_token, I32),
        _ptr(next_sibling, I32), _ptr(status, I32, "status"), _stream(stream)))


def tree_attention_verify(g: TvGeom, max_nodes, q, k_new, v_new, cu_nodes, positions, mask_bits,
                          prompt_len, block_table, n_blocks, k_cache, v_cache, out, workspace,
                          status, stream=None):
    batch = cu_nodes.numel() - 1
    return _check("tv_tree_attention_verify", load().tv_tree_attention_verify(
        ctypes.byref(g), batch, max_nodes, _ptr(q, BF16, "q"), _ptr(k_new, BF16, "k_new"),
        _ptr(v_new, BF16, "v_new"), _ptr(cu_nodes, I32), _ptr(positions, I32),
        _ptr(mask_bits, None), _ptr(prompt_len, I32), _ptr(block_table, I32, "block_table"),
        _ptr(n_blocks, I32), block_table.shape[1], _ptr(k_cache, BF16, "k_cache"),
        _ptr(v_cache, BF16, "v_cache"), k_cache.shape[0], _ptr(out, BF16, "out"),
        _ptr(workspace, None, "workspace"), workspace.numel() * workspace.element_size(),
        _ptr(status, I32), _stream(stream)))


def tree_attention_verify_noalloc(g: TvGeom, max_nodes, q, k_new, v_new, cu_nodes, positions,
                                  mask_bits, prompt_len, block_table, n_blocks, k_cache, v_cache,
                                  out, status, stream=None):
    """tree_attention_verify without a workspace, for callers that cannot
    allocate device memory: scratch comes from a fixed-size array inside the
    library (see include/treeverify.h for its limits and sharing rules)."""
    batch = cu_nodes.numel() - 1
    return _check("tv_tree_attention_verify_noalloc", load().tv_tree_attention_verify_noalloc(
        ctypes.byref(g), batch, max_nodes, _ptr(q, BF16, "q"), _ptr(k_new, BF16, "k_new"),
        _ptr(v_new, BF16, "v_new"), _ptr(cu_nodes, I32), _ptr(positions, I32),
        _ptr(mask_bits, None), _ptr(prompt_len, I32), _ptr(block_table, I32, "block_table"),
        _ptr(n_blocks, I32), block_table.shape[1], _ptr(k_cache, BF16, "k_cache"),
        _ptr(v_cache, BF16, "v_cache"), k_cache.shape[0], _ptr(out, BF16, "out"),
        _ptr(status, I32), _stream(stream)))


def greedy_accept(target_ids, draft_tokens, cu_nodes, next_token, next_sibling, max_nodes,
                  accept_path, accept_len, bonus, status, stream=None):
    batch = cu_nodes.numel() - 1
    max_depth = accept_path.shape[1] - 1
    return _check("tv_greedy_accept", load().tv_greedy_accept(
        _ptr(target_ids, I32, "target_ids"), _ptr(draft_tokens, I32, "draft_tokens"),
        _ptr(cu_nodes, I32), _ptr(next_token, I32), _ptr(next_sibling, I32), batch, max_nodes,
        max_depth, _ptr(accept_path, I32), _ptr(accept_len, I32), _ptr(bonus, I32),
        _ptr(status, I32), _stream(stream)))


def kv_commit(g: TvGeom, accept_path, accept_len, prompt_len, block_table, n_blocks, k_cache,
              v_cache, new_len, released, released_count, status, stream=None):
    batch = accept_len.numel()
    return _check("tv_kv_commit", load().tv_kv_commit(
        ctypes.byref(g), batch, _ptr(accept_path, I32), _ptr(accept_len, I32),
        accept_path.shape[1] - 1, _ptr(prompt_len, I32), _ptr(block_table, I32),
        _ptr(n_blocks, I32), block_table.shape[1], _ptr(k_cache, BF16), _ptr(v_cache, BF16),
        k_cache.shape[0], _ptr(new_len, I32), _ptr(released, I32), _ptr(released_count, I32),
        _ptr(status, I32), _stream(stream)))


def _rows(t, name):
    """(pointer, row stride) of a float32 [rows][>= vocab] CUDA tensor whose
    rows are contiguous; None -> (None, 0)."""
    if t is None:
        return None, 0
    if not t.is_cuda or t.dtype != torch.float32 or t.dim() != 2 or t.stride(1) != 1:
        raise ValueError(f"{name} must be a float32 CUDA matrix with contiguous rows")
    return t.data_ptr(), t.stride(0)


def sample_tokens(logits, gumbel, cu_nodes, temperature, max_nodes, tokens, status, stream=None):
    """The target's token at every node: greedy (temperature 0) or a
    Gumbel-max draw. ``logits``/``gumbel`` are [T][vocab] views (row stride
    may exceed vocab); ``gumbel`` may be None when every temperature is 0."""
    batch = cu_nodes.numel() - 1
    lp, lld = _rows(logits, "logits")
    gp, gld = _rows(gumbel, "gumbel")
    return _check("tv_sample_tokens", load().tv_sample_tokens(
        lp, lld, gp, gld, _ptr(cu_nodes, I32, "cu_nodes"),
        _ptr(temperature, torch.float32, "temperature"), batch, max_nodes, logits.shape[1],
        _ptr(tokens, I32, "tokens"), _ptr(status, I32, "status"), _stream(stream)))


def sampled_accept(logits, gumbel, cu_nodes, temperature, parents, draft_tokens, max_nodes,
                   accept_path, accept_len, bonus, status, stream=None):
    """The verifier walk with the target sampling itself at the nodes it
    visits; same outputs as greedy_accept."""
    batch = cu_nodes.numel() - 1
    lp, lld = _rows(logits, "logits")
    gp, gld = _rows(gumbel, "gumbel")
    return _check("tv_sampled_accept", load().tv_sampled_accept(
        lp, lld, gp, gld, _ptr(cu_nodes, I32, "cu_nodes"),
        _ptr(temperature, torch.float32, "temperature"), _ptr(parents, I32, "parents"),
        _ptr(draft_tokens, I32, "draft_tokens"), batch, max_nodes, accept_path.shape[1] - 1,
        logits.shape[1], _ptr(accept_path, I32), _ptr(accept_len, I32), _ptr(bonus, I32),
        _ptr(status, I32), _stream(stream)))


def rejection_accept(logits, draft_logits, gumbel, uniforms, cu_nodes, temperature, parents,
                     draft_tokens, draft_logp, max_nodes, accept_path, accept_len, bonus, status,
                     stream=None):
    """Rejection-sampling verification along the chosen path (largest
    cumulative draft log-probability): the min(1, p/q) rule per edge, the
    correction drawn from the residual; same outputs as greedy_accept."""
    batch = cu_nodes.numel() - 1
    lp, lld = _rows(logits, "logits")
    dp, dld = _rows(draft_logits, "draft_logits")
    gp, gld = _rows(gumbel, "gumbel")
    return _check("tv_rejection_accept", load().tv_rejection_accept(
        lp, lld, dp, dld, gp, gld, _ptr(uniforms, torch.float32, "uniforms"),
        _ptr(cu_nodes, I32, "cu_nodes"), _ptr(temperature, torch.float32, "temperature"),
        _ptr(parents, I32, "parents"), _ptr(draft_tokens, I32, "draft_tokens"),
        _ptr(draft_logp, torch.float32, "draft_logp"), batch, max_nodes,
        accept_path.shape[1] - 1, logits.shape[1], _ptr(accept_path, I32), _ptr(accept_len, I32),
        _ptr(bonus, I32), _ptr(status, I32), _stream(stream)))


def ddtree_nodes(depth_L: int, k: int, budget: int) -> int:
    """Nodes (root included) of every tree tv_ddtree_build makes for these sizes."""
    n = load().tv_ddtree_nodes(depth_L, k, budget)
    if n < 0:
        raise TvError("tv_ddtree_nodes", n)
    return n


def ddtree_topk(logits, k, top_tokens, top_logq, stream=None):
    """Per row of ``logits`` ([rows][vocab] view with contiguous rows): the k
    most probable tokens (logit descending, token ascending) and their
    log-probabilities."""
    lp, lld = _rows(logits, "logits")
    return _check("tv_ddtree_topk", load().tv_ddtree_topk(
        lp, lld, logits.shape[0], logits.shape[1], k, _ptr(top_tokens, I32, "top_tokens"),
        _ptr(top_logq, torch.float32, "top_logq"), _stream(stream)))


def ddtree_build(top_logq, top_tokens, budget, parents, tokens, cu_nodes, root_tokens=None,
                 stream=None):
    """DDTree best-first construction from per-depth top-K log-probabilities
    ``top_logq`` / ``top_tokens`` of shape [batch][L][k]; writes the flattened
    trees (root first, depth by depth) and their node offsets."""
    batch, depth_l, k = top_logq.shape
    return _check("tv_ddtree_build", load().tv_ddtree_build(
        _ptr(top_logq, torch.float32, "top_logq"), _ptr(top_tokens, I32, "top_tokens"), batch,
        depth_l, k, budget, _ptr(root_tokens, I32, "root_tokens"), _ptr(parents, I32, "parents"),
        _ptr(tokens, I32, "tokens"), _ptr(cu_nodes, I32, "cu_nodes"), _stream(stream)))


def eagle_expand_select(logp, parent, cand_count, layer, k, selected, status, stream=None):
    """Top-k candidates of depth ``layer`` per request. ``logp``/``parent``
    are [batch][max_cands] (generation order), ``selected`` [batch][k]."""
    batch, max_cands = logp.shape
    return _check("tv_eagle_expand_select", load().tv_eagle_expand_select(
        _ptr(logp, torch.float32, "logp"), _ptr(parent, I32, "parent"),
        _ptr(cand_count, I32, "cand_count"), batch, max_cands, layer, k,
        _ptr(selected, I32, "selected"), _ptr(status, I32, "status"), _stream(stream)))


def eagle_rerank(logp, parent, token, cand_count, n_keep, parents, tokens, cu_nodes, status,
                 root_tokens=None, stream=None):
    """Global top-``n_keep`` candidates per request, packed breadth first."""
    batch, max_cands = logp.shape
    return _check("tv_eagle_rerank", load().tv_eagle_rerank(
        _ptr(logp, torch.float32, "logp"), _ptr(parent, I32, "parent"), _ptr(token, I32, "token"),
        _ptr(cand_count, I32, "cand_count"), batch, max_cands, n_keep,
        _ptr(root_tokens, I32, "root_tokens"), _ptr(parents, I32, "parents"),
        _ptr(tokens, I32, "tokens"), _ptr(cu_nodes, I32, "cu_nodes"), _ptr(status, I32, "status"),
        _stream(stream)))


MASK_FULL, MASK_QLEN_ONLY = 0, 1
MASK_BOOL, MASK_ADDITIVE_F32 = 0, 1


def dense_mask_elements(cu_nodes, prompt_len, mode=MASK_FULL) -> int:
    """Elements tv_tree_mask_dense writes (host arrays or tensors)."""
    import numpy as np
    cu = np.asarray(cu_nodes.cpu() if hasattr(cu_nodes, "cpu") else cu_nodes, np.int64)
    n = np.diff(cu)
    if mode == MASK_QLEN_ONLY:
        return int(np.sum(n * n))
    p = np.maximum(np.asarray(prompt_len.cpu() if hasattr(prompt_len, "cpu") else prompt_len,
                              np.int64), 0)
    return int(np.sum(n * (p + n)))


def tree_mask_dense(mask_bits, cu_nodes, prompt_len, status, max_nodes, out, mode=MASK_FULL,
                    dtype=MASK_BOOL, stream=None):
    """Dense [N, P+N] (or [N, N]) masks of all requests, back to back in
    ``out`` (uint8 for MASK_BOOL, float32 for MASK_ADDITIVE_F32)."""
    want = torch.uint8 if dtype == MASK_BOOL else torch.float32
    batch = cu_nodes.numel() - 1
    return _check("tv_tree_mask_dense", load().tv_tree_mask_dense(
        _ptr(mask_bits, None, "mask_bits"), _ptr(cu_nodes, I32, "cu_nodes"),
        _ptr(prompt_len, I32, "prompt_len"), _ptr(status, I32, "status"), batch, max_nodes,
        mode, dtype, _ptr(out, want, "out"), _stream(stream)))


def accept_commit(g: TvGeom, target_ids, draft_tokens, cu_nodes, next_token, next_sibling,
                  max_nodes, accept_path, accept_len, bonus, prompt_len, block_table, n_blocks,
                  k_cache, v_cache, new_len, released, released_count, status, stream=None):
    """greedy_accept followed by kv_commit in one kernel (same outputs)."""
    batch = cu_nodes.numel() - 1
    return _check("tv_accept_commit", load().tv_accept_commit(
        ctypes.byref(g), _ptr(target_ids, I32, "target_ids"), _ptr(draft_tokens, I32, "draft_tokens"),
        _ptr(cu_nodes, I32), _ptr(next_token, I32), _ptr(next_sibling, I32), batch, max_nodes,
        accept_path.shape[1] - 1, _ptr(accept_path, I32), _ptr(accept_len, I32), _ptr(bonus, I32),
        _ptr(prompt_len, I32), _ptr(block_table, I32), _ptr(n_blocks, I32), block_table.shape[1],
        _ptr(k_cache, BF16), _ptr(v_cache, BF16), k_cache.shape[0], _ptr(new_len, I32),
        _ptr(released, I32), _ptr(released_count, I32), _ptr(status, I32), _stream(stream)))
