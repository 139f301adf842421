"""Device buffers for one batch and the four library calls of a verification
step, in order (tree_build -> tree_attention_verify -> greedy_accept ->
kv_commit). torch only provides device memory and the stream."""

from __future__ import annotations

import numpy as np
import torch

from . import (accept_commit, geom as make_geom, greedy_accept, kv_commit, tree_attention_verify,
               tree_build, workspace_bytes)

_STEP_INPUTS = ("parents", "cu_nodes", "prompt_len", "draft_tokens", "target_ids")


def _arena(specs, dev):
    """One device buffer holding several tensors back to back (16-byte
    aligned): (buffer, {name: view}). specs: [(name, shape, dtype)]."""
    offs, off = {}, 0
    for name, shape, dtype in specs:
        nbytes = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
        offs[name] = (off, shape, dtype, nbytes)
        off += -(-nbytes // 16) * 16
    buf = torch.zeros(max(off, 16), dtype=torch.uint8, device=dev)
    views = {name: buf[o:o + n].view(dtype).view(shape) for name, (o, shape, dtype, n) in offs.items()}
    return buf, views


def _i32(a, dev):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(dev)


def _bf16(bits, dev):
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.to(dev).view(torch.bfloat16)


class DeviceBatch:
    """A workload dict (see gen/workloads.py) resident on a CUDA device, plus the
    output buffers and the attention workspace."""

    def __init__(self, w, device="cuda", workspace=None, share=None):
        """``share``: another DeviceBatch of the same batch whose KV pools,
        block table and workspace this one uses (the steps of a multi-step
        run keep their own inputs and outputs over one cache)."""
        dev = torch.device(device)
        self.w = w
        self.device = dev
        self.g = make_geom(w["num_q_heads"], w["num_kv_heads"], w["head_dim"], w["block_size"],
                           w["rope_base"], 0.0, w["rope_style"])
        self.max_nodes = int(w["max_nodes"])
        self.max_depth = int(w["max_depth"])
        self.batch = int(w["batch"])
        table = np.ascontiguousarray(w["block_table"], dtype=np.int32)
        if share is not None:
            self.k_cache, self.v_cache = share.k_cache, share.v_cache
            self.table_state = share.table_state
            workspace = share.workspace if workspace is None else workspace
        else:
            self.k_cache = _bf16(w["k_cache"], dev)
            self.v_cache = _bf16(w["v_cache"], dev)
            # block table and per-request block counts share one buffer, so an
            # allocator can save or restore both with one copy
            nblk = np.ascontiguousarray(w["n_blocks"], dtype=np.int32)
            self.table_state = _i32(np.concatenate([table.reshape(-1), nblk]), dev)
        self.block_table = self.table_state[:table.size].view(table.shape)
        self.n_blocks = self.table_state[table.size:]
        self.load_step_inputs(w)
        ws = workspace_bytes(self.g, self.batch, self.max_nodes)
        if workspace is None:
            workspace = torch.zeros(ws, dtype=torch.uint8, device=dev)
        self.workspace = workspace
        # the step's results live in one buffer too (one device-to-host copy)
        bsz, mb = self.batch, self.block_table.shape[1]
        self.outputs, views = _arena([
            ("status", (bsz,), torch.int32), ("accept_path", (bsz, self.max_depth + 1), torch.int32),
            ("accept_len", (bsz,), torch.int32), ("bonus", (bsz,), torch.int32),
            ("new_len", (bsz,), torch.int32), ("released", (bsz, mb), torch.int32),
            ("released_count", (bsz,), torch.int32)], dev)
        for name, t in views.items():
            setattr(self, name, t)

    def load_step_inputs(self, w):
        """(Re)load the per-step inputs (tree, tokens, fresh Q/K/V) and size
        the per-node outputs. The inputs share one device buffer, so a caller
        feeding them from the host needs one copy per step."""
        dev = self.device
        total = int(w["cu_nodes"][-1])
        hq, hkv, d = w["num_q_heads"], w["num_kv_heads"], w["head_dim"]
        specs = [("parents", (total,), torch.int32), ("cu_nodes", (self.batch + 1,), torch.int32),
                 ("prompt_len", (self.batch,), torch.int32), ("draft_tokens", (total,), torch.int32),
                 ("target_ids", (total,), torch.int32), ("q", (total, hq, d), torch.bfloat16),
                 ("k_new", (total, hkv, d), torch.bfloat16), ("v_new", (total, hkv, d), torch.bfloat16)]
        self.inputs, views = _arena(specs, dev)
        for name, t in views.items():
            setattr(self, name, t)
        for name in ("parents", "cu_nodes", "prompt_len", "draft_tokens", "target_ids"):
            getattr(self, name).copy_(_i32(w[name], dev))
        for name in ("q", "k_new", "v_new"):
            getattr(self, name).copy_(_bf16(w[name], dev).view(getattr(self, name).shape))
        total = int(w["cu_nodes"][-1])
        words = (self.max_nodes + 31) // 32
        self.mask = torch.zeros(total, words, dtype=torch.int32, device=dev)
        self.depth = torch.zeros(total, dtype=torch.int32, device=dev)
        self.positions = torch.zeros(total, dtype=torch.int32, device=dev)
        self.retrieve_index = torch.zeros(total, dtype=torch.int32, device=dev)
        self.next_token = torch.zeros(total, dtype=torch.int32, device=dev)
        self.next_sibling = torch.zeros(total, dtype=torch.int32, device=dev)
        self.out = torch.zeros(total, w["num_q_heads"], w["head_dim"], dtype=torch.bfloat16,
                               device=dev)

    # the four calls -----------------------------------------------------
    def tree_build(self, stream=None):
        tree_build(self.parents, self.cu_nodes, self.prompt_len, self.max_nodes, self.mask,
                   self.depth, self.positions, self.retrieve_index, self.next_token,
                   self.next_sibling, self.status, stream)

    def attention(self, stream=None):
        tree_attention_verify(self.g, self.max_nodes, self.q, self.k_new, self.v_new,
                              self.cu_nodes, self.positions, self.mask, self.prompt_len,
                              self.block_table, self.n_blocks, self.k_cache, self.v_cache,
                              self.out, self.workspace, self.status, stream)

    def accept(self, stream=None):
        greedy_accept(self.target_ids, self.draft_tokens, self.cu_nodes, self.next_token,
                      self.next_sibling, self.max_nodes, self.accept_path, self.accept_len,
                      self.bonus, self.status, stream)

    def commit(self, stream=None):
        kv_commit(self.g, self.accept_path, self.accept_len, self.prompt_len, self.block_table,
                  self.n_blocks, self.k_cache, self.v_cache, self.new_len, self.released,
                  self.released_count, self.status, stream)

    def accept_commit(self, stream=None):
        """accept + commit fused into one kernel (tv_accept_commit)."""
        accept_commit(self.g, self.target_ids, self.draft_tokens, self.cu_nodes, self.next_token,
                      self.next_sibling, self.max_nodes, self.accept_path, self.accept_len,
                      self.bonus, self.prompt_len, self.block_table, self.n_blocks, self.k_cache,
                      self.v_cache, self.new_len, self.released, self.released_count, self.status,
                      stream)

    def step(self, stream=None):
        self.tree_build(stream)
        self.attention(stream)
        self.accept(stream)
        self.commit(stream)

    # host views -----------------------------------------------------------
    def cache_bits(self):
        k = self.k_cache.view(torch.int16).cpu().numpy().view(np.uint16)
        v = self.v_cache.view(torch.int16).cpu().numpy().view(np.uint16)
        return k, v

    def out_f32(self):
        return self.out.float().cpu().numpy()
