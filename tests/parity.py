"""Helpers for the GPU parity tests: run the library on a workload and compare
with the oracle on the same seeded inputs."""

from __future__ import annotations

import numpy as np
import torch

from oracle import bf16_bits_to_f64, verify_step_ref
from speculative_decoding_tree_build_gb300.step import DeviceBatch

ATOL = 2e-2          # max-abs error bound for bf16-input, fp32-accumulate attention
REL_FRO = 5e-3       # relative Frobenius error bound


def sample_pairs(w, per_request, seed=0):
    """(node, q_head) samples per request: the root, the deepest node, the
    last node and random ones."""
    rng = np.random.default_rng(seed)
    cu = w["cu_nodes"]
    hq = w["num_q_heads"]
    out = {}
    for b in range(w["batch"]):
        n = int(cu[b + 1] - cu[b])
        nodes = {0, n - 1} | set(rng.integers(0, n, size=per_request).tolist())
        pairs = set()
        for i in nodes:
            pairs.add((int(i), int(rng.integers(0, hq))))
            pairs.add((int(i), hq - 1))
        out[b] = sorted(pairs)
    return out


COST_TWO, COST_ONE, COST_UNIT = 10, 7, 21   # the kernel's step and unit costs


def attention_plan(w, grid, tile_keys=128):
    """The attention kernel's work plan, restated on the host.

    A unit is one request, one KV head and up to 8 * (32 // G) consecutive
    nodes (one or two M tiles of 32 // G nodes per 32-row quarter); it spans
    ceil((P + N) / tile_keys) key tiles. Units are ordered by request, KV
    head, node range, giving one global tile sequence. In cost units a unit is
    [COST_UNIT + c | c | c ...], c = COST_TWO or COST_ONE per tile by its M
    tiles; tile k starts at 0 (k = 0) or COST_UNIT + k c, and CTA j owns the
    tiles whose start lies in [floor(j W / grid), floor((j + 1) W / grid)).
    Returns (units, starts): units as (request, kv head, first node, end node,
    first global tile, end global tile, tile cost); starts[j] the first global
    tile of CTA j (starts[grid] = total tiles)."""
    hq, hkv = w["num_q_heads"], w["num_kv_heads"]
    g = hq // hkv
    npq = 32 // g
    unit_nodes = 8 * npq
    cu = w["cu_nodes"]
    units, tile_pos = [], []          # tile_pos: cost position of every tile
    t = pos = 0
    for b in range(w["batch"]):
        n = int(cu[b + 1] - cu[b])
        tiles = -(-(int(w["prompt_len"][b]) + n) // tile_keys)
        for kvh in range(hkv):
            for rg in range(-(-n // unit_nodes)):
                i0, i1 = rg * unit_nodes, min(n, (rg + 1) * unit_nodes)
                c = COST_TWO if -(-(i1 - i0) // (4 * npq)) == 2 else COST_ONE
                units.append((b, kvh, i0, i1, t, t + tiles, c))
                tile_pos.extend([pos] + [pos + COST_UNIT + k * c for k in range(1, tiles)])
                t += tiles
                pos += COST_UNIT + tiles * c
    bounds = [j * pos // grid for j in range(grid)] + [None]
    tile_pos = np.asarray(tile_pos, dtype=np.int64)
    starts = [int(np.searchsorted(tile_pos, bnd, side="left")) if bnd is not None else t for bnd in bounds]
    return units, starts


def split_unit_pairs(w, grid, tile_keys=128):
    """(node, q_head) pairs of every attention work unit whose key tiles the
    kernel divides between CTAs (``attention_plan``): a unit is split when a
    CTA's first tile lies strictly inside it; its partial results then go
    through the merge. Returns (pairs per request, number of split units)."""
    hq, hkv = w["num_q_heads"], w["num_kv_heads"]
    g = hq // hkv
    units, starts = attention_plan(w, grid, tile_keys)
    inner = np.asarray(starts[1:-1], dtype=np.int64)
    out, n_split = {}, 0
    for (b, kvh, i0, i1, u0, u1, _) in units:
        if not np.any((inner > u0) & (inner < u1)):
            continue
        n_split += 1
        pairs = out.setdefault(b, set())
        for i in range(i0, i1):
            for h in range(kvh * g, (kvh + 1) * g):
                pairs.add((i, h))
    return {b: sorted(v) for b, v in out.items()}, n_split


def compare_out(gpu_out, ref_out, w, pairs=None):
    """Element-wise attention comparison on all (or the sampled) outputs."""
    cu = w["cu_nodes"]
    g_list, r_list = [], []
    for b in range(w["batch"]):
        t0 = int(cu[b])
        if pairs is None:
            n = int(cu[b + 1] - cu[b])
            g_list.append(gpu_out[t0:t0 + n].reshape(-1))
            r_list.append(ref_out[t0:t0 + n].reshape(-1))
        else:
            for (i, h) in pairs.get(b, []):
                g_list.append(gpu_out[t0 + i, h])
                r_list.append(ref_out[t0 + i, h])
    g = np.concatenate(g_list).astype(np.float64)
    r = np.concatenate(r_list)
    assert np.all(np.isfinite(r)) and np.all(np.isfinite(g))
    max_abs = float(np.max(np.abs(g - r)))
    rel = float(np.linalg.norm(g - r) / max(np.linalg.norm(r), 1e-30))
    assert max_abs <= ATOL, f"max abs error {max_abs:.3e} > {ATOL}"
    assert rel <= REL_FRO, f"relative Frobenius error {rel:.3e} > {REL_FRO}"
    return max_abs, rel


def bf16_ulp_diff(a_bits, b_bits):
    """Distance in bf16 units in the last place between two bit arrays."""
    def ordered(x):
        x = x.astype(np.int32)
        return np.where(x & 0x8000, 0x8000 - (x & 0x7FFF), x + 0x8000)
    return np.abs(ordered(a_bits) - ordered(b_bits))


def rope_close(gpu_bits, x_raw, positions, w):
    """Rotated keys from the GPU against the exact rotation of the same raw
    keys. The GPU rotates in float32 then rounds to bf16, so each value may
    differ from the exact one by one bf16 ulp plus the float32 rotation's
    absolute error (a few 2**-24 * (|a| + |b|) for the pair (a, b); large
    relative to the value when a*cos - b*sin nearly cancels)."""
    from oracle import rope_ref
    exact = rope_ref(x_raw, positions, w["rope_base"], w["rope_style"], round_bf16=False)
    d = x_raw.shape[-1]
    if w["rope_style"] == 0:
        pair = np.abs(x_raw[..., 0::2]) + np.abs(x_raw[..., 1::2])
        pair = np.repeat(pair, 2, axis=-1)
    else:
        half = np.abs(x_raw[..., : d // 2]) + np.abs(x_raw[..., d // 2:])
        pair = np.concatenate([half, half], axis=-1)
    got = bf16_bits_to_f64(gpu_bits)
    _, e = np.frexp(exact)
    ulp = np.ldexp(1.0, np.maximum(e - 8, -133))
    err = np.abs(got - exact)
    tol = ulp + 2.0 ** -20 * pair
    bad = err > tol
    if np.any(bad):
        i = int(np.argmax(err - tol))
        raise AssertionError(
            f"rotated key off: got {got.ravel()[i]!r} exact {exact.ravel()[i]!r} "
            f"pair |a|+|b| {pair.ravel()[i]!r} ({int(bad.sum())} of {bad.size})")
    return float(np.max(err))


def tentative_rows(pool_bits, w, b, n, block_table=None):
    """Rows of slots [P_b, P_b + n) of request b: [n, Hkv, D]."""
    bs = w["block_size"]
    table = w["block_table"] if block_table is None else block_table
    plen = int(w["prompt_len"][b])
    slots = np.arange(plen, plen + n)
    return pool_bits[table[b][slots // bs].astype(np.int64), :, slots % bs, :]


def run_gpu(w, calls=("build", "attn", "accept", "commit"), db=None):
    db = db or DeviceBatch(w)
    for c in calls:
        {"build": db.tree_build, "attn": db.attention, "accept": db.accept,
         "commit": db.commit, "accept_commit": db.accept_commit}[c]()
    torch.cuda.synchronize()
    return db


def check_tree_outputs(db, ref, w):
    cu = w["cu_nodes"]
    st = db.status.cpu().numpy()
    assert not np.any(st & 32), "a bounded device wait expired (TV_ST_TIMEOUT)"
    assert np.array_equal(st & 7, ref["status"] & 7)
    for b in range(w["batch"]):
        if ref["status"][b] & 7:
            continue
        t0, t1 = int(cu[b]), int(cu[b + 1])
        for k in ("depth", "positions", "retrieve_index", "next_token", "next_sibling"):
            got = getattr(db, k)[t0:t1].cpu().numpy()
            assert np.array_equal(got, ref[k][t0:t1]), k
        got = db.mask[t0:t1].cpu().numpy().view(np.uint32)
        assert np.array_equal(got, ref["mask"][t0:t1])


def check_accept_outputs(db, ref, w):
    st = db.status.cpu().numpy()
    paths = db.accept_path.cpu().numpy()
    lens = db.accept_len.cpu().numpy()
    bonus = db.bonus.cpu().numpy()
    for b in range(w["batch"]):
        if ref["paths"][b] is None:
            continue
        path = ref["paths"][b]
        assert st[b] == 0
        assert lens[b] == len(path) - 1 and bonus[b] == ref["bonus"][b]
        want = np.full(paths.shape[1], -1)
        want[:len(path)] = path
        assert np.array_equal(paths[b], want)


def oracle_step(w, sample=None, commit=True):
    return verify_step_ref(w, sample=sample, commit=commit)


__all__ = ["ATOL", "REL_FRO", "sample_pairs", "split_unit_pairs", "attention_plan", "compare_out", "bf16_ulp_diff", "tentative_rows",
           "run_gpu", "rope_close", "check_tree_outputs", "check_accept_outputs", "oracle_step",
           "bf16_bits_to_f64"]
