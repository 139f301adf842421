"""Host checks of the attention kernel's cost-weighted work plan: the
closed-form CTA boundaries (first tile of a CTA, CTA of a tile), written here
as the kernel computes them, against a brute-force walk over every tile's
cost position (``parity.attention_plan``)."""

import numpy as np
import pytest

from gen import workloads as wl
from parity import COST_ONE, COST_TWO, COST_UNIT, attention_plan


def _shape(w, b, tile_keys=128):
    g = w["num_q_heads"] // w["num_kv_heads"]
    npq = 32 // g
    n = int(w["cu_nodes"][b + 1] - w["cu_nodes"][b])
    nrg = -(-n // (8 * npq))
    tiles = -(-(int(w["prompt_len"][b]) + n) // tile_keys)
    return n, npq, nrg, tiles


def _rg_cost(n, npq, rg):
    nodes = min(8 * npq, n - rg * 8 * npq)
    return COST_TWO if -(-nodes // (4 * npq)) == 2 else COST_ONE


def _unit_cost(n, npq, rg, tiles):
    return COST_UNIT + tiles * _rg_cost(n, npq, rg)


def _head_cost(n, npq, nrg, tiles):
    return (nrg - 1) * _unit_cost(n, npq, 0, tiles) + _unit_cost(n, npq, nrg - 1, tiles)


def _prefixes(w):
    hkv = w["num_kv_heads"]
    s_pre, sw_pre = [0], [0]
    for b in range(w["batch"]):
        n, npq, nrg, tiles = _shape(w, b)
        s_pre.append(s_pre[-1] + hkv * nrg * tiles)
        sw_pre.append(sw_pre[-1] + hkv * _head_cost(n, npq, nrg, tiles))
    return s_pre, sw_pre


def _find(pre, batch, x):
    lo, hi = 0, batch - 1
    while lo < hi:
        mid = (lo + hi + 1) >> 1
        if pre[mid] <= x:
            lo = mid
        else:
            hi = mid - 1
    return lo


def _cta_start(w, s_pre, sw_pre, grid, c):
    total_w = sw_pre[-1]
    if c >= grid or total_w == 0:
        return s_pre[-1]
    x = total_w * c // grid
    b = _find(sw_pre, w["batch"], x)
    n, npq, nrg, tiles = _shape(w, b)
    wk = _head_cost(n, npq, nrg, tiles)
    local = x - sw_pre[b]
    kvh, rem = local // wk, local % wk
    rg = 0
    while rg < nrg - 1:
        wu = _unit_cost(n, npq, rg, tiles)
        if rem < wu:
            break
        rem -= wu
        rg += 1
    c_t = _rg_cost(n, npq, rg)
    k = 0 if rem <= 0 else max(1, (rem - COST_UNIT + c_t - 1) // c_t)
    return s_pre[b] + (kvh * nrg + rg) * tiles + k


def _cta_of(w, s_pre, sw_pre, grid, t):
    total_w = sw_pre[-1]
    b = _find(s_pre, w["batch"], t)
    n, npq, nrg, tiles = _shape(w, b)
    local = t - s_pre[b]
    unit, k = local // tiles, local % tiles
    kvh, rg = unit // nrg, unit % nrg
    pos = (sw_pre[b] + kvh * _head_cost(n, npq, nrg, tiles) + rg * _unit_cost(n, npq, 0, tiles)
           + (0 if k == 0 else COST_UNIT + k * _rg_cost(n, npq, rg)))
    return min(grid - 1, ((pos + 1) * grid - 1) // total_w)


def _workloads():
    out = [(f"config{c}", wl.make_config(c)) for c in (1, 2, 3, 4, 5)]
    out.append(("config5_small", wl.make_config(5, batch=6, prompt_scale=0.03)))
    out.append(("config4_small", wl.make_config(4, batch=1, prompt_scale=0.05)))
    return out


@pytest.mark.parametrize("grid", [1, 7, 152])
@pytest.mark.parametrize("name,w", _workloads(), ids=lambda v: v if isinstance(v, str) else "")
def test_closed_form_plan_matches_brute_force(name, w, grid):
    units, starts = attention_plan(w, grid)
    s_pre, sw_pre = _prefixes(w)
    got = [_cta_start(w, s_pre, sw_pre, grid, c) for c in range(grid + 1)]
    assert got == starts
    assert got[0] == 0 and got[-1] == s_pre[-1]
    assert all(a <= b for a, b in zip(got, got[1:]))
    # every tile lies in exactly the CTA the closed form names
    owner = np.searchsorted(np.asarray(got[1:]), np.arange(s_pre[-1]), side="right")
    for t in range(0, s_pre[-1], max(1, s_pre[-1] // 4000)):
        assert _cta_of(w, s_pre, sw_pre, grid, t) == owner[t]
    # the last tile of every unit (the merge's last contributor)
    for u in units:
        assert _cta_of(w, s_pre, sw_pre, grid, u[5] - 1) == owner[u[5] - 1]


def test_cost_balance_on_the_large_workloads():
    """Estimated cost per CTA within 5 % of the mean on configs 3-5."""
    for c in (3, 4, 5):
        w = wl.make_config(c)
        units, starts = attention_plan(w, 152)
        cost = np.zeros(152)
        for (_, _, _, _, u0, u1, ct) in units:
            for j in range(152):
                lo, hi = max(u0, starts[j]), min(u1, starts[j + 1])
                if lo < hi:
                    cost[j] += (hi - lo) * ct + (COST_UNIT if lo == u0 else 0)
        assert cost.max() <= 1.05 * cost.mean()
