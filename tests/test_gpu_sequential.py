"""Tree verification against token-by-token decoding.

"投机解码的树状注意力验证…" advises checking a tree verifier by sampling and
comparing it with plain token-by-token decoding. After one verification step
(tree build, tree attention, greedy accept, KV commit) the accepted tokens are
decoded again one at a time, each as a one-node tree on the prompt extended by
the tokens before it, starting from the pre-step cache:

- the attention output of each accepted node must match the output of its
  one-token decode (same keys, same positions; only the summation order of
  the split key ranges differs), within the attention tolerance;
- the committed cache rows must equal the rows the one-token decodes write,
  bit for bit: a node at depth k is rotated at position P + k in both, and
  the commit moves its bytes unchanged.
"""

import numpy as np
import pytest
import torch

from gen import workloads as wl
from speculative_decoding_tree_build_gb300.build import build
from speculative_decoding_tree_build_gb300.step import DeviceBatch

from parity import ATOL, REL_FRO

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build()
    assert torch.cuda.is_available()


def _one_node_batch(w, node):
    """A one-request, one-node workload over w's pre-step cache and block
    table, whose node carries the raw q / k / v of `node` of w's request 0."""
    w1 = dict(w)
    w1.update(batch=1, max_nodes=1, max_depth=0,
              parents=np.array([-1], np.int32), cu_nodes=np.array([0, 1], np.int32),
              prompt_len=np.array(w["prompt_len"][:1], np.int32),
              draft_tokens=np.array(w["draft_tokens"][node:node + 1], np.int32),
              target_ids=np.array(w["target_ids"][node:node + 1], np.int32),
              q=np.array(w["q"][node:node + 1]), k_new=np.array(w["k_new"][node:node + 1]),
              v_new=np.array(w["v_new"][node:node + 1]))
    return w1


@pytest.mark.parametrize("geom,plen", [(wl.GEOM_8B, 1003), (wl.Geometry(4, 2, 64, rope_style=1), 37),
                                       (wl.Geometry(8, 2, 128), 16)])
def test_tree_step_equals_token_by_token_decoding(geom, plen):
    rng = np.random.default_rng(plen)
    tree = wl.medusa_tree(rng, (4, 3, 2), 1000)
    w = wl.assemble(rng, geom, [plen], [tuple(np.asarray(a, np.int32) for a in tree)], 1000, 1.0)

    # the verification step
    db = DeviceBatch(w)
    db.step()
    torch.cuda.synchronize()
    assert int(db.status.abs().sum()) == 0
    a = int(db.accept_len[0])
    path = db.accept_path[0].cpu().numpy()[:a + 1]
    assert a == 3                          # every node with children matches: a root-to-leaf path
    out_tree = db.out_f32()
    k_tree, v_tree = db.cache_bits()
    table = w["block_table"][0]

    # the same tokens decoded one at a time on the pre-step cache
    seq = DeviceBatch(_one_node_batch(w, int(path[0])))
    for k in range(a + 1):
        node = int(path[k])
        seq.prompt_len.fill_(plen + k)
        seq.q.copy_(db.q[node:node + 1])
        seq.k_new.copy_(db.k_new[node:node + 1])
        seq.v_new.copy_(db.v_new[node:node + 1])
        seq.tree_build()
        seq.attention()
        torch.cuda.synchronize()
        assert int(seq.status.abs().sum()) == 0
        assert int(seq.positions[0]) == plen + k
        got = seq.out_f32()[0].astype(np.float64)
        want = out_tree[node].astype(np.float64)
        assert np.max(np.abs(got - want)) <= ATOL
        assert np.linalg.norm(got - want) <= REL_FRO * np.linalg.norm(want)
    k_seq, v_seq = seq.cache_bits()

    # committed rows: bit for bit; the prompt rows untouched by both
    for slot in range(plen + a + 1):
        blk, row = int(table[slot // 16]), slot % 16
        assert np.array_equal(k_tree[blk, :, row, :], k_seq[blk, :, row, :]), slot
        assert np.array_equal(v_tree[blk, :, row, :], v_seq[blk, :, row, :]), slot
    for slot in range(plen):
        blk, row = int(table[slot // 16]), slot % 16
        assert np.array_equal(k_seq[blk, :, row, :], w["k_cache"][blk, :, row, :]), slot
