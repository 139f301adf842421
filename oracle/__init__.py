"""CPU oracle for the token-tree verification step (TEST INFRASTRUCTURE ONLY).

This package is a plain, slow, obviously correct CPU restatement of what the
verification step computes. It exists so that the CUDA path can be checked
against an independent implementation. Only the test-suite, the smoke check in
``__graft_entry__`` and the CPU-baseline leg of ``bench.py`` may import it; the
library itself never calls it and has no CPU fallback.

It shares no code with the CUDA path (no kernels, headers, helpers, constants or
tables) and never imports the ``speculative_decoding_tree_build_gb300``
package. Floating-point work is done in float64 (the packed-vs-branch
experiment on the Tree/Self-Speculation glossary page also runs in float64).

Sources (web pages, cited by title and section in each function):
  * "Beam Search、约束解码与 Tree/Self Speculation" (decoding-extensions
    glossary) - packed-node table, the runnable packed-vs-branch attention
    experiment and the runnable three-part semantics experiment;
  * "02 · Token Tree 与 Tree Attention" - token-tree definition, mask rules,
    depth positions, verify flow and KV rollback;
  * "投机解码的树状注意力验证：一次前向如何并行校验多条候选路径" - mask
    correctness rule and tree KV layout / page reclamation;
  * "Accelerating Speculative Decoding with Block Diffusion Draft Trees"
    (DDTree notes) - flattened tree, position ids and verifier walk (§6, §7);
  * "解码：采样、束搜索和推测性解码" - the Gumbel-max sampling trick.

Pinning: every function here is pinned by ``tests/test_oracle_pins.py`` to facts
that do not come from the oracle itself (printed example values, brute force,
closed forms, textbook special cases). No function is parity-unpinned.
"""

from .bf16_ref import bf16_bits_to_f64, f64_to_bf16_bits, round_to_bf16
from .tree_ref import (
    ST_OK, ST_BAD_SIZE, ST_BAD_ROOT, ST_BAD_PARENT, ST_BAD_BLOCK,
    ST_PATH_OVERFLOW, ancestor_path, tree_build_ref,
)
from .rope_ref import rope_inv_freq_f32, rope_ref
from .attention_ref import (
    branch_attention_ref, packed_attention_ref, dense_tree_mask_ref,
    gather_prompt_kv_ref, tree_attention_verify_ref,
)
from .accept_ref import greedy_accept_ref, verify_branches_ref
from .commit_ref import kv_commit_ref
from .step_ref import verify_step_ref
from .sample_ref import sample_tokens_ref, sampled_walk_ref
from .ddtree_ref import ddtree_build_ref, ddtree_from_logits_ref, topk_logprobs_ref
from .eagle_ref import eagle_expand_select_ref, eagle_rerank_ref, eagle_scores_ref
from .rejection_ref import chosen_path_ref, rejection_walk_ref

__all__ = [
    "bf16_bits_to_f64", "f64_to_bf16_bits", "round_to_bf16",
    "ST_OK", "ST_BAD_SIZE", "ST_BAD_ROOT", "ST_BAD_PARENT", "ST_BAD_BLOCK",
    "ST_PATH_OVERFLOW", "ancestor_path", "tree_build_ref",
    "rope_inv_freq_f32", "rope_ref",
    "branch_attention_ref", "packed_attention_ref", "dense_tree_mask_ref",
    "gather_prompt_kv_ref", "tree_attention_verify_ref",
    "greedy_accept_ref", "verify_branches_ref", "kv_commit_ref",
    "verify_step_ref", "sample_tokens_ref", "sampled_walk_ref",
    "topk_logprobs_ref", "ddtree_build_ref", "ddtree_from_logits_ref",
    "eagle_scores_ref", "eagle_expand_select_ref", "eagle_rerank_ref",
    "chosen_path_ref", "rejection_walk_ref",
]
