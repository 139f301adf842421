"""Sampling-acceptance oracle (test infrastructure only).

Definitions followed:
  * "解码：采样、束搜索和推测性解码", section "高效离散采样", subsection
    "Gumbel Max技巧": drawing from Categorical(softmax(h)) is the same as taking
    argmax_i (h_i + g_i) with g_i = -log(-log(z_i)), z_i ~ Uniform(0, 1); the
    noise can be prepared ahead of time, so sampling is an add and an argmax.
  * "Accelerating Speculative Decoding with Block Diffusion Draft Trees",
    §7.2 (verifier walk: from the root, at every node the target picks a token
    with its own decoding rule, greedy or temperature sampling; if the token is
    a child of the current node the walk moves there, otherwise it stops and
    the token is the next bonus; no further target forward is needed since
    every node's logits come from the one forward) and §7.3 (this walk is
    lossless: its output follows the target's own autoregressive sampling).
  * "02 · Token Tree 与 Tree Attention" §4 (the greedy rule compares token ids).

Readings where the pages leave a step open:
  * temperature T divides the logits; T == 0 means greedy (argmax of the raw
    logits);
  * the noise g is an input, one float32 value per (node, vocabulary entry),
    as in the page's precomputed sampler;
  * x_v = h_v * (1/T) + g_v is evaluated in float32, the product rounded before
    the sum, and 1/T is the float32 quotient; ties in the argmax go to the
    smallest index. The CUDA kernel takes the same decision in the same
    precision, so the sampled ids are compared bit for bit.
"""

import numpy as np

from .accept_ref import greedy_accept_ref


def sample_tokens_ref(logits, gumbel, temperature):
    """Per-node token picked by the target's decoding rule.

    logits: float32 [nodes][V]; gumbel: float32 [nodes][V] (ignored when
    temperature == 0); returns int32 [nodes].
    """
    h = np.asarray(logits, dtype=np.float32)
    if temperature == 0:
        return np.argmax(h, axis=-1).astype(np.int32)          # first maximum
    inv = np.float32(1.0) / np.float32(temperature)
    scaled = np.multiply(h, inv, dtype=np.float32)              # rounded product
    x = np.add(scaled, np.asarray(gumbel, dtype=np.float32), dtype=np.float32)
    return np.argmax(x, axis=-1).astype(np.int32)


def sampled_walk_ref(parents, draft_tokens, logits, gumbel, temperature, max_depth):
    """The verifier walk of one request with the target sampling itself.

    Returns (status, path, bonus) as greedy_accept_ref does, with the per-node
    target choices drawn by sample_tokens_ref.
    """
    choices = sample_tokens_ref(logits, gumbel, temperature)
    return greedy_accept_ref(parents, draft_tokens, choices, max_depth)
