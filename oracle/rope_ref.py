"""Rotary position embedding at tree depth (oracle, test infrastructure only).

Follows the ``rope`` / ``rotate_half`` helpers of the runnable packed-vs-branch
experiment on "Beam Search、约束解码与 Tree/Self Speculation": for pair index
i in [0, D/2) the rotation angle is position * base**(-2i/D) and the pair
(x[2i], x[2i+1]) is rotated as a complex number, base 10000. The position of a
tree node is prompt length + depth ("02 · Token Tree 与 Tree Attention", §3;
section "Packed tree attention" of the glossary page: siblings share a
position, the packed index must not be used).

Readings where the pages are silent (the CUDA path follows the same reading):
  * inv_freq[i] = base**(-2i/D) evaluated exactly and rounded to float32;
  * the angle is the float32 product position * inv_freq[i] (rounded to
    nearest), because a float32 angle is what a float32 implementation feeds to
    sin/cos - at positions ~3e4 the angle's rounding (~4e-3 rad) is larger than
    bf16 resolution, so the angle's precision must be fixed, not left open;
  * cos/sin of that float32 angle and the rotation itself are exact (float64
    here); the rotated value is then rounded once to bf16 (the tensor-core
    operand type).
  * style 0 pairs (2i, 2i+1) as on the page; style 1 pairs (i, i + D/2)
    (the half-split convention many checkpoints use), offered as a variant.
"""

import numpy as np

from .bf16_ref import round_to_bf16


def rope_inv_freq_f32(head_dim, base):
    """float32 inverse frequencies base**(-2i/D), i = 0 .. D/2-1."""
    i = np.arange(head_dim // 2, dtype=np.float64)
    return (float(base) ** (-2.0 * i / head_dim)).astype(np.float32)


def rope_angles_f32(positions, head_dim, base):
    """float32 angles position * inv_freq (one rounding), shape [N, D/2]."""
    inv = rope_inv_freq_f32(head_dim, base).astype(np.float64)
    pos = np.asarray(positions, dtype=np.float64)
    # pos < 2**24 and inv has 24 significant bits, so the float64 product is
    # exact and its conversion to float32 is the correctly rounded product.
    return (pos[:, None] * inv[None, :]).astype(np.float32)


def rope_ref(x, positions, base=10000.0, style=0, round_bf16=True):
    """Rotate x [N, H, D] (float64 values) at per-row positions [N].

    Returns float64; rounded to bf16 values when ``round_bf16``.
    """
    x = np.asarray(x, dtype=np.float64)
    n, h, d = x.shape
    theta = rope_angles_f32(positions, d, base).astype(np.float64)   # [N, D/2]
    c = np.cos(theta)[:, None, :]
    s = np.sin(theta)[:, None, :]
    out = np.empty_like(x)
    if style == 0:
        a, b = x[..., 0::2], x[..., 1::2]
        out[..., 0::2] = a * c - b * s
        out[..., 1::2] = b * c + a * s
    elif style == 1:
        a, b = x[..., : d // 2], x[..., d // 2:]
        out[..., : d // 2] = a * c - b * s
        out[..., d // 2:] = b * c + a * s
    else:
        raise ValueError("rope style must be 0 (interleaved) or 1 (half split)")
    return round_to_bf16(out) if round_bf16 else out
