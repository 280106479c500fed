"""Oracle: rotary position embedding applied before the KV write, in float64.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

Sources: visual atlas (diomchen.github.io/reference/visual-atlas.html),
fig. 19: RoPE rotates one two-dimensional pair of a head by an angle that grows
with the position (the figure shows a single frequency; a real head has d/2
pairs with d/2 different frequencies), and the engine's order rotates Q and K
but not V.

Readings where the pages are silent (the CUDA path follows the same ones):

* pair i of a head couples dimensions i and i + d/2 (the "rotate half" layout
  of the Qwen3 attention the pages describe), for i < d/2;
* pair i turns by angle pos * base^(-2i/d); ``base`` is a parameter
  (Qwen3-0.6B's model configuration uses 1,000,000);
* the rotation is counter-clockwise: (a, b) -> (a cos t - b sin t, b cos t + a sin t).
"""
from __future__ import annotations

import numpy as np


def rotate_pair(a, b, angle):
    """The atlas fig. 19 picture: the 2-D pair (a, b) turned counter-clockwise
    by ``angle`` radians.  Works elementwise on arrays of pairs."""
    c, s = np.cos(angle), np.sin(angle)
    return a * c - b * s, b * c + a * s


def rope(x, positions, base: float) -> np.ndarray:
    """x: [N, H, d]; positions: [N].  Returns the rotated copy in float64.

    Angle of pair i at position p: p * base^(-2i/d); the rotation is
    ``rotate_pair`` applied to (x[..., i], x[..., i + d/2]) for every token and
    head at once."""
    x = np.asarray(x, dtype=np.float64)
    d = x.shape[-1]
    half = d // 2
    inv_freq = np.array([base ** (-2.0 * i / d) for i in range(half)])
    angle = np.asarray(positions, dtype=np.float64)[:, None] * inv_freq[None, :]   # [N, d/2]
    a_rot, b_rot = rotate_pair(x[..., :half], x[..., half:], angle[:, None, :])
    return np.concatenate([a_rot, b_rot], axis=-1)


def rope_store_kvcache(q, k_cache, v_cache, k, v, positions, slots, block_size: int, base: float):
    """Rotate q and k by their positions, then scatter (rotated k, unrotated v) into the pools.

    Returns (rotated q, new k pool, new v pool); a negative slot skips the write."""
    from .paged_attention import store_kvcache
    q_rot = rope(q, positions, base) if q is not None else None
    k_rot = rope(k, positions, base)
    kc, vc = store_kvcache(k_cache, v_cache, k_rot, np.asarray(v, dtype=np.float64), slots, block_size)
    return q_rot, kc, vc
