"""Rotary position embedding by table lookup, and its fusion with the cache
scatter, in float64.  TEST INFRASTRUCTURE ONLY (see the package header).

Source: "AI Infra入门干货总结：大模型是如何高效推理的", section "Attention Module
(以标准GQA + RoPE为例)".  The page states:
* after the QKV split, Q and K are rotated by RoPE, and then reshape_and_cache
  scatters K and V into the paged cache by slot_mapping;
* the rotation is a block-diagonal rotation matrix, applied element-wise with
  sin/cos instead of as a matrix product;
* sin/cos are not evaluated at run time: a table cos_sin_cache of shape
  [max_position_embeddings, rotary_dim] is built once, and the kernel picks the
  row of each token's position and does element-wise multiply-adds with it.

Readings where the page is silent (each one is a parameter or a stated
convention here):
* Row layout: row p holds rotary_dim / 2 cosines followed by the rotary_dim / 2
  sines of the same angles, angle i of row p belonging to rotation pair i.
* Pairing of dimensions: `is_neox=False` rotates adjacent pairs
  (2i, 2i + 1), the literal block-diagonal form; `is_neox=True` rotates the
  pairs (i, i + rotary_dim / 2), the same matrix with its rows and columns
  permuted.  Both are provided.
* Direction: a pair (x, y) with angle a becomes
  (x cos a - y sin a, y cos a + x sin a), the counter-clockwise rotation
  (multiplication of x + iy by e^{ia}).
* Dimensions at and above rotary_dim pass through unchanged.
* Both Q (all query heads) and K (all KV heads) of a token use the row of that
  token's position; V is not rotated.

The rotation is written as what the page calls it: a dense rotary_dim x
rotary_dim block-diagonal (up to the pairing permutation) rotation matrix per
token, applied by a matrix product.  The fused op is that rotation followed by
the plain scatter of `oracle.paging.write_cache`.
"""

from __future__ import annotations

import numpy as np

from . import paging


def _f64(x) -> np.ndarray:
    try:
        import torch
        if isinstance(x, torch.Tensor):
            return x.detach().to("cpu", torch.float64).numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.asarray(x, dtype=np.float64)


def pair_indices(rotary_dim: int, is_neox: bool):
    """The two dimensions of each rotation pair i < rotary_dim / 2."""
    half = rotary_dim // 2
    i = np.arange(half)
    if is_neox:
        return i, i + half
    return 2 * i, 2 * i + 1


def rotation_matrix(cos_sin_row, rotary_dim: int, is_neox: bool) -> np.ndarray:
    """The rotary_dim x rotary_dim rotation matrix of one table row.

    For pair i on dimensions (a, b) with angle cosine c and sine s, the block
    [[c, -s], [s, c]] sits on rows / columns (a, b); every other entry is 0.
    """
    if rotary_dim % 2:
        raise ValueError("rotary_dim must be even")
    row = _f64(cos_sin_row)
    half = rotary_dim // 2
    cos, sin = row[:half], row[half:rotary_dim]
    a, b = pair_indices(rotary_dim, is_neox)
    R = np.zeros((rotary_dim, rotary_dim), dtype=np.float64)
    R[a, a] = cos
    R[a, b] = -sin
    R[b, a] = sin
    R[b, b] = cos
    return R


def apply_rope(x, positions, cos_sin_cache, rotary_dim: int, is_neox: bool) -> np.ndarray:
    """x: [T, H, D] -> float64 [T, H, D] with the first rotary_dim dimensions of
    every head of token t rotated by the matrix of row positions[t]."""
    x = _f64(x)
    table = _f64(cos_sin_cache)
    T, H, D = x.shape
    if rotary_dim > D:
        raise ValueError("rotary_dim > head_dim")
    out = x.copy()
    for t in range(T):
        p = int(positions[t])
        if not 0 <= p < table.shape[0]:
            raise IndexError(f"position {p} outside the table")
        R = rotation_matrix(table[p], rotary_dim, is_neox)
        out[t, :, :rotary_dim] = x[t, :, :rotary_dim] @ R.T
    return out


def rope_reshape_and_cache(positions, query, key, value, key_cache, value_cache, slots,
                           cos_sin_cache, rotary_dim: int, is_neox: bool):
    """Fused step: rotate Q and K of every token, then scatter the rotated K and
    the unchanged V into the caches (float64 arrays, modified in place) at
    `slots`; a negative slot skips the scatter for that token.

    Returns (rotated query, rotated key), both float64 [T, heads, D].
    """
    q_rot = apply_rope(query, positions, cos_sin_cache, rotary_dim, is_neox)
    k_rot = apply_rope(key, positions, cos_sin_cache, rotary_dim, is_neox)
    paging.write_cache(key_cache, value_cache, k_rot, _f64(value), slots)
    return q_rot, k_rot
