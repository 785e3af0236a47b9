"""CPU oracle for the fused QKV split + per-head RMS norm + rotary embedding +
paged append (ferrum-kernels ``src/backend/cuda/paged.rs``,
``split_qkv_norm_rope_into_paged_cache`` and its ``_varlen`` form).

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import or call
this module; it shares no code with the CUDA library and imports nothing
from the package.

The pages give only the launch of this step, so its arithmetic is read as
follows (each reading is stated where it is used):

* Input row ``qkv[t]`` of token ``t`` holds the ``H`` query heads, then the
  ``Hkv`` key heads, then the ``Hkv`` value heads, ``D`` elements each (the
  launch covers ``q_heads + 2 * kv_heads`` heads per token).
* Token ``t`` of sequence ``s`` sits at position ``p = pos_offsets[s] + t``
  (its row in ``cu_seqlens_q``); ``p`` is both its rotary position and its
  row in the paged cache.
* Query and key heads are RMS-normalised over their ``D`` elements when a
  weight vector is given: ``y = x / sqrt(mean(x^2) + eps) * w``; value heads
  are not.
* Rotary embedding, rotate-half pairing: element ``i < D/2`` pairs with
  ``i + D/2``; with ``c = cos[p][i]``, ``s = sin[p][i]`` the pair ``(a, b)``
  becomes ``(a c - b s, b c + a s)``.  The tables are inputs.
* Queries go to ``q_out[t][h][:]`` (token-major); rotated keys and the value
  rows go to the paged pools at slot ``block_tables[s][p // bs] * bs + p % bs``
  like ``append``.

Everything is float64; the pools and ``q_out`` returned are the float64
results (the pools also receive them rounded to the pool dtype).
"""

from __future__ import annotations

import numpy as np


class QkvInputError(ValueError):
    """The inputs break a precondition of the definition."""


def rms_norm(x: np.ndarray, w, eps: float) -> np.ndarray:
    """``x / sqrt(mean(x^2) + eps) * w`` over the last axis, float64."""
    x = np.asarray(x, np.float64)
    r = np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)
    y = x / r
    return y if w is None else y * np.asarray(w, np.float64)


def rotate(x: np.ndarray, cos_row, sin_row) -> np.ndarray:
    """Rotary embedding of one head vector ``x`` (length D), rotate-half
    pairs ``(i, i + D/2)`` turned by the angle whose cosine and sine are
    ``cos_row[i]``, ``sin_row[i]``."""
    x = np.asarray(x, np.float64)
    half = x.shape[-1] // 2
    a, b = x[..., :half], x[..., half:]
    c = np.asarray(cos_row, np.float64)
    s = np.asarray(sin_row, np.float64)
    return np.concatenate([a * c - b * s, b * c + a * s], axis=-1)


def qkv_norm_rope_append(qkv, q_norm_w, k_norm_w, cos, sin, k_cache, v_cache, cu_seqlens_q,
                         pos_offsets, block_tables, num_heads, num_kv_heads, eps):
    """Returns ``q_out`` float64 ``[total_q][H][D]`` and writes the rotated
    keys and the values into ``k_cache`` / ``v_cache`` (``[NB][Hkv][bs][D]``)
    in place.  Returns also the float64 key rows written, ``[total_q][Hkv][D]``."""
    qkv = np.asarray(qkv)
    total_q, width = qkv.shape
    H, Hkv = int(num_heads), int(num_kv_heads)
    if width % (H + 2 * Hkv):
        raise QkvInputError("qkv row width is not (H + 2 Hkv) * D")
    D = width // (H + 2 * Hkv)
    NB, Hkv_c, bs, Dc = k_cache.shape
    if Hkv_c != Hkv or Dc != D or D % 2:
        raise QkvInputError("cache shape does not match")
    cu = np.asarray(cu_seqlens_q).astype(np.int64)
    if cu[0] != 0 or np.any(np.diff(cu) < 0) or cu[-1] != total_q:
        raise QkvInputError("cu_seqlens_q must rise from 0 to total_q")
    q_out = np.zeros((total_q, H, D), np.float64)
    k_rows = np.zeros((total_q, Hkv, D), np.float64)
    for s in range(len(cu) - 1):
        for t in range(int(cu[s + 1] - cu[s])):
            row = int(cu[s]) + t
            p = int(pos_offsets[s]) + t
            if p < 0 or p >= cos.shape[0] or p >= block_tables.shape[1] * bs:
                raise QkvInputError(f"position {p} outside the tables or the cache")
            blk = int(block_tables[s][p // bs])
            if not 0 <= blk < NB:
                raise QkvInputError(f"block id {blk} out of range")
            x = qkv[row].astype(np.float64).reshape(H + 2 * Hkv, D)
            for h in range(H):
                y = x[h] if q_norm_w is None else rms_norm(x[h], q_norm_w, eps)
                q_out[row, h] = rotate(y, cos[p], sin[p])
            for g in range(Hkv):
                y = x[H + g] if k_norm_w is None else rms_norm(x[H + g], k_norm_w, eps)
                k_rows[row, g] = rotate(y, cos[p], sin[p])
                k_cache[blk, g, p % bs, :] = k_rows[row, g]
                v_cache[blk, g, p % bs, :] = x[H + Hkv + g]
    return q_out, k_rows
