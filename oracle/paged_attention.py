"""CPU oracle for batched paged-KV decode attention and slot-mapped KV append.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import or call
this module: only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` use it.  It shares no code with the CUDA library and it
imports nothing from the package; it receives plain numpy arrays.

It is the plain definition written out, in float64, with no blocking, fusion
or reordering (split-K and online softmax are ways to reach the same result,
so they do not appear here):

* Gather.  For sequence ``s`` and KV head ``g`` the context is the rows
  ``K_s[i] = k_cache[block_tables[s, i // bs], g, i % bs, :]`` for
  ``0 <= i < context_lens[s]``; the same for V.  (ferrum-kernels
  ``src/backend/cuda/paged.rs``, ``paged_decode_attention``: a sequence's
  tokens live in blocks of ``block_size`` reached through its row of the block
  table, ``max_kv_len = block_size * max_num_blocks_per_seq``; kapsl-backends
  ``src/gguf_native.rs``, ``forward_batch_decode_greedy``: ``context_lens[b]``
  is the length *after* this step's token.)
* GQA.  Query head ``h`` reads KV head ``h // (H / Hkv)`` (cortiq-engine
  ``src/gpu_cuda.rs``, plan construction ``hpk = nh / nkv`` and the parity test
  that hands query rows ``g*hpk .. (g+1)*hpk`` to KV head ``g``).
* Scores ``z_i = scale * q . K_s[i]``; ``scale`` is an argument (kapsl
  ``one_token_compute`` passes ``scale = 1/sqrt(head_dim)``).
* Softmax ``p_i = exp(z_i - max z) / sum_j exp(z_j - max z)`` and output
  ``sum_i p_i V_s[i]``.
* ``context_len == 0`` gives zeros (an empty softmax has no value; zeros are
  the plainest total definition).
* Multi-token queries (``varlen``): query ``t`` of a sequence sits at
  ``pos_offset + t`` and attends causally to positions ``0 .. pos_offset + t``.
* Append.  Token ``t`` with ``slot = slot_mapping[t] >= 0`` is written to
  block ``slot // bs``, row ``slot % bs`` of both pools, for every KV head;
  negative slots are skipped (kapsl ``launch_batch_kv_write`` with a
  physical block and position-in-block per token, as one integer).

* vLLM cache layout (ferrum-kernels ``src/backend/cuda/paged.rs``, the
  vLLM-layout paged write and ``paged_decode_attention_v2``; the pages name
  the layout without spelling it out, so it is read as vLLM's published
  paged-attention layout with ``x = 16 bytes / 2 = 8``): K is
  ``[NB][Hkv][D/8][bs][8]``, element ``d`` of the token at row ``o`` of block
  ``b`` at ``[b, h, d // 8, o, d % 8]``; V is ``[NB][Hkv][D][bs]``, at
  ``[b, h, d, o]``.  ``append_vllm_layout`` writes element by element;
  ``blocked_from_vllm_layout`` reads the pools back as ``[NB][Hkv][bs][D]``,
  after which the definitions above apply unchanged (``decode_vllm_layout``,
  ``varlen_vllm_layout``).  Pinned in
  ``tests/test_oracle_vllm_layout.py`` by a round trip through the blocked
  append and by chunk contiguity found by search.

Parity pins (in ``tests/test_oracle_pins.py``): contiguous equivalence against
``torch.nn.functional.scaled_dot_product_attention`` in float64, invariance
under a permutation of physical blocks, ``context_len == 1`` returning that V
row exactly, identical keys (or ``scale == 0``) returning the mean of V, GQA
equal to MHA with repeated KV heads, a hand-derived worked example under
``tests/golden/``, and planted mistakes that each of those must catch.
"""

from __future__ import annotations

import numpy as np


class OracleInputError(ValueError):
    """The inputs break a precondition the definition needs."""


def kv_head_of(h: int, group: int) -> int:
    """KV head read by query head ``h``: consecutive query heads share one."""
    return h // group


def gather_rows(cache: np.ndarray, table_row: np.ndarray, context_len: int,
                kv_head: int) -> np.ndarray:
    """Rows ``0 .. context_len-1`` of one sequence and KV head, as float64."""
    bs = cache.shape[2]
    i = np.arange(context_len)
    blocks = table_row[i // bs]
    return cache[blocks, kv_head, i % bs, :].astype(np.float64)


def softmax(z: np.ndarray) -> np.ndarray:
    """Softmax along the last axis, shifted by its max before ``exp``."""
    e = np.exp(z - z.max(axis=-1, keepdims=True))
    return e / e.sum(axis=-1, keepdims=True)


def _check_tables(block_tables, context_lens, num_blocks, block_size):
    B, mbps = block_tables.shape
    for s in range(B):
        L = int(context_lens[s])
        if L < 0 or L > mbps * block_size:
            raise OracleInputError(f"context_lens[{s}]={L} outside [0, {mbps * block_size}]")
        n = -(-L // block_size)
        ids = block_tables[s, :n]
        if n and (ids.min() < 0 or ids.max() >= num_blocks):
            raise OracleInputError(f"block id out of range in sequence {s}")


def decode(q, k_cache, v_cache, block_tables, context_lens, scale, seqs=None):
    """Attention of one query token per sequence over its paged context.

    Arguments are numpy arrays: ``q`` f16 ``[B][H][D]``, caches f16
    ``[NB][Hkv][bs][D]``, ``block_tables`` int ``[B][MBPS]``, ``context_lens``
    int ``[B]``.  Returns float64 ``[B][H][D]``; with ``seqs`` only those
    sequences are computed (the other rows stay zero).
    """
    q = np.asarray(q)
    B, H, D = q.shape
    NB, Hkv, bs, Dk = k_cache.shape
    if Dk != D or v_cache.shape != k_cache.shape:
        raise OracleInputError("cache shape does not match q")
    if H % Hkv:
        raise OracleInputError("num_heads must be a multiple of num_kv_heads")
    group = H // Hkv
    _check_tables(block_tables, context_lens, NB, bs)
    out = np.zeros((B, H, D), np.float64)
    for s in (range(B) if seqs is None else seqs):
        L = int(context_lens[s])
        if L == 0:
            continue
        row = block_tables[s]
        for h in range(H):
            g = kv_head_of(h, group)
            K = gather_rows(k_cache, row, L, g)
            V = gather_rows(v_cache, row, L, g)
            z = scale * (K @ q[s, h].astype(np.float64))
            p = softmax(z)
            out[s, h] = p @ V
    return out


def decode_fast(q, k_cache, v_cache, block_tables, context_lens, scale, seqs=None):
    """Same definition as :func:`decode`, gathering each (sequence, KV head)
    once and scoring its whole query group with one matrix product.

    Used where the contexts are long (the gather dominates); the arithmetic
    per output element is the same sums in float64.
    """
    q = np.asarray(q)
    B, H, D = q.shape
    NB, Hkv, bs, _ = k_cache.shape
    if H % Hkv:
        raise OracleInputError("num_heads must be a multiple of num_kv_heads")
    group = H // Hkv
    _check_tables(block_tables, context_lens, NB, bs)
    out = np.zeros((B, H, D), np.float64)
    for s in (range(B) if seqs is None else seqs):
        L = int(context_lens[s])
        if L == 0:
            continue
        row = block_tables[s]
        for g in range(Hkv):
            heads = [h for h in range(H) if kv_head_of(h, group) == g]
            K = gather_rows(k_cache, row, L, g)
            V = gather_rows(v_cache, row, L, g)
            Z = scale * (q[s, heads].astype(np.float64) @ K.T)  # [G][L]
            P = softmax(Z)
            out[s, heads] = P @ V
    return out


def varlen(q, k_cache, v_cache, cu_seqlens_q, pos_offsets, block_tables, scale):
    """Multi-token queries over the paged context, causal.

    ``q`` f16 ``[total_q][H][D]`` token-major; the queries of sequence ``s``
    are rows ``cu_seqlens_q[s] .. cu_seqlens_q[s+1]-1``; query ``t`` of ``s``
    sits at position ``pos_offsets[s] + t`` and attends to positions
    ``0 .. pos_offsets[s] + t`` of its sequence (ferrum-kernels
    ``src/backend/cuda/paged.rs``, ``paged_varlen_attention`` and
    ``paged_decode_attention``: ``pos_offset = final_kv_len - q_len``).
    Returns float64 ``[total_q][H][D]``.
    """
    q = np.asarray(q)
    total_q, H, D = q.shape
    NB, Hkv, bs, _ = k_cache.shape
    if H % Hkv:
        raise OracleInputError("num_heads must be a multiple of num_kv_heads")
    group = H // Hkv
    cu = np.asarray(cu_seqlens_q).astype(np.int64)
    B = len(cu) - 1
    if cu[0] != 0 or np.any(np.diff(cu) < 0) or cu[-1] != total_q:
        raise OracleInputError("cu_seqlens_q must rise from 0 to total_q")
    lens = np.array([int(pos_offsets[s]) + int(cu[s + 1] - cu[s]) for s in range(B)])
    if np.any(np.asarray(pos_offsets) < 0):
        raise OracleInputError("negative pos_offset")
    _check_tables(block_tables, lens, NB, bs)
    out = np.zeros((total_q, H, D), np.float64)
    for s in range(B):
        row = block_tables[s]
        for t in range(int(cu[s + 1] - cu[s])):
            L = int(pos_offsets[s]) + t + 1
            i = int(cu[s]) + t
            for h in range(H):
                g = kv_head_of(h, group)
                K = gather_rows(k_cache, row, L, g)
                V = gather_rows(v_cache, row, L, g)
                z = scale * (K @ q[i, h].astype(np.float64))
                out[i, h] = softmax(z) @ V
    return out


def varlen_fast(q, k_cache, v_cache, cu_seqlens_q, pos_offsets, block_tables, scale):
    """Same definition as :func:`varlen`, gathering each (sequence, KV head)
    once up to its last query's position and scoring the group's query heads
    together, one query at a time over its own causal prefix.  Used where the
    contexts are long; the arithmetic per output element is the same sums in
    float64."""
    q = np.asarray(q)
    total_q, H, D = q.shape
    NB, Hkv, bs, _ = k_cache.shape
    if H % Hkv:
        raise OracleInputError("num_heads must be a multiple of num_kv_heads")
    group = H // Hkv
    cu = np.asarray(cu_seqlens_q).astype(np.int64)
    B = len(cu) - 1
    if cu[0] != 0 or np.any(np.diff(cu) < 0) or cu[-1] != total_q:
        raise OracleInputError("cu_seqlens_q must rise from 0 to total_q")
    if np.any(np.asarray(pos_offsets) < 0):
        raise OracleInputError("negative pos_offset")
    lens = np.array([int(pos_offsets[s]) + int(cu[s + 1] - cu[s]) for s in range(B)])
    _check_tables(block_tables, lens, NB, bs)
    out = np.zeros((total_q, H, D), np.float64)
    for s in range(B):
        n = int(cu[s + 1] - cu[s])
        if n == 0:
            continue
        row = block_tables[s]
        for g in range(Hkv):
            K = gather_rows(k_cache, row, int(lens[s]), g)
            V = gather_rows(v_cache, row, int(lens[s]), g)
            heads = [h for h in range(H) if kv_head_of(h, group) == g]
            for t in range(n):
                L = int(pos_offsets[s]) + t + 1
                i = int(cu[s]) + t
                Z = scale * (q[i, heads].astype(np.float64) @ K[:L].T)
                out[i, heads] = softmax(Z) @ V[:L]
    return out


def append(k, v, slot_mapping, k_cache, v_cache):
    """Scatter new K/V rows into the pools in place; returns the skipped
    out-of-range token indices (slots ``>= num_blocks * block_size``)."""
    NB, Hkv, bs, D = k_cache.shape
    bad = []
    for t, slot in enumerate(np.asarray(slot_mapping).tolist()):
        if slot < 0:
            continue
        if slot >= NB * bs:
            bad.append(t)
            continue
        blk, off = divmod(slot, bs)
        k_cache[blk, :, off, :] = k[t]
        v_cache[blk, :, off, :] = v[t]
    return bad


VLLM_X = 8  # f16 elements in one 16-byte K chunk of the vLLM layout


def append_vllm_layout(k, v, slot_mapping, k_cache, v_cache):
    """``append`` into vLLM-layout pools (K ``[NB][Hkv][D/8][bs][8]``, V
    ``[NB][Hkv][D][bs]``), one element at a time; returns the skipped
    out-of-range token indices."""
    NB, Hkv, D8, bs, x = k_cache.shape
    bad = []
    for t, slot in enumerate(np.asarray(slot_mapping).tolist()):
        if slot < 0:
            continue
        if slot >= NB * bs:
            bad.append(t)
            continue
        blk, off = divmod(slot, bs)
        for h in range(Hkv):
            for d in range(D8 * x):
                k_cache[blk, h, d // x, off, d % x] = k[t, h, d]
                v_cache[blk, h, d, off] = v[t, h, d]
    return bad


def blocked_from_vllm_layout(k_cache, v_cache, blocks=None):
    """The vLLM-layout pools read as ``[n][Hkv][bs][D]`` pools (all blocks,
    or those listed in ``blocks``, in that order)."""
    NB, Hkv, D8, bs, x = k_cache.shape
    D = D8 * x
    idx = np.arange(NB) if blocks is None else np.asarray(blocks)
    kb = np.empty((len(idx), Hkv, bs, D), dtype=k_cache.dtype)
    vb = np.empty((len(idx), Hkv, bs, D), dtype=v_cache.dtype)
    for d in range(D):
        kb[:, :, :, d] = k_cache[idx, :, d // x, :, d % x]
        vb[:, :, :, d] = v_cache[idx, :, d, :]
    return kb, vb


def _blocked_view_of_used(k_cache, v_cache, block_tables, context_lens, seqs):
    """The blocks that ``seqs`` read (positions below ``context_lens``) from
    vLLM-layout pools, as blocked pools, with the tables renumbered to match."""
    bs = k_cache.shape[3]
    bt = np.asarray(block_tables)
    lens = np.asarray(context_lens)
    _check_tables(bt, lens, k_cache.shape[0], bs)
    chosen = range(len(lens)) if seqs is None else seqs
    used = sorted({int(bt[s, j]) for s in chosen for j in range(-(-int(lens[s]) // bs))}) or [0]
    where = {b: i for i, b in enumerate(used)}
    kb, vb = blocked_from_vllm_layout(k_cache, v_cache, used)
    bt2 = np.zeros_like(bt)
    for s in chosen:
        for j in range(-(-int(lens[s]) // bs)):
            bt2[s, j] = where[int(bt[s, j])]
    return kb, vb, bt2


def decode_vllm_layout(q, k_cache, v_cache, block_tables, context_lens, scale, seqs=None,
                       fast=False):
    """``decode`` (``decode_fast`` with ``fast``) over vLLM-layout pools: the
    blocks the chosen sequences read are read back as blocked pools (tables
    renumbered to match), then the definition runs on those."""
    kb, vb, bt2 = _blocked_view_of_used(k_cache, v_cache, block_tables, context_lens, seqs)
    return (decode_fast if fast else decode)(q, kb, vb, bt2, np.asarray(context_lens), scale,
                                             seqs)


def varlen_vllm_layout(q, k_cache, v_cache, cu_seqlens_q, pos_offsets, block_tables, scale):
    """``varlen`` over vLLM-layout pools (ferrum-kernels
    ``src/backend/cuda/paged.rs``, ``paged_varlen_attention_vllm_layout``):
    the blocks the sequences read, up to their last query's position, are
    read back as blocked pools, then ``varlen`` runs on those."""
    cu = np.asarray(cu_seqlens_q).astype(np.int64)
    ends = np.asarray(pos_offsets).astype(np.int64) + np.diff(cu)
    kb, vb, bt2 = _blocked_view_of_used(k_cache, v_cache, block_tables, ends, None)
    return varlen(q, kb, vb, cu_seqlens_q, pos_offsets, bt2, scale)
