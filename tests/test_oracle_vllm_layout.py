"""Pins of the oracle's vLLM-layout functions (ferrum-kernels
src/backend/cuda/paged.rs, the vLLM-layout paged write and
paged_decode_attention_v2), on the CPU.

The layout is vLLM's published paged-attention layout: K
``[NB][Hkv][D/8][bs][8]``, V ``[NB][Hkv][D][bs]``.  What pins it here:

* round trip: tokens appended with ``append_vllm_layout`` and read back with
  ``blocked_from_vllm_layout`` give, bit for bit, the pools the (separately
  pinned) blocked ``append`` builds from the same tokens, untouched entries
  included;
* chunk contiguity found by search: every 16-byte K chunk that holds data
  is an aligned run of 8 consecutive head-dim values of one token row, and
  every V row ``[b, h, d, :]`` holds element d of the block's tokens in slot
  order;
* ``decode_vllm_layout`` equals ``decode``, and ``varlen_vllm_layout`` equals
  ``varlen``, on the same logical cache.

Each planted mistake below must break one of them.  D = 64 makes D/8 = 8,
so swapping the chunk and element axes keeps every shape valid.
"""

import inspect
import types

import numpy as np
import pytest

import oracle
from oracle import paged_attention as OPA


def _tokens(rng, T, Hkv, D):
    # distinct integers (exact in f16 up to 2048), so a value identifies its
    # (token, head, d)
    n = T * Hkv * D
    assert n <= 2048
    vals = rng.permutation(n).astype(np.float64) + 1.0
    k = vals.reshape(T, Hkv, D).astype(np.float16)
    v = (-vals).reshape(T, Hkv, D).astype(np.float16)
    return k, v


def _case(seed=0, NB=6, Hkv=2, bs=16, D=64, T=16):
    rng = np.random.default_rng(seed)
    k, v = _tokens(rng, T, Hkv, D)
    slots = rng.choice(NB * bs, size=T, replace=False).astype(np.int32)
    slots[rng.choice(T, size=4, replace=False)] = -1
    return k, v, slots, NB, Hkv, bs, D


def round_trip_ok(mod, seed=0):
    k, v, slots, NB, Hkv, bs, D = _case(seed)
    kb = np.zeros((NB, Hkv, bs, D), np.float16)
    vb = np.zeros_like(kb)
    oracle.append(k, v, slots, kb, vb)
    kv = np.zeros((NB, Hkv, D // 8, bs, 8), np.float16)
    vv = np.zeros((NB, Hkv, D, bs), np.float16)
    mod.append_vllm_layout(k, v, slots, kv, vv)
    k2, v2 = mod.blocked_from_vllm_layout(kv, vv)
    return (np.array_equal(k2.view(np.uint16), kb.view(np.uint16))
            and np.array_equal(v2.view(np.uint16), vb.view(np.uint16)))


def contiguity_ok(mod, seed=1):
    k, v, slots, NB, Hkv, bs, D = _case(seed)
    kv = np.zeros((NB, Hkv, D // 8, bs, 8), np.float16)
    vv = np.zeros((NB, Hkv, D, bs), np.float16)
    mod.append_vllm_layout(k, v, slots, kv, vv)
    where = {}  # value -> (token, head, d)
    for t in range(k.shape[0]):
        for h in range(Hkv):
            for d in range(D):
                where[float(k[t, h, d])] = (t, h, d)
    chunks = kv.reshape(-1, 8)
    for ch in chunks:
        if not ch.any():
            continue
        hits = [where.get(float(x)) for x in ch]
        if any(hh is None for hh in hits):
            return False
        t0, h0, d0 = hits[0]
        if d0 % 8 or hits != [(t0, h0, d0 + e) for e in range(8)]:
            return False
    # V: row [b, h, d, :] is element d of the tokens at rows 0..bs-1 of block b
    slot_of = {int(s): t for t, s in enumerate(slots) if s >= 0}
    for b in range(NB):
        for o in range(bs):
            t = slot_of.get(b * bs + o)
            want = v[t] if t is not None else np.zeros((Hkv, D), np.float16)
            if not np.array_equal(vv[b, :, :, o], want):
                return False
    return True


def decode_ok(mod, seed=2):
    rng = np.random.default_rng(seed)
    NB, Hkv, bs, D, H = 10, 2, 16, 64, 8
    lens = np.array([1, 17, 40, 64], np.int32)
    perm = rng.permutation(NB).astype(np.int32)
    bt = np.full((4, 4), 9, np.int32)
    cur = 0
    for s, L in enumerate(lens):
        n = -(-int(L) // bs)
        bt[s, :n] = perm[cur:cur + n]
        cur += n
    T = int(lens.sum())
    k = rng.standard_normal((T, Hkv, D)).astype(np.float16)
    v = rng.standard_normal((T, Hkv, D)).astype(np.float16)
    slots = np.concatenate([bt[s, np.arange(L) // bs] * bs + np.arange(L) % bs
                            for s, L in enumerate(lens)]).astype(np.int32)
    kb = np.zeros((NB, Hkv, bs, D), np.float16)
    vb = np.zeros_like(kb)
    oracle.append(k, v, slots, kb, vb)
    kv = np.zeros((NB, Hkv, D // 8, bs, 8), np.float16)
    vv = np.zeros((NB, Hkv, D, bs), np.float16)
    mod.append_vllm_layout(k, v, slots, kv, vv)
    q = rng.standard_normal((4, H, D)).astype(np.float16)
    ref = oracle.decode(q, kb, vb, bt, lens, 0.125)
    got = mod.decode_vllm_layout(q, kv, vv, bt, lens, 0.125)
    part = mod.decode_vllm_layout(q, kv, vv, bt, lens, 0.125, seqs=[2])
    return (np.array_equal(got, ref) and np.array_equal(part[2], ref[2])
            and not part[[0, 1, 3]].any())


def varlen_ok(mod, seed=5):
    """Several causal queries per sequence: the vLLM-layout varlen equals the
    blocked varlen on the same logical cache."""
    rng = np.random.default_rng(seed)
    NB, Hkv, bs, D, H = 12, 2, 16, 64, 4
    prefix = np.array([0, 15, 30], np.int32)
    q_lens = np.array([3, 1, 5], np.int32)
    lens = prefix + q_lens
    perm = rng.permutation(NB).astype(np.int32)
    bt = np.full((3, 3), 11, np.int32)
    cur = 0
    for s, L in enumerate(lens):
        n = -(-int(L) // bs)
        bt[s, :n] = perm[cur:cur + n]
        cur += n
    T = int(lens.sum())
    k = rng.standard_normal((T, Hkv, D)).astype(np.float16)
    v = rng.standard_normal((T, Hkv, D)).astype(np.float16)
    slots = np.concatenate([bt[s, np.arange(L) // bs] * bs + np.arange(L) % bs
                            for s, L in enumerate(lens)]).astype(np.int32)
    kb = np.zeros((NB, Hkv, bs, D), np.float16)
    vb = np.zeros_like(kb)
    oracle.append(k, v, slots, kb, vb)
    kv = np.zeros((NB, Hkv, D // 8, bs, 8), np.float16)
    vv = np.zeros((NB, Hkv, D, bs), np.float16)
    mod.append_vllm_layout(k, v, slots, kv, vv)
    cu = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    q = rng.standard_normal((int(cu[-1]), H, D)).astype(np.float16)
    ref = oracle.varlen(q, kb, vb, cu, prefix, bt, 0.125)
    got = mod.varlen_vllm_layout(q, kv, vv, cu, prefix, bt, 0.125)
    return np.array_equal(got, ref)


def all_pins(mod):
    return {"round_trip": round_trip_ok(mod), "contiguity": contiguity_ok(mod),
            "decode": decode_ok(mod), "varlen": varlen_ok(mod)}


def test_oracle_vllm_layout_pins():
    res = all_pins(OPA)
    assert all(res.values()), res


def test_vllm_adapter_on_selected_blocks():
    k, v, slots, NB, Hkv, bs, D = _case(3)
    kv = np.zeros((NB, Hkv, D // 8, bs, 8), np.float16)
    vv = np.zeros((NB, Hkv, D, bs), np.float16)
    oracle.append_vllm_layout(k, v, slots, kv, vv)
    full_k, full_v = oracle.blocked_from_vllm_layout(kv, vv)
    sel_k, sel_v = oracle.blocked_from_vllm_layout(kv, vv, [4, 1])
    assert np.array_equal(sel_k, full_k[[4, 1]]) and np.array_equal(sel_v, full_v[[4, 1]])


def test_vllm_append_reports_out_of_range_slots():
    k, v, slots, NB, Hkv, bs, D = _case(4)
    slots = slots.copy()
    slots[0] = NB * bs
    kv = np.zeros((NB, Hkv, D // 8, bs, 8), np.float16)
    vv = np.zeros((NB, Hkv, D, bs), np.float16)
    assert oracle.append_vllm_layout(k, v, slots, kv, vv) == [0]


def test_vllm_decode_rejects_bad_block_ids():
    kv = np.zeros((2, 1, 8, 16, 8), np.float16)
    vv = np.zeros((2, 1, 64, 16), np.float16)
    q = np.zeros((1, 1, 64), np.float16)
    with pytest.raises(oracle.OracleInputError):
        oracle.decode_vllm_layout(q, kv, vv, np.array([[5]], np.int32),
                                  np.array([3], np.int32), 0.125)


MUTATIONS = {
    "k_chunk_and_element_swapped": ("k_cache[blk, h, d // x, off, d % x] = k[t, h, d]",
                                    "k_cache[blk, h, d % x, off, d // x] = k[t, h, d]"),
    "v_not_transposed": ("v_cache[blk, h, d, off] = v[t, h, d]",
                         "v_cache.reshape(v_cache.shape[0], Hkv, -1)[blk, h, off * (D8 * x) + d] = v[t, h, d]"),
    "adapter_k_axes_swapped": ("kb[:, :, :, d] = k_cache[idx, :, d // x, :, d % x]",
                               "kb[:, :, :, d] = k_cache[idx, :, d % x, :, d // x]"),
    "adapter_v_from_k": ("vb[:, :, :, d] = v_cache[idx, :, d, :]",
                         "vb[:, :, :, d] = k_cache[idx, :, d // x, :, d % x]"),
    "decode_tables_not_renumbered": ("bt2[s, j] = where[int(bt[s, j])]", "bt2[s, j] = int(bt[s, j]) % len(used)"),
    "varlen_reads_only_the_prefix": ("ends = np.asarray(pos_offsets).astype(np.int64) + np.diff(cu)",
                                     "ends = np.asarray(pos_offsets).astype(np.int64) + 1"),
}


def mutant(name):
    old, new = MUTATIONS[name]
    src = inspect.getsource(OPA)
    assert src.count(old) == 1, f"mutation {name} does not apply"
    mod = types.ModuleType(f"oracle_vllm_mutant_{name}")
    exec(compile(src.replace(old, new), f"<mutant {name}>", "exec"), mod.__dict__)
    return mod


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_vllm_mistake_is_caught(name):
    res = all_pins(mutant(name))
    assert not all(res.values()), f"{name} passed every pin: {res}"
