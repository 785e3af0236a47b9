"""Pins of the CPU oracle to things other than itself (no GPU needed).

Each pin is a function of a ``decode`` implementation so that the same checks
can be run against deliberately broken copies of the oracle (the planted
mistakes at the bottom): every plausible mistake must trip at least one pin.
"""

import inspect
import json
import math
import os
import types
from fractions import Fraction

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from oracle import paged_attention as OPA
from paged_kv_decode_08_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_example.json")


# ---------------------------------------------------------------------------
# pins
# ---------------------------------------------------------------------------

def sdpa_contiguous(w: W.Workload) -> np.ndarray:
    """Attention on each sequence's contiguous rows (never paged), computed by
    torch's scaled_dot_product_attention in float64, KV heads repeated so query
    head h reads KV head h // G."""
    G = w.group
    out = np.zeros((w.num_seqs, w.num_heads, w.head_dim), np.float64)
    for s in range(w.num_seqs):
        L = int(w.context_lens[s])
        if L == 0:
            continue
        K = torch.from_numpy(w.seq_k[s].astype(np.float64)).permute(1, 0, 2)  # [Hkv][L][D]
        V = torch.from_numpy(w.seq_v[s].astype(np.float64)).permute(1, 0, 2)
        K = K.repeat_interleave(G, dim=0)
        V = V.repeat_interleave(G, dim=0)
        q = torch.from_numpy(w.q[s].astype(np.float64)).unsqueeze(1)  # [H][1][D]
        o = F.scaled_dot_product_attention(q, K, V, scale=w.scale)
        out[s] = o.squeeze(1).numpy()
    return out


def run(decode_fn, w, kc=None, vc=None, tables=None):
    if kc is None:
        kc, vc = W.host_pool(w)
    return decode_fn(w.q, kc, vc, w.block_tables if tables is None else tables,
                     w.context_lens, w.scale)


def pin_sdpa(decode_fn, w):
    ref = sdpa_contiguous(w)
    got = run(decode_fn, w)
    return np.allclose(got, ref, rtol=1e-10, atol=1e-12)


def pin_permutation(decode_fn, w, seed=7):
    kc, vc = W.host_pool(w)
    base = run(decode_fn, w, kc, vc)
    rng = np.random.default_rng(seed)
    perm = rng.permutation(w.num_blocks)  # new position of old block b is perm[b]
    kc2 = np.empty_like(kc)
    vc2 = np.empty_like(vc)
    kc2[perm] = kc
    vc2[perm] = vc
    tables2 = perm[w.block_tables].astype(np.int32)
    moved = run(decode_fn, w, kc2, vc2, tables2)
    return np.array_equal(base, moved)


def _single_token_case(seed):
    return W.small_random(seed, num_seqs=3, num_heads=4, num_kv_heads=2, head_dim=64,
                          block_size=16, lens=[1, 1, 1])


def pin_len1(decode_fn, seed=11):
    w = _single_token_case(seed)
    got = run(decode_fn, w)
    for s in range(w.num_seqs):
        for h in range(w.num_heads):
            if not np.array_equal(got[s, h], w.seq_v[s][0, h // w.group].astype(np.float64)):
                return False
    return True


def pin_identical_keys(decode_fn, seed=13):
    w = W.small_random(seed, num_seqs=2, num_heads=4, num_kv_heads=2, head_dim=64,
                       block_size=16, lens=[37, 5])
    for s in range(w.num_seqs):
        w.seq_k[s][:] = w.seq_k[s][0]
    got = run(decode_fn, w)
    for s in range(w.num_seqs):
        mean = w.seq_v[s].astype(np.float64).mean(axis=0)  # [Hkv][D]
        for h in range(w.num_heads):
            if not np.allclose(got[s, h], mean[h // w.group], rtol=1e-12, atol=1e-13):
                return False
    return True


def pin_scale_zero(decode_fn, seed=17):
    w = W.small_random(seed, num_seqs=2, num_heads=2, num_kv_heads=1, head_dim=64,
                       block_size=32, lens=[33, 64])
    kc, vc = W.host_pool(w)
    got = decode_fn(w.q, kc, vc, w.block_tables, w.context_lens, 0.0)
    for s in range(w.num_seqs):
        mean = w.seq_v[s].astype(np.float64).mean(axis=0)
        for h in range(w.num_heads):
            if not np.allclose(got[s, h], mean[h // w.group], rtol=1e-12, atol=1e-13):
                return False
    return True


def pin_gqa_is_repeated_mha(decode_fn, w):
    """Repeating each KV head G times (as separate KV heads) must not change
    the result, with query head h then reading KV head h."""
    G = w.group
    kc, vc = W.host_pool(w)
    got = decode_fn(w.q, kc, vc, w.block_tables, w.context_lens, w.scale)
    kr = np.repeat(kc, G, axis=1)
    vr = np.repeat(vc, G, axis=1)
    mha = decode_fn(w.q, kr, vr, w.block_tables, w.context_lens, w.scale)
    # a BLAS product may round differently for a 1-row and a G-row operand
    return np.allclose(got, mha, rtol=1e-13, atol=1e-15)


def _load_golden():
    g = json.load(open(GOLDEN))

    def arr(x):
        return np.array([[[[float(v) for v in r] for r in h] for h in b] for b in x], np.float16)

    kc = arr(g["k_cache"])
    vc = arr(g["v_cache"])
    q = np.array(g["q"], np.float16)
    tables = np.array(g["block_tables"], np.int32)
    lens = np.array(g["context_lens"], np.int32)
    scale = math.log(3.0)
    exp = np.array([[[float(Fraction(v)) for v in h] for h in b] for b in g["expected_out"]])
    return q, kc, vc, tables, lens, scale, exp


def pin_golden(decode_fn):
    q, kc, vc, tables, lens, scale, exp = _load_golden()
    got = decode_fn(q, kc, vc, tables, lens, scale)
    return np.allclose(got, exp, rtol=1e-13, atol=1e-13)


def all_pins(decode_fn):
    w_a = W.small_random(101, num_seqs=3, num_heads=8, num_kv_heads=2, head_dim=64,
                         block_size=16, lens=[1, 17, 48])
    w_b = W.small_random(102, num_seqs=2, num_heads=7, num_kv_heads=1, head_dim=128,
                         block_size=32, lens=[31, 65])
    w_c = W.tiny()
    results = {}
    for name, fn in [
        ("sdpa_a", lambda: pin_sdpa(decode_fn, w_a)),
        ("sdpa_b", lambda: pin_sdpa(decode_fn, w_b)),
        ("sdpa_tiny", lambda: pin_sdpa(decode_fn, w_c)),
        ("permutation", lambda: pin_permutation(decode_fn, w_a)),
        ("len1", lambda: pin_len1(decode_fn)),
        ("identical_keys", lambda: pin_identical_keys(decode_fn)),
        ("scale_zero", lambda: pin_scale_zero(decode_fn)),
        ("gqa_repeat", lambda: pin_gqa_is_repeated_mha(decode_fn, w_a)),
        ("golden", lambda: pin_golden(decode_fn)),
    ]:
        try:
            results[name] = bool(fn())
        except Exception as exc:  # a broken oracle may also crash
            results[name] = f"raised {type(exc).__name__}: {exc}"
    return results


# ---------------------------------------------------------------------------
# the oracle against its pins
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("fn", [oracle.decode, oracle.decode_fast], ids=["decode", "decode_fast"])
def test_oracle_passes_every_pin(fn):
    res = all_pins(fn)
    assert all(v is True for v in res.values()), res


def test_decode_fast_equals_decode():
    w = W.small_random(5, num_seqs=4, num_heads=8, num_kv_heads=2, head_dim=64,
                       block_size=16, lens=[1, 15, 16, 100])
    kc, vc = W.host_pool(w)
    a = oracle.decode(w.q, kc, vc, w.block_tables, w.context_lens, w.scale)
    b = oracle.decode_fast(w.q, kc, vc, w.block_tables, w.context_lens, w.scale)
    assert np.allclose(a, b, rtol=1e-12, atol=1e-14)


def test_empty_context_gives_zeros():
    w = W.small_random(9, num_seqs=2, num_heads=2, num_kv_heads=1, head_dim=64,
                       block_size=16, lens=[5, 3])
    kc, vc = W.host_pool(w)
    lens = w.context_lens.copy()
    lens[0] = 0
    out = oracle.decode(w.q, kc, vc, w.block_tables, lens, w.scale)
    assert np.all(out[0] == 0.0)
    assert np.all(np.isfinite(out[1]))


def test_poison_is_never_read():
    """Unused pool blocks and rows past a length are NaN; the output is finite."""
    w = W.tiny()
    kc, vc = W.host_pool(w, fill=np.nan)
    out = oracle.decode(w.q, kc, vc, w.block_tables, w.context_lens, w.scale)
    assert np.all(np.isfinite(out))


def test_sharp_key_dominates():
    """A key scaled far above the rest takes (almost) all the softmax mass."""
    w = W.small_random(21, num_seqs=1, num_heads=1, num_kv_heads=1, head_dim=64,
                       block_size=16, lens=[40])
    pos = 23
    w.seq_k[0][pos] = (w.q[0, 0] * 60).astype(np.float16)
    kc, vc = W.host_pool(w)
    out = oracle.decode(w.q, kc, vc, w.block_tables, w.context_lens, w.scale)
    assert np.allclose(out[0, 0], w.seq_v[0][pos, 0].astype(np.float64), atol=1e-6)


def test_bad_inputs_are_rejected():
    w = W.tiny()
    kc, vc = W.host_pool(w)
    t = w.block_tables.copy()
    t[0, 0] = w.num_blocks
    with pytest.raises(oracle.OracleInputError):
        oracle.decode(w.q, kc, vc, t, w.context_lens, w.scale)
    lens = w.context_lens.copy()
    lens[1] = w.max_blocks_per_seq * w.block_size + 1
    with pytest.raises(oracle.OracleInputError):
        oracle.decode(w.q, kc, vc, w.block_tables, lens, w.scale)


# ---------------------------------------------------------------------------
# append pins
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("make", [W.tiny, lambda: W.small_random(
    31, num_seqs=5, num_heads=4, num_kv_heads=4, head_dim=64, block_size=32,
    lens=[1, 32, 33, 64, 70])], ids=["tiny", "random"])
def test_append_lands_where_the_table_says(make):
    """Slot arithmetic against the position layout the generator builds from
    contiguous rows by reshaping (no slot arithmetic there)."""
    w = make()
    before_k, before_v = W.host_pool(w, upto_last=True)
    after_k, after_v = W.host_pool(w, upto_last=False)
    k_new, v_new, slots = w.last_token_append()
    bad = oracle.append(k_new, v_new, slots, before_k, before_v)
    assert bad == []
    assert np.array_equal(before_k.view(np.uint16), after_k.view(np.uint16))
    assert np.array_equal(before_v.view(np.uint16), after_v.view(np.uint16))


def test_append_skips_negative_and_reports_out_of_range():
    w = W.tiny()
    kc, vc = W.host_pool(w)
    k0, v0 = kc.copy(), vc.copy()
    k_new = np.ones((3, w.num_kv_heads, w.head_dim), np.float16)
    slots = np.array([-1, -7, w.num_blocks * w.block_size], np.int32)
    bad = oracle.append(k_new, k_new, slots, kc, vc)
    assert bad == [2]
    assert np.array_equal(kc.view(np.uint16), k0.view(np.uint16))
    assert np.array_equal(vc.view(np.uint16), v0.view(np.uint16))


# ---------------------------------------------------------------------------
# planted mistakes: each must trip at least one pin
# ---------------------------------------------------------------------------

MUTATIONS = {
    "dropped_scale": ("z = scale * (K @ q[s, h]", "z = (K @ q[s, h]"),
    "wrong_gqa_mapping": ("g = kv_head_of(h, group)\n            K = gather_rows(k_cache, row, L, g)\n"
                          "            V = gather_rows(v_cache, row, L, g)\n            z = scale * (K @ q[s, h]",
                          "g = h % Hkv\n            K = gather_rows(k_cache, row, L, g)\n"
                          "            V = gather_rows(v_cache, row, L, g)\n            z = scale * (K @ q[s, h]"),
    "values_from_keys": ("V = gather_rows(v_cache, row, L, g)\n            z = scale",
                         "V = gather_rows(k_cache, row, L, g)\n            z = scale"),
    "row_index_off_by_one": ("cache[blocks, kv_head, i % bs, :]", "cache[blocks, kv_head, (i + 1) % bs, :]"),
    "block_index_from_offset": ("blocks = table_row[i // bs]", "blocks = table_row[i % table_row.shape[0]]"),
    "unnormalised_softmax": ("return e / e.sum(axis=-1, keepdims=True)", "return e"),
    "drops_newest_token": ("L = int(context_lens[s])\n        if L == 0:\n            continue\n        row = block_tables[s]\n        for h",
                           "L = int(context_lens[s]) - 1\n        if L <= 0:\n            continue\n        row = block_tables[s]\n        for h"),
    "kv_head_of_modulo": ("    return h // group", "    return h % group"),
    # decode_fast only: it scores a whole query group at once, so the softmax
    # axis matters there.
    "fast:softmax_over_whole_group": ("e = np.exp(z - z.max(axis=-1, keepdims=True))\n    return e / e.sum(axis=-1, keepdims=True)",
                                      "e = np.exp(z - z.max())\n    return e / e.sum()"),
    "fast:group_heads_from_modulo": ("heads = [h for h in range(H) if kv_head_of(h, group) == g]\n            K = gather_rows",
                                     "heads = [h for h in range(H) if h % Hkv == g]\n            K = gather_rows"),
    "fast:transposed_scores": ("Z = scale * (q[s, heads].astype(np.float64) @ K.T)",
                               "Z = scale * (q[s, heads].astype(np.float64) @ K.T)[:, ::-1]"),
}


def mutant_decode(name):
    old, new = MUTATIONS[name]
    src = inspect.getsource(OPA)
    assert src.count(old) == 1, f"mutation {name} does not apply"
    mod = types.ModuleType(f"oracle_mutant_{name.replace(':', '_')}")
    exec(compile(src.replace(old, new), f"<mutant {name}>", "exec"), mod.__dict__)
    return mod.decode_fast if name.startswith("fast:") else mod.decode


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(name):
    res = all_pins(mutant_decode(name))
    assert any(v is not True for v in res.values()), f"{name} passed every pin: {res}"
