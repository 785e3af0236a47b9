"""Pins of the oracle's multi-token (varlen, causal) attention (no GPU)."""

import inspect
import types

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from oracle import paged_attention as OPA
from paged_kv_decode_08_gb300 import workloads as W


def sdpa_causal(v: W.VarlenWorkload) -> np.ndarray:
    """torch SDPA in float64 on each sequence's contiguous rows, with an
    explicit mask: query t (at position prefix + t) sees keys 0..prefix+t."""
    w = v.base
    G = w.group
    out = np.zeros((v.total_q, w.num_heads, w.head_dim), np.float64)
    for s in range(w.num_seqs):
        a, b = int(v.cu_seqlens_q[s]), int(v.cu_seqlens_q[s + 1])
        if b == a:
            continue
        L = int(w.context_lens[s])
        K = torch.from_numpy(w.seq_k[s].astype(np.float64)).permute(1, 0, 2).repeat_interleave(G, 0)
        V = torch.from_numpy(w.seq_v[s].astype(np.float64)).permute(1, 0, 2).repeat_interleave(G, 0)
        q = torch.from_numpy(v.q[a:b].astype(np.float64)).permute(1, 0, 2)  # [H][n][D]
        pos = int(v.pos_offsets[s]) + torch.arange(b - a)
        mask = torch.arange(L)[None, :] <= pos[:, None]  # [n][L], True = attend
        o = F.scaled_dot_product_attention(q, K, V, attn_mask=mask, scale=w.scale)
        out[a:b] = o.permute(1, 0, 2).numpy()
    return out


CASES = [
    dict(seed=201, num_heads=8, num_kv_heads=2, head_dim=64, block_size=16,
         q_lens=[1, 4, 7, 2], prefix_lens=[0, 15, 33, 100]),
    dict(seed=202, num_heads=7, num_kv_heads=1, head_dim=128, block_size=32,
         q_lens=[3, 1, 8], prefix_lens=[29, 0, 64]),
]


def run(fn, v):
    kc, vc = W.host_pool(v.base)
    return fn(v.q, kc, vc, v.cu_seqlens_q, v.pos_offsets, v.base.block_tables, v.base.scale)


def pins(fn):
    res = {}
    for i, c in enumerate(CASES):
        v = W.varlen_random(**c)
        try:
            res[f"sdpa{i}"] = bool(np.allclose(run(fn, v), sdpa_causal(v), rtol=1e-10, atol=1e-12))
        except Exception as exc:
            res[f"sdpa{i}"] = f"raised {type(exc).__name__}"
    # the first query of a sequence with no prefix sees only itself
    v = W.varlen_random(203, 4, 2, 64, 16, [3, 2], [0, 0])
    try:
        got = run(fn, v)
        ok = True
        for s in range(2):
            i = int(v.cu_seqlens_q[s])
            for h in range(4):
                ok &= np.array_equal(got[i, h], v.base.seq_v[s][0, h // 2].astype(np.float64))
        res["first_token"] = bool(ok)
    except Exception as exc:
        res["first_token"] = f"raised {type(exc).__name__}"
    return res


def test_varlen_oracle_passes_its_pins():
    res = pins(oracle.varlen)
    assert all(v is True for v in res.values()), res


def test_varlen_fast_passes_the_same_pins():
    res = pins(oracle.varlen_fast)
    assert all(v is True for v in res.values()), res


def test_single_token_queries_are_decode():
    v = W.varlen_random(204, 8, 2, 64, 16, [1, 1, 1], [5, 0, 47])
    kc, vc = W.host_pool(v.base)
    a = oracle.varlen(v.q, kc, vc, v.cu_seqlens_q, v.pos_offsets, v.base.block_tables, v.base.scale)
    b = oracle.decode(v.q, kc, vc, v.base.block_tables, v.pos_offsets + 1, v.base.scale)
    assert np.allclose(a, b, rtol=1e-13, atol=1e-15)


def test_last_query_is_decode_over_the_full_context():
    v = W.varlen_random(205, 4, 4, 64, 32, [5, 2], [40, 7])
    kc, vc = W.host_pool(v.base)
    a = oracle.varlen(v.q, kc, vc, v.cu_seqlens_q, v.pos_offsets, v.base.block_tables, v.base.scale)
    last = v.cu_seqlens_q[1:] - 1
    b = oracle.decode(v.q[last], kc, vc, v.base.block_tables, v.base.context_lens, v.base.scale)
    assert np.allclose(a[last], b, rtol=1e-13, atol=1e-15)


def test_bad_inputs_are_rejected():
    v = W.varlen_random(206, 4, 2, 64, 16, [2, 2], [3, 3])
    kc, vc = W.host_pool(v.base)
    with pytest.raises(oracle.OracleInputError):
        oracle.varlen(v.q, kc, vc, np.array([0, 2, 5], np.int32), v.pos_offsets,
                      v.base.block_tables, v.base.scale)
    with pytest.raises(oracle.OracleInputError):
        oracle.varlen(v.q, kc, vc, v.cu_seqlens_q, v.pos_offsets + 100, v.base.block_tables,
                      v.base.scale)


LOOP = "for t in range(int(cu[s + 1] - cu[s])):\n            "
MUTATIONS = {
    "no_causal_mask": (LOOP + "L = int(pos_offsets[s]) + t + 1\n",
                       LOOP + "L = int(pos_offsets[s]) + int(cu[s + 1] - cu[s])\n"),
    "mask_off_by_one": (LOOP + "L = int(pos_offsets[s]) + t + 1\n",
                        LOOP + "L = int(pos_offsets[s]) + t + (t > 0)\n"),
    "wrong_query_row": ("i = int(cu[s]) + t\n            for h in range(H):",
                        "i = int(cu[s + 1]) - 1 - t\n            for h in range(H):"),
}


# varlen_fast only
FAST_MUTATIONS = {
    "fast:no_causal_mask": ("Z = scale * (q[i, heads].astype(np.float64) @ K[:L].T)\n                out[i, heads] = softmax(Z) @ V[:L]",
                            "Z = scale * (q[i, heads].astype(np.float64) @ K.T)\n                out[i, heads] = softmax(Z) @ V"),
    "fast:softmax_over_group": ("out[i, heads] = softmax(Z) @ V[:L]",
                                "out[i, heads] = (np.exp(Z - Z.max()) / np.exp(Z - Z.max()).sum()) @ V[:L]"),
    "fast:heads_by_modulo": ("heads = [h for h in range(H) if kv_head_of(h, group) == g]\n            for t in range(n):",
                             "heads = [h for h in range(H) if h % Hkv == g]\n            for t in range(n):"),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS) + sorted(FAST_MUTATIONS))
def test_planted_mistake_is_caught(name):
    old, new = MUTATIONS[name] if name in MUTATIONS else FAST_MUTATIONS[name]
    src = inspect.getsource(OPA)
    assert src.count(old) == 1, name
    mod = types.ModuleType("varlen_mutant")
    exec(compile(src.replace(old, new), "<mutant>", "exec"), mod.__dict__)
    res = pins(mod.varlen_fast if name.startswith("fast:") else mod.varlen)
    assert any(v is not True for v in res.values()), (name, res)
