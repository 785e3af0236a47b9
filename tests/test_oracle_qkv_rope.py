"""Pins of the oracle's fused QKV split + per-head RMS norm + rotary
embedding + paged append (no GPU).  What pins it: a hand-derived example
(tests/golden/qkv_rope_hand_example.json), the identity at angle 0, rotation
preserving each pair's norm, q.k depending only on the distance of the two
positions, RMS 1 after the norm and its scale invariance, and the layout
found by search with distinct values.  Each planted mistake below breaks one
of them."""

import inspect
import json
import math
import os
import types

import numpy as np
import pytest

from oracle import qkv_norm_rope as Q

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "qkv_rope_hand_example.json")


def tables(max_pos, D, base=10000.0):
    """cos/sin of the standard rotary angles p * base^(-2i/D) (an input here)."""
    inv = base ** (-np.arange(D // 2) * 2.0 / D)
    ang = np.arange(max_pos)[:, None] * inv[None, :]
    return np.cos(ang), np.sin(ang)


def one_seq_case(rng, H, Hkv, D, bs, T, pos0, NB=None, norm=True, angles=True):
    width = (H + 2 * Hkv) * D
    qkv = rng.standard_normal((T, width)).astype(np.float16)
    n_blocks = -(-(pos0 + T) // bs)
    NB = NB or n_blocks + 2
    perm = rng.permutation(NB).astype(np.int32)
    bt = perm[:n_blocks][None, :]
    cos, sin = tables(pos0 + T, D) if angles else (np.ones((pos0 + T, D // 2)),
                                                  np.zeros((pos0 + T, D // 2)))
    qw = rng.uniform(0.5, 1.5, D).astype(np.float16) if norm else None
    kw = rng.uniform(0.5, 1.5, D).astype(np.float16) if norm else None
    kc = np.zeros((NB, Hkv, bs, D), np.float16)
    vc = np.zeros_like(kc)
    cu = np.array([0, T], np.int32)
    pos = np.array([pos0], np.int32)
    return dict(qkv=qkv, q_norm_w=qw, k_norm_w=kw, cos=cos, sin=sin, k_cache=kc, v_cache=vc,
                cu_seqlens_q=cu, pos_offsets=pos, block_tables=bt, num_heads=H,
                num_kv_heads=Hkv, eps=1e-6)


def golden_ok(mod):
    g = json.load(open(GOLDEN))
    qkv = np.array([g["qkv"]], np.float16)
    kc = np.zeros((2, 1, 2, 4), np.float16)
    vc = np.zeros_like(kc)
    q_out, k_rows = mod.qkv_norm_rope_append(
        qkv, None, np.ones(4, np.float16), np.array(g["cos"]), np.array(g["sin"]), kc, vc,
        np.array([0, 1], np.int32), np.array([g["position"]], np.int32),
        np.array([[1]], np.int32), 1, 1, 0.0)
    return (np.allclose(q_out[0, 0], g["q_out"], atol=1e-12)
            and np.allclose(k_rows[0, 0], g["k"], atol=1e-12)
            and np.array_equal(vc[1, 0, 1].astype(np.float64), g["v"]))


def identity_ok(mod):
    """Angle 0 and no norm: every row is copied unchanged to where it belongs."""
    rng = np.random.default_rng(1)
    H, Hkv, D, bs, T, pos0 = 4, 2, 8, 4, 6, 3
    c = one_seq_case(rng, H, Hkv, D, bs, T, pos0, norm=False, angles=False)
    # distinct values so a misplaced element cannot match by chance
    n = c["qkv"].size
    c["qkv"] = (np.arange(n, dtype=np.float64) % 1900 + 1).reshape(c["qkv"].shape).astype(np.float16)
    q_out, _ = mod.qkv_norm_rope_append(**c)
    x = c["qkv"].astype(np.float64).reshape(T, H + 2 * Hkv, D)
    if not np.array_equal(q_out, x[:, :H]):
        return False
    for t in range(T):
        p = pos0 + t
        blk = int(c["block_tables"][0][p // bs])
        if not (np.array_equal(c["k_cache"][blk, :, p % bs].astype(np.float64), x[t, H:H + Hkv])
                and np.array_equal(c["v_cache"][blk, :, p % bs].astype(np.float64), x[t, H + Hkv:])):
            return False
    return True


def rotation_ok(mod):
    """A rotation keeps each pair's norm, and q.k after rotation depends only
    on the distance between the two positions."""
    rng = np.random.default_rng(2)
    D = 16
    cos, sin = tables(64, D)
    x = rng.standard_normal(D)
    y = mod.rotate(x, cos[37], sin[37])
    pair = lambda v: v[: D // 2] ** 2 + v[D // 2:] ** 2  # noqa: E731
    if not np.allclose(pair(y), pair(x), rtol=1e-12, atol=1e-12):
        return False
    q, k = rng.standard_normal(D), rng.standard_normal(D)
    a = mod.rotate(q, cos[20], sin[20]) @ mod.rotate(k, cos[7], sin[7])
    b = mod.rotate(q, cos[33], sin[33]) @ mod.rotate(k, cos[20], sin[20])
    return bool(abs(a - b) < 1e-10 and abs(a - q @ k) > 1e-6)


def norm_ok(mod):
    rng = np.random.default_rng(3)
    x = rng.standard_normal(128) * 3.0
    y = mod.rms_norm(x, np.ones(128), 0.0)
    z = mod.rms_norm(7.5 * x, np.ones(128), 0.0)
    w = rng.uniform(0.5, 2.0, 128)
    yw = mod.rms_norm(x, w, 0.0)
    return bool(abs(np.mean(y * y) - 1.0) < 1e-12 and np.allclose(y, z, atol=1e-12)
                and np.allclose(yw / w, y, atol=1e-12))


def full_ok(mod):
    """Several tokens, norms and angles: each output equals the composition
    written out directly for one element pair."""
    rng = np.random.default_rng(4)
    H, Hkv, D, bs, T, pos0 = 4, 2, 16, 8, 5, 11
    c = one_seq_case(rng, H, Hkv, D, bs, T, pos0)
    q_out, k_rows = mod.qkv_norm_rope_append(**c)
    t, h, i = 3, 2, 5
    p = pos0 + t
    x = c["qkv"][t].astype(np.float64).reshape(H + 2 * Hkv, D)[h]
    r = math.sqrt(np.mean(x * x) + c["eps"])
    w = c["q_norm_w"].astype(np.float64)
    a, b = x[i] / r * w[i], x[i + D // 2] / r * w[i + D // 2]
    ang_c, ang_s = c["cos"][p][i], c["sin"][p][i]
    return bool(np.isclose(q_out[t, h, i], a * ang_c - b * ang_s, atol=1e-12)
                and np.isclose(q_out[t, h, i + D // 2], b * ang_c + a * ang_s, atol=1e-12))


def all_pins(mod):
    out = {}
    for name, fn in (("golden", golden_ok), ("identity", identity_ok), ("rotation", rotation_ok),
                     ("norm", norm_ok), ("full", full_ok)):
        try:
            out[name] = fn(mod)
        except Exception as exc:  # a mutant may also fail by raising
            out[name] = f"raised {type(exc).__name__}"
    return out


def test_qkv_rope_oracle_pins():
    res = all_pins(Q)
    assert all(v is True for v in res.values()), res


def test_qkv_rope_rejects_bad_inputs():
    rng = np.random.default_rng(5)
    c = one_seq_case(rng, 2, 1, 8, 4, 3, 0)
    c["pos_offsets"] = np.array([100], np.int32)
    with pytest.raises(Q.QkvInputError):
        Q.qkv_norm_rope_append(**c)
    c = one_seq_case(rng, 2, 1, 8, 4, 3, 0)
    c["block_tables"] = c["block_tables"] + 1000
    with pytest.raises(Q.QkvInputError):
        Q.qkv_norm_rope_append(**c)


MUTATIONS = {
    "rotation_sign": ("np.concatenate([a * c - b * s, b * c + a * s], axis=-1)",
                      "np.concatenate([a * c + b * s, b * c - a * s], axis=-1)"),
    "adjacent_pairs": ("a, b = x[..., :half], x[..., half:]", "a, b = x[..., 0::2], x[..., 1::2]"),
    "norm_without_square_root": ("r = np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)",
                                 "r = np.mean(x * x, axis=-1, keepdims=True) + eps"),
    "keys_from_value_heads": ("y = x[H + g] if k_norm_w is None", "y = x[H + Hkv + g] if k_norm_w is None"),
    "values_normalised": ("v_cache[blk, g, p % bs, :] = x[H + Hkv + g]",
                          "v_cache[blk, g, p % bs, :] = rms_norm(x[H + Hkv + g], None, eps)"),
    "position_off_by_one": ("p = int(pos_offsets[s]) + t\n", "p = int(pos_offsets[s]) + t + 1\n"),
    "query_weight_from_keys": ("rms_norm(x[h], q_norm_w, eps)", "rms_norm(x[h], k_norm_w, eps)"),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(name):
    old, new = MUTATIONS[name]
    src = inspect.getsource(Q)
    assert src.count(old) == 1, name
    mod = types.ModuleType(f"qkv_mutant_{name}")
    exec(compile(src.replace(old, new), f"<mutant {name}>", "exec"), mod.__dict__)
    res = all_pins(mod)
    assert any(v is not True for v in res.values()), (name, res)
