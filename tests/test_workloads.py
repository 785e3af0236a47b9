"""The seeded input generator: determinism and the structure of each workload."""

import numpy as np
import pytest

import oracle
from paged_kv_decode_08_gb300 import workloads as W


def _digest(w):
    import hashlib

    h = hashlib.sha256()
    for a in [w.context_lens, w.block_tables, w.q] + w.seq_k + w.seq_v:
        h.update(np.ascontiguousarray(a).tobytes())
    return h.hexdigest()


def test_same_seed_same_bytes():
    assert _digest(W.tiny()) == _digest(W.tiny())
    a = W.small_random(3, 2, 4, 2, 64, 16, [5, 40])
    b = W.small_random(3, 2, 4, 2, 64, 16, [5, 40])
    assert _digest(a) == _digest(b)


def _check_structure(w):
    B, mbps = w.block_tables.shape
    assert B == w.num_seqs and mbps == w.max_blocks_per_seq
    used = np.concatenate([w.blocks_of(s) for s in range(B)])
    assert len(np.unique(used)) == len(used), "a block is shared between positions"
    assert used.min() >= 0 and used.max() < w.num_blocks
    assert w.poison_block not in set(used.tolist())
    for s in range(B):
        n = len(w.blocks_of(s))
        assert np.all(w.block_tables[s, n:] == w.poison_block)
        assert w.seq_k[s].shape == (int(w.context_lens[s]), w.num_kv_heads, w.head_dim)
    assert w.q.shape == (w.num_seqs, w.num_heads, w.head_dim)
    assert w.num_heads % w.num_kv_heads == 0


def test_tiny_matches_its_description():
    w = W.tiny()
    _check_structure(w)
    assert list(w.context_lens) == [17, 40]
    assert (w.num_heads, w.num_kv_heads, w.head_dim, w.block_size, w.num_blocks) == (4, 2, 64, 16, 8)
    assert w.scale == 1 / 8
    k_new, v_new, slots = w.last_token_append()
    # positions 16 and 39
    assert slots[0] == w.block_tables[0, 1] * 16 + 0
    assert slots[1] == w.block_tables[1, 2] * 16 + 7


def test_llama8b_structure():
    w = W.llama8b()
    _check_structure(w)
    assert w.context_lens.min() >= 512 and w.context_lens.max() <= 2048
    assert (w.num_seqs, w.num_heads, w.num_kv_heads, w.head_dim, w.block_size) == (32, 32, 8, 128, 16)


def test_ragged_lengths():
    rng = W._rng(W.BASE_SEED + 3)
    lens = W.ragged_lens(rng)
    assert lens.min() == 1 and lens.max() <= 16384
    assert (lens == 1).sum() >= 8
    assert 600 < np.median(lens) < 1700


def test_loop_schedule_is_consistent():
    loop = W.AppendDecodeLoop(steps=6, num_seqs=8, max_len=40, min_len=1, num_blocks=64,
                              max_blocks_per_seq=4, num_pad=2)
    seen = set()
    for t in range(loop.steps):
        st = loop.step(t)
        real = st.slot_mapping >= 0
        assert real.sum() == loop.num_seqs and (~real).sum() == loop.num_pad
        assert np.all(np.isnan(st.k_new[~real].astype(np.float32)))
        for s, slot in enumerate(st.slot_mapping[real]):
            pos = int(st.context_lens[s]) - 1
            assert slot == st.block_tables[s, pos // 16] * 16 + pos % 16
            assert slot not in seen
            seen.add(int(slot))
    # no block is owned by two sequences
    last = loop.tables[-1]
    owned = np.concatenate([last[s, : -(-int(loop.end_lens[s]) // 16)] for s in range(loop.num_seqs)])
    assert len(np.unique(owned)) == len(owned)
    assert loop.poison_block not in set(owned.tolist())


def test_vllm_layout_pools_hold_the_blocked_pools_values():
    """The generator's vLLM-layout pools, read back by the oracle's adapter,
    are the blocked pools bit for bit (NaN poison included)."""
    import oracle

    for w in (W.make("tiny"), W.small_random(7, 3, 8, 2, 128, 32, [1, 40, 65])):
        kb, vb = W.host_pool(w, fill=np.nan)
        kv, vv = W.host_pool_vllm(w, fill=np.nan)
        assert kv.shape == (w.num_blocks, w.num_kv_heads, w.head_dim // 8, w.block_size, 8)
        assert vv.shape == (w.num_blocks, w.num_kv_heads, w.head_dim, w.block_size)
        k2, v2 = oracle.blocked_from_vllm_layout(kv, vv)
        assert np.array_equal(k2.view(np.uint16), kb.view(np.uint16))
        assert np.array_equal(v2.view(np.uint16), vb.view(np.uint16))


def test_loop_allocator_reports_exhaustion_and_overflow():
    """The loop harness's block allocator fails loudly, never silently: a
    pool too small for the start lengths or for a later step, and a sequence
    growing past its table row."""
    kw = dict(num_seqs=2, num_heads=2, head_dim=64, block_size=16, min_len=32, max_len=32)
    with pytest.raises(RuntimeError, match="free list exhausted"):
        W.AppendDecodeLoop(steps=1, num_blocks=4, max_blocks_per_seq=4, **kw)  # needs 4 + poison
    with pytest.raises(RuntimeError, match="free list exhausted"):
        W.AppendDecodeLoop(steps=1, num_blocks=5, max_blocks_per_seq=4, **kw)  # step 0 needs a 6th
    with pytest.raises(ValueError, match="max_blocks_per_seq"):
        W.AppendDecodeLoop(steps=1, num_blocks=50, max_blocks_per_seq=2, **kw)
    ok = W.AppendDecodeLoop(steps=1, num_blocks=7, max_blocks_per_seq=4, **kw)  # 2 + 2 + 2 + poison
    assert ok.end_lens.tolist() == [33, 33]


def test_compact_pool_keeps_the_attention():
    """The compact pool renumbers the used blocks (and the poison block) and
    changes nothing the oracle computes."""
    w = W.small_random(5, num_seqs=5, num_heads=4, num_kv_heads=2, head_dim=64, block_size=16,
                       lens=[40, 1, 77, 16, 130], num_blocks=500)
    c = W.compact_pool(w)
    assert c.num_blocks < w.num_blocks
    assert len(np.unique(c.block_tables)) == len(np.unique(w.block_tables))
    kc, vc = W.host_pool(w)
    kc2, vc2 = W.host_pool(c)
    a = oracle.decode(w.q, kc, vc, w.block_tables, w.context_lens, w.scale)
    b = oracle.decode(c.q, kc2, vc2, c.block_tables, c.context_lens, c.scale)
    assert np.array_equal(a, b)
