"""GPU parity: the CUDA path through the C ABI against the CPU oracle.

Append is compared bit for bit; attention within |gpu-ref| <= 2e-3 + 1e-2|ref|
(see tests/tolerance.py).  Inputs come from the seeded generator; unused pool
blocks, rows past a sequence's length and table entries past its blocks all
hold or point at NaN, so a stray read shows up as NaN.
"""

import dataclasses

import numpy as np
import pytest

import oracle
from paged_kv_decode_08_gb300 import workloads as W
from tests.tolerance import assert_attention_close, assert_bits_equal

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def pk(cuda_device):
    from paged_kv_decode_08_gb300 import pagedkv

    pagedkv.pkv_read_device_status()  # start from a clean status word
    return pagedkv


@pytest.fixture(params=[0, 1], ids=["mma_sync", "tcgen05"])
def varlen_path(request, pk):
    """The kernel varlen attention runs for chunks of more than 8 (query,
    head) columns at head_dim 128 (pkv_set_varlen_tensor_path): the
    mma.sync kernel or the tcgen05 one; other shapes run the same kernel
    under both."""
    prev = pk.pkv_set_varlen_tensor_path(request.param)
    yield request.param
    pk.pkv_set_varlen_tensor_path(prev)


_CACHE = {}


def workload(name):
    if name not in _CACHE:
        w = W.make(name)
        kc, vc = W.host_pool(w)
        ref = oracle.decode_fast(w.q, kc, vc, w.block_tables, w.context_lens, w.scale)
        del kc, vc
        _CACHE[name] = (w, ref)
    return _CACHE[name]


def to_np(t):
    return t.float().cpu().numpy().astype(np.float64)


def appended_device(pk, w, dev):
    """Device pools without each sequence's newest token, then pkv_append it."""
    d = W.to_device(w, dev, upto_last=True)
    k_new, v_new, slots = w.last_token_append()
    pk.pkv_append(torch.from_numpy(k_new).to(dev), torch.from_numpy(v_new).to(dev),
                  torch.from_numpy(slots).to(dev), d["k_cache"], d["v_cache"])
    return d


def decode_all(pk, w, d, splits):
    """{label: output} for single pass and the requested split counts."""
    outs = {"single": pk.pkv_decode(d["q"], d["k_cache"], d["v_cache"], d["block_tables"],
                                    d["context_lens"], w.scale)}
    for S in splits:
        outs[f"splitk{S}"] = pk.pkv_decode_splitk(d["q"], d["k_cache"], d["v_cache"],
                                                  d["block_tables"], d["context_lens"], w.scale,
                                                  num_splits=S)
    torch.cuda.synchronize()
    return {k: to_np(v) for k, v in outs.items()}


# ---------------------------------------------------------------------------
# append
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("name", ["tiny", "llama8b", "long", "ragged"])
def test_append_is_bit_exact(pk, cuda_device, name):
    w, _ = workload(name)
    d = appended_device(pk, w, cuda_device)
    ids, kb, vb = W.compact_blocks(w, upto_last=False)
    idx = torch.from_numpy(ids).to(cuda_device)
    got_k = d["k_cache"].index_select(0, idx).cpu().numpy()
    got_v = d["v_cache"].index_select(0, idx).cpu().numpy()
    # expected: the oracle's scatter applied to the host pool without the token
    hk, hv = W.host_pool(w, upto_last=True)
    k_new, v_new, slots = w.last_token_append()
    assert oracle.append(k_new, v_new, slots, hk, hv) == []
    assert_bits_equal(got_k, hk[ids], f"{name} K")
    assert_bits_equal(got_v, hv[ids], f"{name} V")
    assert pk.pkv_read_device_status() == 0


def test_append_skips_padding_and_flags_bad_slots(pk, cuda_device):
    w, _ = workload("tiny")
    d = W.to_device(w, cuda_device)
    before_k = d["k_cache"].clone()
    before_v = d["v_cache"].clone()
    T = 3
    k = torch.ones((T, w.num_kv_heads, w.head_dim), dtype=torch.float16, device=cuda_device)
    slots = torch.tensor([-1, -5, w.num_blocks * w.block_size], dtype=torch.int32,
                         device=cuda_device)
    pk.pkv_append(k, k, slots, d["k_cache"], d["v_cache"])
    flags = pk.pkv_read_device_status()
    assert flags & pk.PKV_DEV_BAD_SLOT
    assert torch.equal(d["k_cache"].view(torch.int16), before_k.view(torch.int16))
    assert torch.equal(d["v_cache"].view(torch.int16), before_v.view(torch.int16))


# ---------------------------------------------------------------------------
# decode parity on the workloads
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("name,splits", [
    ("tiny", [0, 2, 3]),
    ("llama8b", [0, 2, 4, 16]),
    ("long", [0, 4, 16, 64]),
    ("ragged", [0, 3, 8, 32]),
])
def test_decode_matches_oracle(pk, cuda_device, name, splits):
    w, ref = workload(name)
    d = appended_device(pk, w, cuda_device)
    outs = decode_all(pk, w, d, splits)
    for label, got in outs.items():
        assert_attention_close(got, ref, f"{name}/{label}")
    assert pk.pkv_read_device_status() == 0


@pytest.mark.parametrize("name", ["llama8b", "long"])
def test_overprovisioned_tables_split_the_real_contexts(pk, cuda_device, name):
    """Tables four times wider than the longest context (a server sizes them
    for the model's maximum context): the split chunks are cut from the real
    longest context, so with S forced to 4 the last split of the longest
    sequence holds work (its partial max is finite, not the -inf of an empty
    split), and every split count matches the oracle."""
    w0, ref = workload(name)
    w = W.widen_tables(w0, 4)
    d = appended_device(pk, w, cuda_device)
    S = 4
    S_run, need = pk.pkv_decode_splitk_plan(w.num_seqs, w.num_heads, w.num_kv_heads, w.head_dim,
                                            w.max_blocks_per_seq, w.block_size, S)
    assert S_run == S and need == pk.pkv_splitk_scratch_bytes(w.num_seqs, w.num_heads,
                                                              w.head_dim, S)
    scratch = torch.empty(need, dtype=torch.uint8, device=cuda_device)
    out = pk.pkv_decode_splitk(d["q"], d["k_cache"], d["v_cache"], d["block_tables"],
                               d["context_lens"], w.scale, num_splits=S, scratch=scratch)
    torch.cuda.synchronize()
    assert_attention_close(to_np(out), ref, f"{name} x4 tables, S=4")
    # scratch layout: a 256-byte header, f32 part_out [B][H][S][D], then
    # part_m [B][H][S] (each 256-byte aligned)
    a256 = lambda x: (x + 255) // 256 * 256  # noqa: E731
    rows = w.num_seqs * w.num_heads * S
    part_m = scratch[256 + a256(rows * w.head_dim * 4):][:rows * 4].view(torch.float32)
    part_m = part_m.view(w.num_seqs, w.num_heads, S).cpu().numpy()
    longest = int(np.argmax(w.context_lens))
    assert np.all(np.isfinite(part_m[longest, :, S - 1])), "last split of the longest sequence"
    for label, got in decode_all(pk, w, d, [0, 16]).items():
        assert_attention_close(got, ref, f"{name} x4 tables, {label}")
    assert pk.pkv_read_device_status() == 0


def test_overprovisioned_tables_varlen_splitk(pk, cuda_device, varlen_path):
    """Long speculative verification with tables four times wider than the
    contexts: the varlen split chunks are cut from the real longest context."""
    v0 = W.spec_verify_long()
    kc, vc = W.host_pool(v0.base)
    ref = oracle.varlen_fast(v0.q, kc, vc, v0.cu_seqlens_q, v0.pos_offsets, v0.base.block_tables,
                             v0.base.scale)
    del kc, vc
    v = dataclasses.replace(v0, base=W.widen_tables(v0.base, 4))
    d = varlen_device(v, cuda_device)
    for S_req in (0, 8):
        got = pk.pkv_varlen_attention_splitk(d["q"], d["k_cache"], d["v_cache"], d["cu"],
                                             d["pos"], d["block_tables"], v.base.scale,
                                             max_q_len=v.max_q_len, num_splits=S_req)
        torch.cuda.synchronize()
        assert_attention_close(to_np(got), ref, f"x4 tables, varlen S={S_req}")
    assert pk.pkv_read_device_status() == 0


def test_heuristic_split_counts(pk, cuda_device):
    sms = torch.cuda.get_device_properties(cuda_device).multi_processor_count
    for name in ["tiny", "llama8b", "long", "ragged"]:
        w, _ = workload(name)
        S = pk.pkv_pick_num_splits(w.num_seqs, w.num_kv_heads,
                                   w.max_blocks_per_seq * w.block_size, w.block_size, sms)
        assert 1 <= S <= 64
    w, _ = workload("long")
    assert pk.pkv_pick_num_splits(4, 8, 131072, 16, sms) > 1


def test_context_len_one_is_exact(pk, cuda_device):
    """One token: its softmax weight is exactly 1, so the f16 output is that V
    row bit for bit, in the single-pass and split-K kernels alike."""
    w = W.small_random(41, num_seqs=6, num_heads=14, num_kv_heads=2, head_dim=128,
                       block_size=32, lens=[1, 1, 33, 1, 64, 1])
    d = appended_device(pk, w, cuda_device)
    for S in (1, 2, 3):
        out = pk.pkv_decode_splitk(d["q"], d["k_cache"], d["v_cache"], d["block_tables"],
                                   d["context_lens"], w.scale, num_splits=S).cpu().numpy()
        for s in range(w.num_seqs):
            if int(w.context_lens[s]) != 1:
                continue
            for h in range(w.num_heads):
                exp = w.seq_v[s][0, h // w.group]
                assert np.array_equal(out[s, h].view(np.uint16), exp.view(np.uint16)), (S, s, h)


@pytest.mark.parametrize("D,bs,G", [(64, 16, 1), (64, 32, 3), (128, 16, 5), (128, 32, 8),
                                    (64, 16, 8), (128, 16, 2)])
def test_ragged_small_shapes(pk, cuda_device, D, bs, G):
    lens = [1, bs - 1, bs, bs + 1, 5 * bs + 3, 37, 300]
    w = W.small_random(1000 + D + bs + G, num_seqs=len(lens), num_heads=2 * G, num_kv_heads=2,
                       head_dim=D, block_size=bs, lens=lens)
    kc, vc = W.host_pool(w)
    ref = oracle.decode(w.q, kc, vc, w.block_tables, w.context_lens, w.scale)
    d = appended_device(pk, w, cuda_device)
    for label, got in decode_all(pk, w, d, [0, 2, 5, 128]).items():
        assert_attention_close(got, ref, f"D{D} bs{bs} G{G} {label}")


def test_empty_context_gives_zeros(pk, cuda_device):
    w = W.small_random(51, num_seqs=3, num_heads=4, num_kv_heads=2, head_dim=64, block_size=16,
                       lens=[20, 1, 40])
    kc, vc = W.host_pool(w)
    d = W.to_device(w, cuda_device)
    lens = w.context_lens.copy()
    lens[1] = 0
    d["context_lens"] = torch.from_numpy(lens).to(cuda_device)
    ref = oracle.decode(w.q, kc, vc, w.block_tables, lens, w.scale)
    for label, got in decode_all(pk, w, d, [2, 3]).items():
        assert np.all(got[1] == 0.0), label
        assert_attention_close(got, ref, label)


def test_scale_zero_gives_mean_of_v(pk, cuda_device):
    w = W.small_random(61, num_seqs=2, num_heads=8, num_kv_heads=2, head_dim=128, block_size=16,
                       lens=[100, 17])
    d = W.to_device(w, cuda_device)
    got = to_np(pk.pkv_decode(d["q"], d["k_cache"], d["v_cache"], d["block_tables"],
                              d["context_lens"], 0.0))
    for s in range(2):
        mean = w.seq_v[s].astype(np.float64).mean(axis=0)
        for h in range(8):
            assert_attention_close(got[s, h], mean[h // 4], f"seq {s} head {h}")


# ---------------------------------------------------------------------------
# bad device data is skipped and flagged, never dereferenced
# ---------------------------------------------------------------------------

def test_bad_block_id_is_skipped_and_flagged(pk, cuda_device):
    w = W.small_random(71, num_seqs=2, num_heads=4, num_kv_heads=2, head_dim=64, block_size=16,
                       lens=[48, 40])
    kc, vc = W.host_pool(w)
    ref = oracle.decode(w.q, kc, vc, w.block_tables, w.context_lens, w.scale)
    d = W.to_device(w, cuda_device)
    tables = w.block_tables.copy()
    tables[0, 1] = w.num_blocks + 5  # out of range: tokens 16..31 of sequence 0 are skipped
    d["block_tables"] = torch.from_numpy(tables).to(cuda_device)
    for S in (1, 3, 2):
        out = to_np(pk.pkv_decode_splitk(d["q"], d["k_cache"], d["v_cache"], d["block_tables"],
                                         d["context_lens"], w.scale, num_splits=S))
        assert pk.pkv_read_device_status() & pk.PKV_DEV_BAD_BLOCK_ID
        assert np.all(np.isfinite(out))
        assert_attention_close(out[1], ref[1], "untouched sequence")
        # sequence 0 equals attention over its remaining 32 tokens
        keep = [i for i in range(48) if not 16 <= i < 32]
        K = w.seq_k[0][keep].astype(np.float64)
        V = w.seq_v[0][keep].astype(np.float64)
        for h in range(4):
            z = w.scale * K[:, h // 2] @ w.q[0, h].astype(np.float64)
            p = np.exp(z - z.max())
            p /= p.sum()
            assert_attention_close(out[0, h], p @ V[:, h // 2], f"S={S} head {h}")


def test_context_len_above_capacity_is_clamped_and_flagged(pk, cuda_device):
    w = W.small_random(81, num_seqs=2, num_heads=2, num_kv_heads=1, head_dim=64, block_size=16,
                       lens=[32, 10])
    kc, vc = W.host_pool(w)
    ref = oracle.decode(w.q, kc, vc, w.block_tables, w.context_lens, w.scale)
    d = W.to_device(w, cuda_device)
    lens = w.context_lens.copy()
    lens[0] = 10 ** 6  # capacity is 2 blocks * 16 = 32 tokens, the real length
    d["context_lens"] = torch.from_numpy(lens).to(cuda_device)
    out = to_np(pk.pkv_decode(d["q"], d["k_cache"], d["v_cache"], d["block_tables"],
                              d["context_lens"], w.scale))
    assert pk.pkv_read_device_status() & pk.PKV_DEV_BAD_CONTEXT_LEN
    assert_attention_close(out, ref, "clamped")


# ---------------------------------------------------------------------------
# the append+decode loop (128 steps on one stream)
# ---------------------------------------------------------------------------

def test_append_decode_loop(pk, cuda_device):
    loop = W.AppendDecodeLoop()
    w0 = loop.initial_workload()
    d = W.to_device(w0, cuda_device)
    kc, vc = d["k_cache"], d["v_cache"]
    hk, hv = W.host_pool(w0, fill=np.nan)  # unused blocks are NaN on the device too
    sample = {0, 63, 127} | set(int(x) for x in np.random.default_rng(5).choice(128, 3, False))
    stream = torch.cuda.current_stream()
    outs = {}
    for t in range(loop.steps):
        st = loop.step(t)
        k_new = torch.from_numpy(st.k_new).to(cuda_device)
        v_new = torch.from_numpy(st.v_new).to(cuda_device)
        slots = torch.from_numpy(st.slot_mapping).to(cuda_device)
        q = torch.from_numpy(st.q).to(cuda_device)
        bt = torch.from_numpy(st.block_tables).to(cuda_device)
        cl = torch.from_numpy(st.context_lens).to(cuda_device)
        pk.pkv_append(k_new, v_new, slots, kc, vc, stream=stream)
        out = pk.pkv_decode_splitk(q, kc, vc, bt, cl, loop.scale, stream=stream)
        assert oracle.append(st.k_new, st.v_new, st.slot_mapping, hk, hv) == []
        if t in sample:
            single = pk.pkv_decode(q, kc, vc, bt, cl, loop.scale, stream=stream)
            ref = oracle.decode_fast(st.q, hk, hv, st.block_tables, st.context_lens, loop.scale)
            outs[t] = (to_np(out), to_np(single), ref)
    for t, (split, single, ref) in sorted(outs.items()):
        assert_attention_close(split, ref, f"step {t} split-K")
        assert_attention_close(single, ref, f"step {t} single pass")
    owned = np.unique(loop.tables[-1][loop.tables[-1] != loop.poison_block])
    idx = torch.from_numpy(owned.astype(np.int64)).to(cuda_device)
    assert_bits_equal(kc.index_select(0, idx).cpu().numpy(), hk[owned], "K pool after 128 steps")
    assert_bits_equal(vc.index_select(0, idx).cpu().numpy(), hv[owned], "V pool after 128 steps")
    assert pk.pkv_read_device_status() == 0


def test_splitk_on_many_short_and_empty_sequences(pk, cuda_device):
    """Hundreds of sequences of 0-70 tokens: most fit one chunk (phase 1
    writes their output), a few span several, and empty ones must come out as
    zeros from the combine."""
    rng = np.random.default_rng(77)
    lens = [int(x) for x in rng.integers(0, 70, size=300)]
    lens[:5] = [0, 1, 0, 70, 2]
    w = W.small_random(1077, num_seqs=len(lens), num_heads=8, num_kv_heads=2, head_dim=64,
                       block_size=16, lens=[max(L, 1) for L in lens])
    kc, vc = W.host_pool(w)
    real = np.array(lens, np.int32)
    ref = oracle.decode(w.q, kc, vc, w.block_tables, real, w.scale)
    d = W.to_device(w, cuda_device)
    d["context_lens"] = torch.from_numpy(real).to(cuda_device)
    for S in (0, 2, 5):
        out = torch.full_like(d["q"], float("nan"))
        got = to_np(pk.pkv_decode_splitk(d["q"], d["k_cache"], d["v_cache"], d["block_tables"],
                                         d["context_lens"], w.scale, num_splits=S, out=out))
        assert_attention_close(got, ref, f"many short, S={S}")
        assert np.all(got[real == 0] == 0.0)
    assert pk.pkv_read_device_status() == 0


def test_splitk_with_every_length_zero(pk, cuda_device):
    w = W.small_random(1088, num_seqs=3, num_heads=4, num_kv_heads=2, head_dim=128,
                       block_size=32, lens=[5, 6, 7])
    d = W.to_device(w, cuda_device)
    d["context_lens"] = torch.zeros(3, dtype=torch.int32, device=cuda_device)
    for S in (1, 2):
        out = torch.full_like(d["q"], float("nan"))
        pk.pkv_decode_splitk(d["q"], d["k_cache"], d["v_cache"], d["block_tables"],
                             d["context_lens"], w.scale, num_splits=S, out=out)
        assert torch.count_nonzero(out).item() == 0


def test_host_resident_inputs_and_output(pk, cuda_device):
    """q, the new rows, slots, tables, lengths and out in page-locked host
    memory, passed straight to the C ABI (the kernels read and write them
    over the host link; the pools stay on the device): the same result, bit
    for bit, as with every buffer on the device."""
    w, ref = workload("llama8b")
    k_new, v_new, slots = w.last_token_append()
    host = {name: torch.from_numpy(np.ascontiguousarray(a)).pin_memory()
            for name, a in (("q", w.q), ("k", k_new), ("v", v_new), ("slots", slots),
                            ("bt", w.block_tables), ("cl", w.context_lens))}
    for S in (1, 4):
        d = W.to_device(w, cuda_device, upto_last=True)
        dev = {name: t.to(cuda_device) for name, t in host.items()}
        scratch = pk.alloc_scratch(dev["q"], d["k_cache"], dev["bt"], S)
        out_dev = pk.pkv_append_decode(dev["k"], dev["v"], dev["slots"], d["k_cache"],
                                       d["v_cache"], dev["q"], dev["bt"], dev["cl"], w.scale,
                                       num_splits=S, scratch=scratch)
        d2 = W.to_device(w, cuda_device, upto_last=True)
        out_host = torch.full(tuple(w.q.shape), float("nan"), dtype=torch.float16).pin_memory()
        status = pk.lib.pkv_append_decode(
            host["k"].data_ptr(), host["v"].data_ptr(), host["slots"].data_ptr(),
            d2["k_cache"].data_ptr(), d2["v_cache"].data_ptr(), host["q"].data_ptr(),
            host["bt"].data_ptr(), host["cl"].data_ptr(), w.num_seqs, w.max_blocks_per_seq,
            w.num_blocks, float(w.scale), w.num_heads, w.num_kv_heads, w.head_dim, w.block_size,
            out_host.data_ptr(), S, scratch.data_ptr(), scratch.numel(),
            torch.cuda.current_stream().cuda_stream)
        assert status == pk.PKV_OK, pk.last_error()
        torch.cuda.synchronize()
        assert_bits_equal(out_host.numpy(), out_dev.cpu().numpy(), f"host-resident, S={S}")
        assert_attention_close(out_host.float().numpy().astype(np.float64), ref, f"S={S}")
        assert torch.equal(d2["k_cache"].view(torch.int16), d["k_cache"].view(torch.int16))
    assert pk.pkv_read_device_status() == 0


# ---------------------------------------------------------------------------
# graphs and streams
# ---------------------------------------------------------------------------

def test_append_and_decode_replay_from_a_cuda_graph(pk, cuda_device):
    w, ref = workload("llama8b")
    d = W.to_device(w, cuda_device, upto_last=True)
    k_new, v_new, slots = w.last_token_append()
    k_new = torch.from_numpy(k_new).to(cuda_device)
    v_new = torch.from_numpy(v_new).to(cuda_device)
    slots = torch.from_numpy(slots).to(cuda_device)
    out = torch.empty_like(d["q"])
    scratch = pk.alloc_scratch(d["q"], d["k_cache"], d["block_tables"], 4)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):  # warm-up outside capture
        pk.pkv_append(k_new, v_new, slots, d["k_cache"], d["v_cache"])
        pk.pkv_decode_splitk(d["q"], d["k_cache"], d["v_cache"], d["block_tables"],
                             d["context_lens"], w.scale, num_splits=4, scratch=scratch, out=out)
    torch.cuda.current_stream().wait_stream(s)
    out.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        pk.pkv_append(k_new, v_new, slots, d["k_cache"], d["v_cache"])
        pk.pkv_decode_splitk(d["q"], d["k_cache"], d["v_cache"], d["block_tables"],
                             d["context_lens"], w.scale, num_splits=4, scratch=scratch, out=out)
    for _ in range(3):
        out.zero_()
        g.replay()
    torch.cuda.synchronize()
    assert_attention_close(to_np(out), ref, "graph replay")


# ---------------------------------------------------------------------------
# fused append + decode
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("name,splits", [
    ("tiny", [0, 2]),
    ("llama8b", [0, 1, 3]),
    ("ragged", [0, 8]),
    ("long", [0, 1]),
])
def test_append_decode_matches_oracle(pk, cuda_device, name, splits):
    """One launch appends each sequence's newest token and decodes: the cache
    ends bit-exact and the output matches the oracle over the full context."""
    w, ref = workload(name)
    k_new, v_new, slots = w.last_token_append()
    kd = torch.from_numpy(k_new).to(cuda_device)
    vd = torch.from_numpy(v_new).to(cuda_device)
    sd = torch.from_numpy(slots).to(cuda_device)
    ids, _, _ = W.compact_blocks(w, upto_last=False)
    idx = torch.from_numpy(ids).to(cuda_device)
    hk, hv = W.host_pool(w, upto_last=True)
    assert oracle.append(k_new, v_new, slots, hk, hv) == []
    for S in splits:
        d = W.to_device(w, cuda_device, upto_last=True)
        out = pk.pkv_append_decode(kd, vd, sd, d["k_cache"], d["v_cache"], d["q"],
                                   d["block_tables"], d["context_lens"], w.scale, num_splits=S)
        torch.cuda.synchronize()
        assert_attention_close(to_np(out), ref, f"{name} fused S={S}")
        assert_bits_equal(d["k_cache"].index_select(0, idx).cpu().numpy(), hk[ids], f"{name} K S={S}")
        assert_bits_equal(d["v_cache"].index_select(0, idx).cpu().numpy(), hv[ids], f"{name} V S={S}")
        assert pk.pkv_read_device_status() == 0


def test_append_decode_skips_negative_and_flags_wrong_slots(pk, cuda_device):
    w = W.small_random(1111, num_seqs=3, num_heads=4, num_kv_heads=2, head_dim=128,
                       block_size=16, lens=[40, 17, 5])
    kc, vc = W.host_pool(w)
    ref = oracle.decode(w.q, kc, vc, w.block_tables, w.context_lens, w.scale)
    d = W.to_device(w, cuda_device)  # the pool already holds every row
    before_k = d["k_cache"].clone()
    before_v = d["v_cache"].clone()
    junk = torch.full((3, 2, 128), 7.0, dtype=torch.float16, device=cuda_device)
    wrong = int(w.block_tables[1, 0]) * 16 + 3  # a slot of sequence 1, not its newest position
    slots = torch.tensor([-1, wrong, -5], dtype=torch.int32, device=cuda_device)
    out = pk.pkv_append_decode(junk, junk, slots, d["k_cache"], d["v_cache"], d["q"],
                               d["block_tables"], d["context_lens"], w.scale, num_splits=1)
    assert pk.pkv_read_device_status() & pk.PKV_DEV_BAD_SLOT
    assert torch.equal(d["k_cache"].view(torch.int16), before_k.view(torch.int16))
    assert torch.equal(d["v_cache"].view(torch.int16), before_v.view(torch.int16))
    assert_attention_close(to_np(out), ref, "nothing appended")


# ---------------------------------------------------------------------------
# multi-token queries (varlen, causal)
# ---------------------------------------------------------------------------

def varlen_device(v, dev):
    d = W.to_device(v.base, dev)
    d["q"] = torch.from_numpy(v.q).to(dev)
    d["cu"] = torch.from_numpy(v.cu_seqlens_q).to(dev)
    d["pos"] = torch.from_numpy(v.pos_offsets).to(dev)
    return d


# A chunk covers 8 NT (query, head) columns: NT = 2 once a sequence has more
# than 8, else 1.
@pytest.mark.parametrize("H,Hkv,D,bs,q_lens,prefix", [
    (8, 8, 64, 16, [1, 9, 0, 17], [0, 15, 3, 40]),       # G=1, NT=2: 16 queries per CTA, 2 chunks
    (4, 2, 64, 32, [5, 2, 1], [31, 0, 64]),              # G=2, NT=2: 1 chunk
    (32, 8, 128, 16, [4, 4, 7, 1], [500, 16, 1, 77]),    # G=4, NT=2: 4 queries per CTA
    (28, 4, 128, 32, [3, 1, 6], [33, 1000, 0]),          # G=7, NT=2: 2 queries, 2 unused columns
    (16, 2, 128, 16, [2, 5], [9, 130]),                  # G=8, NT=2: 2 queries per CTA
    (4, 4, 64, 16, [3, 8, 1, 0], [10, 0, 100, 5]),       # G=1, NT=1: 8 queries per CTA
    (8, 4, 128, 32, [4, 1, 3], [64, 200, 1]),            # G=2, NT=1: 4 queries per CTA
    (32, 8, 128, 16, [40, 3], [100, 0]),                 # G=4, NT=2: a 40-token prefill chunk
])
def test_varlen_matches_oracle(pk, cuda_device, varlen_path, H, Hkv, D, bs, q_lens, prefix):
    v = W.varlen_random(3000 + H + D + bs, H, Hkv, D, bs, q_lens, prefix)
    kc, vc = W.host_pool(v.base)
    ref = oracle.varlen(v.q, kc, vc, v.cu_seqlens_q, v.pos_offsets, v.base.block_tables,
                        v.base.scale)
    d = varlen_device(v, cuda_device)
    out = pk.pkv_varlen_attention(d["q"], d["k_cache"], d["v_cache"], d["cu"], d["pos"],
                                  d["block_tables"], v.base.scale, max_q_len=v.max_q_len)
    torch.cuda.synchronize()
    assert_attention_close(to_np(out), ref, f"varlen H{H} Hkv{Hkv} D{D} bs{bs}")
    assert pk.pkv_read_device_status() == 0


def test_varlen_speculative_verification(pk, cuda_device, varlen_path):
    """Four draft tokens per sequence on the Llama-3-8B attention shape."""
    v = W.spec_verify()
    kc, vc = W.host_pool(v.base)
    ref = oracle.varlen(v.q, kc, vc, v.cu_seqlens_q, v.pos_offsets, v.base.block_tables,
                        v.base.scale)
    d = varlen_device(v, cuda_device)
    out = pk.pkv_varlen_attention(d["q"], d["k_cache"], d["v_cache"], d["cu"], d["pos"],
                                  d["block_tables"], v.base.scale, max_q_len=4)
    torch.cuda.synchronize()
    assert_attention_close(to_np(out), ref, "spec verify")
    assert pk.pkv_read_device_status() == 0


def test_varlen_single_queries_match_decode(pk, cuda_device):
    v = W.varlen_random(3100, 32, 8, 128, 16, [1] * 5, [0, 17, 300, 511, 63])
    d = varlen_device(v, cuda_device)
    a = pk.pkv_varlen_attention(d["q"], d["k_cache"], d["v_cache"], d["cu"], d["pos"],
                                d["block_tables"], v.base.scale, max_q_len=1)
    lens = (d["pos"] + 1).contiguous()
    b = pk.pkv_decode(d["q"], d["k_cache"], d["v_cache"], d["block_tables"], lens, v.base.scale)
    torch.cuda.synchronize()
    assert_attention_close(to_np(a), to_np(b), "varlen q_len=1 vs decode")


def test_varlen_bad_block_id_is_skipped_and_flagged(pk, cuda_device, varlen_path):
    """A table entry outside the pool: its 16 positions are left out (never
    read) and flagged; the other sequence is untouched.  Group 4 with 4 and 3
    queries: more than 8 columns per CTA at head_dim 128."""
    v = W.varlen_random(3300, 8, 2, 128, 16, [4, 3], [300, 20])
    kc, vc = W.host_pool(v.base)
    ref = oracle.varlen(v.q, kc, vc, v.cu_seqlens_q, v.pos_offsets, v.base.block_tables,
                        v.base.scale)
    d = varlen_device(v, cuda_device)
    tables = v.base.block_tables.copy()
    tables[0, 5] = v.base.num_blocks + 7  # positions 80..95 of sequence 0
    d["block_tables"] = torch.from_numpy(tables).to(cuda_device)
    for S in (1, 3):
        out = to_np(pk.pkv_varlen_attention_splitk(d["q"], d["k_cache"], d["v_cache"], d["cu"],
                                                   d["pos"], d["block_tables"], v.base.scale,
                                                   max_q_len=4, num_splits=S))
        assert pk.pkv_read_device_status() & pk.PKV_DEV_BAD_BLOCK_ID
        assert np.all(np.isfinite(out))
        assert_attention_close(out[4:], ref[4:], f"S={S} untouched sequence")
        K = v.base.seq_k[0].astype(np.float64)
        V = v.base.seq_v[0].astype(np.float64)
        for t in range(4):
            keep = [j for j in range(300 + t + 1) if not 80 <= j < 96]
            for h in range(8):
                z = v.base.scale * K[keep, h // 4] @ v.q[t, h].astype(np.float64)
                p = np.exp(z - z.max())
                p /= p.sum()
                assert_attention_close(out[t, h], p @ V[keep, h // 4], f"S={S} query {t} head {h}")


def test_varlen_kernels_agree(pk, cuda_device):
    """The mma.sync and tcgen05 kernels on speculative verification: both
    within the oracle tolerance of each other (they round P and the sums
    differently, so not bit for bit)."""
    v = W.spec_verify()
    d = varlen_device(v, cuda_device)
    outs = []
    prev = pk.pkv_set_varlen_tensor_path(0)
    try:
        for path in (0, 1):
            pk.pkv_set_varlen_tensor_path(path)
            outs.append(to_np(pk.pkv_varlen_attention(d["q"], d["k_cache"], d["v_cache"], d["cu"],
                                                      d["pos"], d["block_tables"], v.base.scale,
                                                      max_q_len=4)))
    finally:
        pk.pkv_set_varlen_tensor_path(prev)
    assert_attention_close(outs[1], outs[0].astype(np.float64), "tcgen05 vs mma.sync")
    assert pk.pkv_read_device_status() == 0


# chunked prefill: at least 128 (query, head) rows per sequence at head_dim
# 128 run the tcgen05 prefill kernel (tiles of 128 / G queries)
@pytest.mark.parametrize("H,Hkv,bs,q_lens,prefix", [
    (32, 8, 16, [256, 100, 1, 0, 37], [300, 0, 513, 7, 2000]),   # G=4: 32-query tiles
    (8, 8, 32, [130, 129, 3], [0, 64, 1000]),                      # G=1: 128-query tiles
    (28, 4, 16, [40, 19], [100, 5]),                               # G=7: 18 queries, 2 idle rows
    (16, 2, 16, [33, 16], [50, 0]),                                # G=8: 16-query tiles
    (4, 2, 32, [70, 64, 1], [17, 0, 300]),                         # G=2: 64-query tiles
])
def test_prefill_matches_oracle(pk, cuda_device, H, Hkv, bs, q_lens, prefix):
    v = W.varlen_random(3400 + H + bs + len(q_lens), H, Hkv, 128, bs, q_lens, prefix)
    kc, vc = W.host_pool(v.base)
    ref = oracle.varlen(v.q, kc, vc, v.cu_seqlens_q, v.pos_offsets, v.base.block_tables,
                        v.base.scale)
    d = varlen_device(v, cuda_device)
    out = pk.pkv_varlen_attention(d["q"], d["k_cache"], d["v_cache"], d["cu"], d["pos"],
                                  d["block_tables"], v.base.scale, max_q_len=v.max_q_len)
    torch.cuda.synchronize()
    assert_attention_close(to_np(out), ref, f"prefill single H{H} Hkv{Hkv} bs{bs}")
    # split-K on the prefill kernel: the heuristic and forced counts (many
    # splits empty for the short contexts, one split for some pairs)
    for S in (0, 2, 5):
        out = pk.pkv_varlen_attention_splitk(d["q"], d["k_cache"], d["v_cache"], d["cu"], d["pos"],
                                             d["block_tables"], v.base.scale,
                                             max_q_len=v.max_q_len, num_splits=S)
        torch.cuda.synchronize()
        assert_attention_close(to_np(out), ref, f"prefill splitk S={S} H{H} Hkv{Hkv} bs{bs}")
    assert pk.pkv_read_device_status() == 0


def _prefill_rule(num_seqs, H, Hkv, max_q_len, mbps, bs, sms):
    """The chunked-prefill split rule written out: pairs of 128 / G-query
    tiles against one CTA per SM, nearest one wave when fewer, >= 512 tokens
    of table capacity per split, at most 64, at most max_blocks_per_seq."""
    G = H // Hkv
    qc = 2 * (128 // G)
    pairs = num_seqs * Hkv * -(-max_q_len // qc)
    s = 1 if pairs >= sms else (2 * sms + pairs) // (2 * pairs)
    s = min(s, mbps * bs // 512, 64)
    return max(1, min(s, mbps))


@pytest.mark.parametrize("num_seqs,total_q,max_q_len,H,Hkv,mbps,bs", [
    (1, 512, 512, 32, 8, 160, 16),     # one sequence: 64 pairs
    (4, 2048, 512, 32, 8, 160, 16),    # four: 256 pairs, a full wave
    (1, 128, 128, 8, 8, 64, 16),       # G = 1 (one 128-query tile per pair): capped by capacity
    (1, 64, 64, 32, 8, 1000, 16),      # 8 pairs, long tables
    (3, 300, 100, 28, 4, 40, 32),      # G = 7
])
def test_prefill_split_plan_follows_the_rule(pk, cuda_device, num_seqs, total_q, max_q_len, H,
                                             Hkv, mbps, bs):
    sms = torch.cuda.get_device_properties(cuda_device).multi_processor_count
    S, n = pk.pkv_varlen_splitk_plan(num_seqs, total_q, max_q_len, H, Hkv, 128, mbps, bs, 0)
    assert S == _prefill_rule(num_seqs, H, Hkv, max_q_len, mbps, bs, sms)
    assert n == (0 if S == 1 else pk.pkv_splitk_scratch_bytes(total_q, H, 128, S))
    # head_dim 64 is not chunked prefill: the varlen rule
    S64, _ = pk.pkv_varlen_splitk_plan(num_seqs, total_q, max_q_len, H, Hkv, 64, mbps, bs, 0)
    assert S64 == max(1, min(pk.pkv_varlen_pick_num_splits(num_seqs, H, Hkv, max_q_len, mbps,
                                                           bs, sms), mbps))


@pytest.mark.parametrize("scale_mul", [-1.0, 0.0])
def test_prefill_nonpositive_scale(pk, cuda_device, scale_mul):
    """A negative or zero scale (the maximum of the scaled scores is then not
    the raw maximum scaled): softmax(scale q.k) as defined."""
    v = W.varlen_random(3450, 32, 8, 128, 16, [200, 64], [400, 0])
    kc, vc = W.host_pool(v.base)
    scale = scale_mul * v.base.scale
    ref = oracle.varlen(v.q, kc, vc, v.cu_seqlens_q, v.pos_offsets, v.base.block_tables, scale)
    d = varlen_device(v, cuda_device)
    out = pk.pkv_varlen_attention(d["q"], d["k_cache"], d["v_cache"], d["cu"], d["pos"],
                                  d["block_tables"], scale, max_q_len=v.max_q_len)
    torch.cuda.synchronize()
    assert_attention_close(to_np(out), ref, f"prefill scale x{scale_mul}")
    assert pk.pkv_read_device_status() == 0


def test_prefill_bad_block_id_is_skipped_and_flagged(pk, cuda_device):
    """A table entry outside the pool inside a prefill tile's context: its 16
    positions are left out and flagged, the other sequence is untouched."""
    v = W.varlen_random(3500, 8, 2, 128, 16, [64, 40], [200, 30])
    kc, vc = W.host_pool(v.base)
    ref = oracle.varlen(v.q, kc, vc, v.cu_seqlens_q, v.pos_offsets, v.base.block_tables,
                        v.base.scale)
    d = varlen_device(v, cuda_device)
    tables = v.base.block_tables.copy()
    tables[0, 5] = v.base.num_blocks + 3  # positions 80..95 of sequence 0
    d["block_tables"] = torch.from_numpy(tables).to(cuda_device)
    K = v.base.seq_k[0].astype(np.float64)
    V = v.base.seq_v[0].astype(np.float64)
    for S in (1, 3):  # one pass, and split-K (the entry falls in the first split)
        out = to_np(pk.pkv_varlen_attention_splitk(d["q"], d["k_cache"], d["v_cache"], d["cu"],
                                                   d["pos"], d["block_tables"], v.base.scale,
                                                   max_q_len=64, num_splits=S))
        assert pk.pkv_read_device_status() & pk.PKV_DEV_BAD_BLOCK_ID
        assert np.all(np.isfinite(out))
        assert_attention_close(out[64:], ref[64:], f"untouched sequence, S={S}")
        for t in (0, 17, 63):
            keep = [j for j in range(200 + t + 1) if not 80 <= j < 96]
            for h in range(8):
                z = v.base.scale * K[keep, h // 4] @ v.q[t, h].astype(np.float64)
                p = np.exp(z - z.max())
                p /= p.sum()
                assert_attention_close(out[t, h], p @ V[keep, h // 4],
                                       f"query {t} head {h}, S={S}")


def test_varlen_flags_bad_query_ranges(pk, cuda_device):
    v = W.varlen_random(3200, 4, 2, 64, 16, [2, 2], [5, 5])
    d = varlen_device(v, cuda_device)
    d["cu"] = torch.tensor([0, 2, 9], dtype=torch.int32, device=cuda_device)  # past total_q
    out = torch.zeros_like(d["q"])
    pk.pkv_varlen_attention(d["q"], d["k_cache"], d["v_cache"], d["cu"], d["pos"],
                            d["block_tables"], v.base.scale, max_q_len=4, out=out)
    assert pk.pkv_read_device_status() & pk.PKV_DEV_BAD_CONTEXT_LEN
    assert torch.count_nonzero(out[2:]).item() == 0  # sequence 1 skipped


# ---------------------------------------------------------------------------
# varlen split-K (each chunk of queries' context split over CTAs, merged)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("H,Hkv,D,bs,q_lens,prefix", [
    (8, 8, 64, 16, [1, 9, 0, 17], [0, 15, 3, 40]),
    (28, 4, 128, 32, [3, 1, 6], [33, 1000, 0]),
    (8, 4, 128, 32, [4, 1, 3], [64, 200, 1]),
    (32, 8, 128, 16, [40, 3], [100, 0]),  # early queries see none of the later splits
])
def test_varlen_splitk_matches_oracle(pk, cuda_device, varlen_path, H, Hkv, D, bs, q_lens,
                                      prefix):
    v = W.varlen_random(5000 + H + D + bs, H, Hkv, D, bs, q_lens, prefix)
    kc, vc = W.host_pool(v.base)
    ref = oracle.varlen(v.q, kc, vc, v.cu_seqlens_q, v.pos_offsets, v.base.block_tables,
                        v.base.scale)
    d = varlen_device(v, cuda_device)
    for S in (0, 2, 3, 7, 128):
        out = pk.pkv_varlen_attention_splitk(d["q"], d["k_cache"], d["v_cache"], d["cu"],
                                             d["pos"], d["block_tables"], v.base.scale,
                                             max_q_len=v.max_q_len, num_splits=S)
        torch.cuda.synchronize()
        assert_attention_close(to_np(out), ref, f"varlen split-K S={S} H{H} Hkv{Hkv} D{D} bs{bs}")
    assert pk.pkv_read_device_status() == 0


def test_varlen_splitk_long_context_speculative_verification(pk, cuda_device, varlen_path):
    """Four draft tokens after 32K..128K-token prefixes: the heuristic splits
    each context (the unsplit grid is 32 CTAs), and the result matches the
    oracle, for the blocked layout (either kernel) and the vLLM layout (the
    mma.sync kernel) alike."""
    v = W.spec_verify_long()
    kc, vc = W.host_pool(v.base)
    ref = oracle.varlen_fast(v.q, kc, vc, v.cu_seqlens_q, v.pos_offsets, v.base.block_tables,
                             v.base.scale)
    del kc, vc
    d = varlen_device(v, cuda_device)
    S = pk.varlen_splits_for(d["q"], d["k_cache"], d["block_tables"], 4)
    assert S > 1
    outs = {}
    for label, S_req in (("heuristic", 0), ("S=16", 16)):
        outs[label] = pk.pkv_varlen_attention_splitk(d["q"], d["k_cache"], d["v_cache"], d["cu"],
                                                     d["pos"], d["block_tables"], v.base.scale,
                                                     max_q_len=4, num_splits=S_req)
        torch.cuda.synchronize()
        assert_attention_close(to_np(outs[label]), ref, f"long spec verify {label}")
    del d["k_cache"], d["v_cache"]
    dv = W.to_device_vllm(v.base, cuda_device)
    got_v = pk.pkv_varlen_attention_splitk_vllm_layout(d["q"], dv["k_cache"], dv["v_cache"],
                                                       d["cu"], d["pos"], d["block_tables"],
                                                       v.base.scale, max_q_len=4, num_splits=0)
    torch.cuda.synchronize()
    assert_attention_close(to_np(got_v), ref, "long spec verify, vLLM layout")
    assert pk.pkv_read_device_status() == 0


def test_varlen_splitk_rejects_small_scratch(pk, cuda_device):
    v = W.varlen_random(5100, 8, 2, 64, 16, [3, 2], [100, 40])
    d = varlen_device(v, cuda_device)
    small = torch.empty(16, dtype=torch.uint8, device=cuda_device)
    with pytest.raises(pk.PagedKVError) as e:
        pk.pkv_varlen_attention_splitk(d["q"], d["k_cache"], d["v_cache"], d["cu"], d["pos"],
                                       d["block_tables"], v.base.scale, max_q_len=3,
                                       num_splits=4, scratch=small)
    assert e.value.status == pk.PKV_ERR_SCRATCH_TOO_SMALL


def test_varlen_splitk_replays_from_a_cuda_graph(pk, cuda_device, varlen_path):
    """Phase 1 and the combine, captured once and replayed, reproduce the
    eager result bit for bit (no host reads; the split count and scratch
    are fixed at capture)."""
    v = W.varlen_random(5200, 16, 4, 128, 16, [4, 2, 5], [3000, 1500, 4090])
    d = varlen_device(v, cuda_device)
    S = 6
    n = pk.pkv_splitk_scratch_bytes(v.total_q, 16, 128, S)
    scratch = torch.empty(n, dtype=torch.uint8, device=cuda_device)
    eager = pk.pkv_varlen_attention_splitk(d["q"], d["k_cache"], d["v_cache"], d["cu"], d["pos"],
                                           d["block_tables"], v.base.scale, max_q_len=5,
                                           num_splits=S, scratch=scratch).clone()
    out = torch.zeros_like(eager)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(g):
            pk.pkv_varlen_attention_splitk(d["q"], d["k_cache"], d["v_cache"], d["cu"],
                                           d["pos"], d["block_tables"], v.base.scale,
                                           max_q_len=5, num_splits=S, scratch=scratch, out=out)
    torch.cuda.current_stream().wait_stream(side)
    for _ in range(2):
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert_bits_equal(out.cpu().numpy(), eager.cpu().numpy(), "graph replay")
    kc, vc = W.host_pool(v.base)
    ref = oracle.varlen(v.q, kc, vc, v.cu_seqlens_q, v.pos_offsets, v.base.block_tables,
                        v.base.scale)
    assert_attention_close(to_np(out), ref, "graph replay vs oracle")
    assert pk.pkv_read_device_status() == 0
