"""GPU parity of the vLLM-layout calls (pkv_append_vllm_layout,
pkv_decode_vllm_layout, pkv_varlen_attention_vllm_layout) against the CPU
oracle, through the C ABI.

Pools are K [NB][Hkv][D/8][bs][8] and V [NB][Hkv][D][bs], built from the
same seeded workloads as the blocked tests, with NaN in every unused block and
in the rows past each sequence's length.  Append is compared bit for bit;
attention within |gpu-ref| <= 2e-3 + 1e-2|ref|.  The vLLM-layout decode does
the same arithmetic on the same values as the blocked decode, so the two
outputs are also compared bit for bit.
"""

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

    pagedkv.pkv_read_device_status()
    return pagedkv


def to_np(t):
    return t.float().cpu().numpy().astype(np.float64)


def vllm_appended(pk, w, dev):
    """vLLM-layout device pools without each sequence's newest token, then
    pkv_append_vllm_layout writes it."""
    d = W.to_device_vllm(w, dev, upto_last=True)
    k_new, v_new, slots = w.last_token_append()
    pk.pkv_append_vllm_layout(torch.from_numpy(k_new).to(dev), torch.from_numpy(v_new).to(dev),
                              torch.from_numpy(slots).to(dev), d["k_cache"], d["v_cache"])
    return d


def oracle_ref(w, seqs=None):
    kc, vc = W.host_pool_vllm(w)
    return oracle.decode_vllm_layout(w.q, kc, vc, w.block_tables, w.context_lens, w.scale,
                                     seqs=seqs, fast=True)


@pytest.mark.parametrize("name", ["tiny", "llama8b"])
def test_vllm_append_is_bit_exact(pk, cuda_device, name):
    w = W.make(name)
    d = vllm_appended(pk, w, cuda_device)
    ids, _, _ = W.compact_blocks(w)
    idx = torch.from_numpy(ids).to(cuda_device)
    got_k = d["k_cache"].index_select(0, idx).cpu().numpy()
    got_v = d["v_cache"].index_select(0, idx).cpu().numpy()
    hk, hv = W.host_pool_vllm(w, upto_last=True)
    k_new, v_new, slots = w.last_token_append()
    assert oracle.append_vllm_layout(k_new, v_new, slots, hk, hv) == []
    assert_bits_equal(got_k, hk[ids], f"{name} K")
    assert_bits_equal(got_v, hv[ids], f"{name} V")
    assert pk.pkv_read_device_status() == 0


def test_vllm_append_of_many_tokens_with_padding(pk, cuda_device):
    """A prefill-sized append (every token of every sequence, shuffled, with
    padding rows at slot -1) over random pool contents."""
    w = W.small_random(211, num_seqs=5, num_heads=8, num_kv_heads=4, head_dim=128, block_size=32,
                       lens=[1, 31, 32, 33, 200])
    rng = np.random.default_rng(5)
    NB, Hkv, bs, D = w.num_blocks, w.num_kv_heads, w.block_size, w.head_dim
    hk = rng.standard_normal((NB, Hkv, D // 8, bs, 8)).astype(np.float16)
    hv = rng.standard_normal((NB, Hkv, D, bs)).astype(np.float16)
    ks, vs, slots = [], [], []
    for s in range(w.num_seqs):
        L = int(w.context_lens[s])
        ks.append(w.seq_k[s][:L])
        vs.append(w.seq_v[s][:L])
        pos = np.arange(L)
        slots.append(w.block_tables[s, pos // bs] * bs + pos % bs)
    k = np.concatenate(ks)
    v = np.concatenate(vs)
    sl = np.concatenate(slots).astype(np.int32)
    order = rng.permutation(len(sl))
    k, v, sl = k[order], v[order], sl[order]
    pad = rng.choice(len(sl), size=7, replace=False)
    k = np.insert(k, pad, np.nan, axis=0).astype(np.float16)
    v = np.insert(v, pad, np.nan, axis=0).astype(np.float16)
    sl = np.insert(sl, pad, -1).astype(np.int32)
    dk = torch.from_numpy(hk).to(cuda_device)
    dv = torch.from_numpy(hv).to(cuda_device)
    pk.pkv_append_vllm_layout(torch.from_numpy(k).to(cuda_device),
                              torch.from_numpy(v).to(cuda_device),
                              torch.from_numpy(sl).to(cuda_device), dk, dv)
    assert oracle.append_vllm_layout(k, v, sl, hk, hv) == []
    assert_bits_equal(dk.cpu().numpy(), hk, "K")
    assert_bits_equal(dv.cpu().numpy(), hv, "V")
    assert pk.pkv_read_device_status() == 0


def test_vllm_append_skips_padding_and_flags_bad_slots(pk, cuda_device):
    w = W.make("tiny")
    d = W.to_device_vllm(w, cuda_device)
    before_k = d["k_cache"].clone()
    before_v = d["v_cache"].clone()
    k = torch.ones((3, w.num_kv_heads, w.head_dim), dtype=torch.float16, device=cuda_device)
    slots = torch.tensor([-1, -5, w.num_blocks * w.block_size], dtype=torch.int32,
                         device=cuda_device)
    pk.pkv_append_vllm_layout(k, k, slots, d["k_cache"], d["v_cache"])
    assert pk.pkv_read_device_status() & pk.PKV_DEV_BAD_SLOT
    assert torch.equal(d["k_cache"].view(torch.int16), before_k.view(torch.int16))
    assert torch.equal(d["v_cache"].view(torch.int16), before_v.view(torch.int16))


@pytest.mark.parametrize("name,splits,seqs", [
    ("tiny", [1, 0, 2, 3], None),
    ("llama8b", [1, 0, 4, 16], None),
    ("long", [0, 16, 64], None),
    ("ragged", [1, 0, 8], list(range(0, 256, 5))),
])
def test_vllm_decode_matches_oracle(pk, cuda_device, name, splits, seqs):
    w = W.make(name)
    ref = oracle_ref(w, seqs)
    d = vllm_appended(pk, w, cuda_device)
    rows = slice(None) if seqs is None else seqs
    for S in splits:
        got = to_np(pk.pkv_decode_vllm_layout(d["q"], d["k_cache"], d["v_cache"],
                                              d["block_tables"], d["context_lens"], w.scale,
                                              num_splits=S))
        assert_attention_close(got[rows], ref[rows], f"{name}/S={S}")
    assert pk.pkv_read_device_status() == 0


@pytest.mark.parametrize("name,S", [("tiny", 1), ("llama8b", 1), ("llama8b", 4)])
def test_vllm_decode_equals_blocked_decode_bit_for_bit(pk, cuda_device, name, S):
    """At block size 16 both layouts stage whole blocks and fold them in the
    same order, so the outputs agree bit for bit."""
    w = W.make(name)
    dv = W.to_device_vllm(w, cuda_device)
    db = W.to_device(w, cuda_device)
    got_v = pk.pkv_decode_vllm_layout(dv["q"], dv["k_cache"], dv["v_cache"], dv["block_tables"],
                                      dv["context_lens"], w.scale, num_splits=S)
    del dv
    got_b = pk.pkv_decode_splitk(db["q"], db["k_cache"], db["v_cache"], db["block_tables"],
                                 db["context_lens"], w.scale, num_splits=S)
    assert_bits_equal(got_v.cpu().numpy(), got_b.cpu().numpy(), f"{name} S={S}")


def test_vllm_and_blocked_decode_at_block_size_32_both_match_the_oracle(pk, cuda_device):
    """At block size 32 the blocked layout is staged in 16-row sub-tiles and
    the vLLM layout in whole blocks, so the online softmax folds the tokens in
    different steps and the outputs may differ in the last bit; both stay
    within the attention tolerance of the oracle (the ragged workload)."""
    w = W.make("ragged")
    kc, vc = W.host_pool(w)
    ref = oracle.decode_fast(w.q, kc, vc, w.block_tables, w.context_lens, w.scale)
    del kc, vc
    dv = W.to_device_vllm(w, cuda_device)
    got_v = to_np(pk.pkv_decode_vllm_layout(dv["q"], dv["k_cache"], dv["v_cache"],
                                            dv["block_tables"], dv["context_lens"], w.scale,
                                            num_splits=0))
    del dv
    db = W.to_device(w, cuda_device)
    got_b = to_np(pk.pkv_decode_splitk(db["q"], db["k_cache"], db["v_cache"], db["block_tables"],
                                       db["context_lens"], w.scale, num_splits=0))
    assert_attention_close(got_v, ref, "ragged, vLLM layout")
    assert_attention_close(got_b, ref, "ragged, blocked layout")
    assert pk.pkv_read_device_status() == 0


@pytest.mark.parametrize("D,bs,G", [(64, 16, 1), (64, 32, 3), (128, 16, 5), (128, 32, 8),
                                    (64, 16, 8), (128, 32, 7)])
def test_vllm_ragged_small_shapes(pk, cuda_device, D, bs, G):
    lens = [1, bs - 1, bs, bs + 1, 5 * bs + 3, 9, 37, 300]
    w = W.small_random(2000 + D + bs + G, num_seqs=len(lens), num_heads=2 * G, num_kv_heads=2,
                       head_dim=D, block_size=bs, lens=lens)
    kc, vc = W.host_pool_vllm(w)
    ref = oracle.decode_vllm_layout(w.q, kc, vc, w.block_tables, w.context_lens, w.scale)
    d = vllm_appended(pk, w, cuda_device)
    for S in (1, 0, 2, 5, 128):
        got = to_np(pk.pkv_decode_vllm_layout(d["q"], d["k_cache"], d["v_cache"],
                                              d["block_tables"], d["context_lens"], w.scale,
                                              num_splits=S))
        assert_attention_close(got, ref, f"D{D} bs{bs} G{G} S={S}")
    assert pk.pkv_read_device_status() == 0


def test_vllm_context_len_one_is_exact(pk, cuda_device):
    w = W.small_random(241, num_seqs=5, num_heads=8, num_kv_heads=2, head_dim=64, block_size=16,
                       lens=[1, 20, 1, 1, 3])
    d = vllm_appended(pk, w, cuda_device)
    for S in (1, 2):
        out = pk.pkv_decode_vllm_layout(d["q"], d["k_cache"], d["v_cache"], d["block_tables"],
                                        d["context_lens"], w.scale, num_splits=S).cpu().numpy()
        for s in range(w.num_seqs):
            if int(w.context_lens[s]) != 1:
                continue
            for h in range(w.num_heads):
                exp = w.seq_v[s][0, h // w.group]
                assert np.array_equal(out[s, h].view(np.uint16), exp.view(np.uint16)), (S, s, h)


def test_vllm_bad_block_id_is_skipped_and_flagged(pk, cuda_device):
    w = W.small_random(251, num_seqs=2, num_heads=4, num_kv_heads=2, head_dim=128,
                       block_size=16, lens=[48, 40])
    kc, vc = W.host_pool_vllm(w)
    ref = oracle.decode_vllm_layout(w.q, kc, vc, w.block_tables, w.context_lens, w.scale)
    d = W.to_device_vllm(w, cuda_device)
    tables = w.block_tables.copy()
    tables[0, 1] = w.num_blocks + 5
    d["block_tables"] = torch.from_numpy(tables).to(cuda_device)
    for S in (1, 3):
        out = to_np(pk.pkv_decode_vllm_layout(d["q"], d["k_cache"], d["v_cache"],
                                              d["block_tables"], d["context_lens"], w.scale,
                                              num_splits=S))
        assert pk.pkv_read_device_status() & pk.PKV_DEV_BAD_BLOCK_ID
        assert np.all(np.isfinite(out))
        assert_attention_close(out[1], ref[1], "untouched sequence")


def test_vllm_negative_split_count_is_rejected(pk, cuda_device):
    w = W.make("tiny")
    d = W.to_device_vllm(w, cuda_device)
    scratch = torch.empty(1 << 20, dtype=torch.uint8, device=cuda_device)
    with pytest.raises(pk.PagedKVError) as e:
        pk.pkv_decode_vllm_layout(d["q"], d["k_cache"], d["v_cache"], d["block_tables"],
                                  d["context_lens"], w.scale, num_splits=-1, scratch=scratch)
    assert e.value.status == pk.PKV_ERR_INVALID_ARG


# ---------------------------------------------------------------------------
# several causal queries per sequence on the vLLM layout
# ---------------------------------------------------------------------------

def varlen_device_vllm(v, dev):
    d = W.to_device_vllm(v.base, dev)
    d["q"] = torch.from_numpy(v.q).to(dev)
    d["cu"] = torch.from_numpy(v.cu_seqlens_q).to(dev)
    d["pos"] = torch.from_numpy(v.pos_offsets).to(dev)
    return d


@pytest.mark.parametrize("H,Hkv,D,bs,q_lens,prefix", [
    (8, 8, 64, 16, [1, 9, 0, 17], [0, 15, 3, 40]),       # G=1, NT=2, 2 chunks
    (32, 8, 128, 16, [4, 4, 7, 1], [500, 16, 1, 77]),    # G=4, NT=2
    (28, 4, 128, 32, [3, 1, 6], [33, 1000, 0]),          # G=7, NT=2
    (8, 4, 128, 32, [4, 1, 3], [64, 200, 1]),            # G=2, NT=1
])
def test_vllm_varlen_matches_oracle(pk, cuda_device, H, Hkv, D, bs, q_lens, prefix):
    v = W.varlen_random(4000 + H + D + bs, H, Hkv, D, bs, q_lens, prefix)
    kc, vc = W.host_pool_vllm(v.base)
    ref = oracle.varlen_vllm_layout(v.q, kc, vc, v.cu_seqlens_q, v.pos_offsets,
                                    v.base.block_tables, v.base.scale)
    d = varlen_device_vllm(v, cuda_device)
    out = pk.pkv_varlen_attention_vllm_layout(d["q"], d["k_cache"], d["v_cache"], d["cu"],
                                              d["pos"], d["block_tables"], v.base.scale,
                                              max_q_len=v.max_q_len)
    torch.cuda.synchronize()
    assert_attention_close(to_np(out), ref, f"vLLM varlen H{H} Hkv{Hkv} D{D} bs{bs}")
    assert pk.pkv_read_device_status() == 0


def test_vllm_and_blocked_speculative_verification_match_the_oracle(pk, cuda_device):
    """Four draft tokens per sequence on the Llama-3-8B shape: the vLLM-layout
    call (mma.sync kernel) and the blocked call (tcgen05 kernel at head_dim
    128) both match the oracle."""
    v = W.spec_verify()
    kc, vc = W.host_pool_vllm(v.base)
    ref = oracle.varlen_vllm_layout(v.q, kc, vc, v.cu_seqlens_q, v.pos_offsets,
                                    v.base.block_tables, v.base.scale)
    del kc, vc
    d = varlen_device_vllm(v, cuda_device)
    got = pk.pkv_varlen_attention_vllm_layout(d["q"], d["k_cache"], d["v_cache"], d["cu"],
                                              d["pos"], d["block_tables"], v.base.scale,
                                              max_q_len=4)
    del d["k_cache"], d["v_cache"]
    db = W.to_device(v.base, cuda_device)
    blocked = pk.pkv_varlen_attention(d["q"], db["k_cache"], db["v_cache"], d["cu"], d["pos"],
                                      d["block_tables"], v.base.scale, max_q_len=4)
    torch.cuda.synchronize()
    assert_attention_close(to_np(got), ref, "vLLM spec verify")
    assert_attention_close(to_np(blocked), ref, "blocked spec verify")
    assert pk.pkv_read_device_status() == 0
