"""GPU parity of pkv_qkv_norm_rope_append_decode (a whole decode attention
step in one launch: norm + rotary of each sequence's newest query and key
heads, append of the key and value rows, paged decode) against the CPU
oracle, through the C ABI.

The oracle runs the two definitions in order: qkv_norm_rope_append at
position context_lens[s] - 1, then decode with the rotated queries rounded
to f16.  The output must meet the attention tolerance; the appended key rows
must be within one f16 ulp of the float64 result, value rows bit-exact, and
every other pool entry unchanged."""

import numpy as np
import pytest

import oracle
from oracle import qkv_norm_rope as Q
from paged_kv_decode_08_gb300 import workloads as W
from tests.tolerance import assert_attention_close, assert_bits_equal

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def pk(cuda_device):
    from paged_kv_decode_08_gb300 import pagedkv

    pagedkv.pkv_read_device_status()
    return pagedkv


def assert_within_one_ulp(gpu16, ref64, what):
    ref16 = np.asarray(ref64, np.float64).astype(np.float16)
    ulp = np.spacing(np.abs(ref16)).astype(np.float64)
    diff = np.abs(np.asarray(gpu16, np.float16).astype(np.float64) - ref16.astype(np.float64))
    bad = ~(diff <= ulp)
    assert not bad.any(), f"{what}: {int(bad.sum())} elements off by more than one ulp"


def step_case(seed, H, Hkv, D, bs, prefix, norm=True):
    """One new token per sequence after a random earlier context of
    ``prefix[s]`` rows; unused pool entries hold NaN."""
    c = W.qkv_case(seed, H, Hkv, D, bs, [1] * len(prefix), prefix, norm=norm)
    rng = np.random.default_rng(seed + 1)
    shape = (c.num_blocks, Hkv, bs, D)
    kc = np.full(shape, np.nan, np.float16)
    vc = np.full(shape, np.nan, np.float16)
    for s, p0 in enumerate(prefix):
        for p in range(p0):
            blk = int(c.block_tables[s][p // bs])
            kc[blk, :, p % bs] = rng.standard_normal((Hkv, D)).astype(np.float16)
            vc[blk, :, p % bs] = rng.standard_normal((Hkv, D)).astype(np.float16)
    lens = (np.asarray(prefix) + 1).astype(np.int32)
    return c, kc, vc, lens


def oracle_step(c, kc, vc, lens, scale):
    kc_ref, vc_ref = kc.copy(), vc.copy()
    q_ref, k_rows = Q.qkv_norm_rope_append(c.qkv, c.q_norm_w, c.k_norm_w, c.cos, c.sin, kc_ref,
                                           vc_ref, c.cu_seqlens_q, c.pos_offsets,
                                           c.block_tables, c.num_heads, c.num_kv_heads, c.eps)
    out = oracle.decode(q_ref.astype(np.float16), kc_ref, vc_ref, c.block_tables, lens, scale)
    return out, k_rows, kc_ref, vc_ref


def dev(a, d):
    return None if a is None else torch.from_numpy(np.ascontiguousarray(a)).to(d)


def run_step(pk, c, kc, vc, lens, scale, d, num_splits, cos=None, sin=None, bt=None):
    kc_d, vc_d = dev(kc, d), dev(vc, d)
    out = pk.pkv_qkv_norm_rope_append_decode(
        dev(c.qkv, d), dev(c.q_norm_w, d), dev(c.k_norm_w, d),
        dev(c.cos if cos is None else cos, d), dev(c.sin if sin is None else sin, d), kc_d, vc_d,
        dev(c.block_tables if bt is None else bt, d), dev(lens, d), c.num_heads, scale,
        eps=c.eps, num_splits=num_splits)
    torch.cuda.synchronize()
    return out.float().cpu().numpy().astype(np.float64), kc_d.cpu().numpy(), vc_d.cpu().numpy()


@pytest.mark.parametrize("H,Hkv,D,bs,prefix,norm,S", [
    (32, 8, 128, 16, [300, 17, 1023, 64, 0, 511], True, 1),     # Llama-3-8B shape, one pass
    (32, 8, 128, 16, [300, 17, 1023, 64, 0, 511], True, 4),     # the same, split-K
    (32, 8, 128, 16, [4095, 2048, 15, 16, 1], True, 0),         # heuristic split count
    (8, 8, 64, 32, [5, 100, 31, 32], False, 1),                 # MHA, no norm weights
    (28, 4, 128, 32, [1000, 63], True, 3),                      # group of 7
    (16, 2, 64, 16, [7, 200, 33], True, 2),                     # group of 8
])
def test_qkv_norm_rope_append_decode_matches_oracle(pk, cuda_device, H, Hkv, D, bs, prefix, norm,
                                                    S):
    c, kc, vc, lens = step_case(7000 + H + D + bs + S, H, Hkv, D, bs, prefix, norm)
    scale = 1.0 / np.sqrt(D)
    ref, k_rows, kc_ref, vc_ref = oracle_step(c, kc, vc, lens, scale)
    got, kc_got, vc_got = run_step(pk, c, kc, vc, lens, scale, cuda_device, S)
    assert_attention_close(got, ref, f"fused qkv step S={S}")
    new = set()
    for s, p0 in enumerate(prefix):
        blk, off = int(c.block_tables[s][p0 // bs]), p0 % bs
        new.add((blk, off))
        assert_within_one_ulp(kc_got[blk, :, off], k_rows[s], f"k row of sequence {s}")
        assert_bits_equal(vc_got[blk, :, off], vc_ref[blk, :, off], f"v row of sequence {s}")
    # every other entry is as it was (NaN poison included)
    mask = np.ones(kc.shape[0:1] + kc.shape[2:3], bool)
    for blk, off in new:
        mask[blk, off] = False
    keep = np.broadcast_to(mask[:, None, :, None], kc.shape)
    assert_bits_equal(kc_got[keep], kc[keep], "untouched k entries")
    assert_bits_equal(vc_got[keep], vc[keep], "untouched v entries")
    assert pk.pkv_read_device_status() == 0


def test_fused_step_agrees_with_the_two_launch_step(pk, cuda_device):
    """The same step through pkv_qkv_norm_rope_append + pkv_decode_splitk and
    through the fused call: both within tolerance of the oracle and of each
    other."""
    H, Hkv, D, bs = 32, 8, 128, 16
    prefix = [129, 4000, 77, 2047]
    c, kc, vc, lens = step_case(7100, H, Hkv, D, bs, prefix)
    scale = 1.0 / np.sqrt(D)
    ref, _, _, _ = oracle_step(c, kc, vc, lens, scale)
    fused, kc_f, vc_f = run_step(pk, c, kc, vc, lens, scale, cuda_device, 0)
    d = cuda_device
    kc_d, vc_d = dev(kc, d), dev(vc, d)
    q = pk.pkv_qkv_norm_rope_append(dev(c.qkv, d), dev(c.q_norm_w, d), dev(c.k_norm_w, d),
                                    dev(c.cos, d), dev(c.sin, d), kc_d, vc_d,
                                    dev(c.cu_seqlens_q, d), dev(c.pos_offsets, d),
                                    dev(c.block_tables, d), H, eps=c.eps)
    two = pk.pkv_decode_splitk(q, kc_d, vc_d, dev(c.block_tables, d), dev(lens, d), scale)
    torch.cuda.synchronize()
    two = two.float().cpu().numpy().astype(np.float64)
    assert_attention_close(fused, ref, "fused")
    assert_attention_close(two, ref, "two launches")
    assert_attention_close(fused, two, "fused vs two launches")
    assert_bits_equal(vc_f, vc_d.cpu().numpy(), "value pools")
    assert pk.pkv_read_device_status() == 0


def test_fused_step_flags_positions_without_angles_and_bad_blocks(pk, cuda_device):
    """A sequence whose newest position is past the rotary tables is flagged
    and appends nothing; a table entry out of range at the newest position is
    flagged and that row is neither written nor used.  The other sequences
    are unaffected."""
    H, Hkv, D, bs = 16, 4, 128, 16
    prefix = [50, 10, 30]
    c, kc, vc, lens = step_case(7200, H, Hkv, D, bs, prefix)
    scale = 1.0 / np.sqrt(D)
    ref, _, kc_ref, vc_ref = oracle_step(c, kc, vc, lens, scale)

    # sequence 0 (newest position 50) has no angles with 40-row tables
    got, kc_got, vc_got = run_step(pk, c, kc, vc, lens, scale, cuda_device, 1,
                                   cos=c.cos[:40], sin=c.sin[:40])
    assert pk.pkv_read_device_status() & pk.PKV_DEV_BAD_CONTEXT_LEN
    blk0 = int(c.block_tables[0][50 // bs])
    assert np.isnan(kc_got[blk0, :, 50 % bs].astype(np.float32)).all()
    assert np.isnan(vc_got[blk0, :, 50 % bs].astype(np.float32)).all()
    for s in (1, 2):
        assert_attention_close(got[s:s + 1], ref[s:s + 1], f"sequence {s} beside a flagged one")

    # sequence 2's newest position maps to a block id past the pool
    bt = c.block_tables.copy()
    bt[2, 30 // bs] = c.num_blocks + 5
    got, kc_got, vc_got = run_step(pk, c, kc, vc, lens, scale, cuda_device, 1, bt=bt)
    flags = pk.pkv_read_device_status()
    assert flags & pk.PKV_DEV_BAD_SLOT
    assert flags & pk.PKV_DEV_BAD_BLOCK_ID
    for s in (0, 1):
        assert_attention_close(got[s:s + 1], ref[s:s + 1], f"sequence {s} beside a bad table")
    # nothing was written for sequence 2; sequences 0 and 1 appended as usual
    changed = ~((kc_got == kc) | (np.isnan(kc_got.astype(np.float32)) &
                                  np.isnan(kc.astype(np.float32))))
    assert int(changed.any(axis=(1, 3)).sum()) == 2
    assert pk.pkv_read_device_status() == 0


def test_fused_step_at_the_llama8b_size(pk, cuda_device):
    """The step_qkv bench configuration: the Llama-3-8B decode workload's
    pools and tables (32 sequences, contexts up to 2048), each sequence's
    newest token given as its fused projection row; the heuristic split
    count (what the bench times) and a forced split-K."""
    w = W.make("llama8b")
    H, Hkv = w.num_heads, w.num_kv_heads
    lens = w.context_lens.astype(np.int32)
    c = W.qkv_case(7300, H, Hkv, w.head_dim, w.block_size, [1] * w.num_seqs,
                   (lens - 1).tolist())
    kc, vc = W.host_pool(w)
    q_ref, k_rows = Q.qkv_norm_rope_append(c.qkv, c.q_norm_w, c.k_norm_w, c.cos, c.sin, kc, vc,
                                           c.cu_seqlens_q, lens - 1, w.block_tables, H, Hkv,
                                           c.eps)
    ref = oracle.decode_fast(q_ref.astype(np.float16), kc, vc, w.block_tables, lens, w.scale)
    d = W.to_device(w, cuda_device)
    for S in (0, 4):
        kc_d, vc_d = d["k_cache"].clone(), d["v_cache"].clone()
        out = pk.pkv_qkv_norm_rope_append_decode(
            dev(c.qkv, cuda_device), dev(c.q_norm_w, cuda_device), dev(c.k_norm_w, cuda_device),
            dev(c.cos, cuda_device), dev(c.sin, cuda_device), kc_d, vc_d, d["block_tables"],
            d["context_lens"], H, w.scale, eps=c.eps, num_splits=S)
        torch.cuda.synchronize()
        assert_attention_close(out.float().cpu().numpy().astype(np.float64), ref,
                               f"llama8b fused step S={S}")
        got_k = kc_d.cpu().numpy()
        got_v = vc_d.cpu().numpy()
        for s in range(w.num_seqs):
            p = int(lens[s]) - 1
            blk, off = int(w.block_tables[s][p // w.block_size]), p % w.block_size
            assert_within_one_ulp(got_k[blk, :, off], k_rows[s], f"k row of sequence {s}")
            assert_bits_equal(got_v[blk, :, off], vc[blk, :, off], f"v row of sequence {s}")
        assert pk.pkv_read_device_status() == 0
