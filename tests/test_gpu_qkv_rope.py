"""GPU parity of pkv_qkv_norm_rope_append (fused QKV split + per-head RMS
norm + rotary embedding + paged append) against the CPU oracle, through the
C ABI.

Queries and keys must be within one f16 ulp of the float64 result rounded to
f16 (the kernel computes in f32 and rounds once); values are copied bit for
bit; pool entries the step does not write keep their NaN poison."""

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
    assert not bad.any(), f"{what}: {int(bad.sum())} elements off by more than one ulp, first at {np.argwhere(bad)[0]}"


def device_inputs(c, dev):
    t = lambda a: None if a is None else torch.from_numpy(np.ascontiguousarray(a)).to(dev)  # noqa: E731
    return dict(qkv=t(c.qkv), q_norm_w=t(c.q_norm_w), k_norm_w=t(c.k_norm_w), cos=t(c.cos),
                sin=t(c.sin), cu=t(c.cu_seqlens_q), pos=t(c.pos_offsets), bt=t(c.block_tables))


def nan_pools(c, dev):
    shape = (c.num_blocks, c.num_kv_heads, c.block_size, c.head_dim)
    return (torch.full(shape, float("nan"), dtype=torch.float16, device=dev),
            torch.full(shape, float("nan"), dtype=torch.float16, device=dev))


def run_oracle(c):
    shape = (c.num_blocks, c.num_kv_heads, c.block_size, c.head_dim)
    kc = np.full(shape, np.nan, np.float16)
    vc = np.full(shape, np.nan, np.float16)
    q_out, k_rows = Q.qkv_norm_rope_append(c.qkv, c.q_norm_w, c.k_norm_w, c.cos, c.sin, kc, vc,
                                           c.cu_seqlens_q, c.pos_offsets, c.block_tables,
                                           c.num_heads, c.num_kv_heads, c.eps)
    return q_out, k_rows, kc, vc


def slots_of(c):
    out = []
    for s in range(len(c.pos_offsets)):
        for t in range(int(c.cu_seqlens_q[s + 1] - c.cu_seqlens_q[s])):
            p = int(c.pos_offsets[s]) + t
            out.append((int(c.block_tables[s][p // c.block_size]), p % c.block_size))
    return out


@pytest.mark.parametrize("H,Hkv,D,bs,q_lens,prefix,norm", [
    (32, 8, 128, 16, [1] * 6, [100, 2047, 5, 0, 16, 31], True),   # a decode step
    (8, 8, 64, 32, [5, 17, 1], [0, 40, 300], False),             # prefill chunks, no norm
    (28, 4, 128, 32, [3, 3], [31, 1000], True),
    (16, 2, 64, 16, [9, 2], [7, 60], True),
    # the kernel's slots per warp follow the head count: 48 heads of 64
    # take 2, 64 heads of 128 and 128 heads of 64 take 4
    (32, 8, 64, 16, [4, 3], [10, 100], True),
    (32, 16, 128, 16, [2, 5], [33, 0], True),
    (64, 32, 64, 32, [3], [47], True),
])
def test_qkv_norm_rope_append_matches_oracle(pk, cuda_device, H, Hkv, D, bs, q_lens, prefix,
                                             norm):
    c = W.qkv_case(6000 + H + D + bs, H, Hkv, D, bs, q_lens, prefix, norm=norm)
    q_ref, k_ref, kc_ref, vc_ref = run_oracle(c)
    d = device_inputs(c, cuda_device)
    kc, vc = nan_pools(c, cuda_device)
    q_out = pk.pkv_qkv_norm_rope_append(d["qkv"], d["q_norm_w"], d["k_norm_w"], d["cos"],
                                        d["sin"], kc, vc, d["cu"], d["pos"], d["bt"], H,
                                        eps=c.eps)
    torch.cuda.synchronize()
    assert_within_one_ulp(q_out.cpu().numpy(), q_ref, "q_out")
    got_k = kc.cpu().numpy()
    got_v = vc.cpu().numpy()
    for row, (blk, off) in enumerate(slots_of(c)):
        assert_within_one_ulp(got_k[blk, :, off], k_ref[row], f"k row {row}")
        assert_bits_equal(got_v[blk, :, off], vc_ref[blk, :, off], f"v row {row}")
    # nothing else was written
    assert np.isnan(got_k.astype(np.float32)).sum() == np.isnan(kc_ref.astype(np.float32)).sum()
    assert np.isnan(got_v.astype(np.float32)).sum() == np.isnan(vc_ref.astype(np.float32)).sum()
    assert pk.pkv_read_device_status() == 0


def test_qkv_bad_block_and_position_are_flagged_and_skipped(pk, cuda_device):
    c = W.qkv_case(6100, 8, 2, 128, 16, [2, 2], [20, 40])
    d = device_inputs(c, cuda_device)
    kc, vc = nan_pools(c, cuda_device)
    bt = c.block_tables.copy()
    bt[0, :] = c.num_blocks + 7  # sequence 0: every entry out of range
    d["bt"] = torch.from_numpy(bt).to(cuda_device)
    q_out = torch.full((4, 8, 128), 3.0, dtype=torch.float16, device=cuda_device)
    pk.pkv_qkv_norm_rope_append(d["qkv"], d["q_norm_w"], d["k_norm_w"], d["cos"], d["sin"], kc, vc,
                                d["cu"], d["pos"], d["bt"], 8, eps=c.eps, q_out=q_out)
    torch.cuda.synchronize()
    assert pk.pkv_read_device_status() & pk.PKV_DEV_BAD_BLOCK_ID
    # sequence 1's rows landed; sequence 0 wrote queries but no cache rows
    assert int((~torch.isnan(kc.float())).sum()) == 2 * 2 * 128
    q_ref, _, _, _ = run_oracle(c)
    assert_within_one_ulp(q_out.cpu().numpy(), q_ref, "q_out with a bad table")
    # a position past the tables: the row is skipped entirely
    pos = torch.tensor([20, c.cos.shape[0]], dtype=torch.int32, device=cuda_device)
    q_out.fill_(3.0)
    pk.pkv_qkv_norm_rope_append(d["qkv"], d["q_norm_w"], d["k_norm_w"], d["cos"], d["sin"], kc, vc,
                                d["cu"], pos, d["bt"], 8, eps=c.eps, q_out=q_out)
    torch.cuda.synchronize()
    assert pk.pkv_read_device_status() & pk.PKV_DEV_BAD_CONTEXT_LEN
    assert bool((q_out[2:] == 3.0).all())


def test_qkv_step_then_decode_matches_oracle(pk, cuda_device):
    """A whole decode step: the fused projection rows of each sequence's new
    token go through pkv_qkv_norm_rope_append (keys and values appended after
    a random earlier context), then pkv_decode attends with the rotated
    queries."""
    H, Hkv, D, bs = 32, 8, 128, 16
    prefix = [300, 17, 1023, 64, 0, 511]
    c = W.qkv_case(6200, H, Hkv, D, bs, [1] * 6, prefix)
    rng = np.random.default_rng(6201)
    shape = (c.num_blocks, Hkv, bs, D)
    kc_h = np.full(shape, np.nan, np.float16)
    vc_h = np.full(shape, np.nan, np.float16)
    for s, p0 in enumerate(prefix):  # the earlier context, positions 0 .. p0 - 1
        for p in range(p0):
            blk = int(c.block_tables[s][p // bs])
            kc_h[blk, :, p % bs] = rng.standard_normal((Hkv, D)).astype(np.float16)
            vc_h[blk, :, p % bs] = rng.standard_normal((Hkv, D)).astype(np.float16)
    kc = torch.from_numpy(kc_h).to(cuda_device)
    vc = torch.from_numpy(vc_h).to(cuda_device)
    q_ref, _ = Q.qkv_norm_rope_append(c.qkv, c.q_norm_w, c.k_norm_w, c.cos, c.sin, kc_h, vc_h,
                                      c.cu_seqlens_q, c.pos_offsets, c.block_tables, H, Hkv,
                                      c.eps)
    lens = (c.pos_offsets + 1).astype(np.int32)
    ref = oracle.decode(q_ref.astype(np.float16), kc_h, vc_h, c.block_tables, lens,
                        1.0 / np.sqrt(D))
    d = device_inputs(c, cuda_device)
    q_out = pk.pkv_qkv_norm_rope_append(d["qkv"], d["q_norm_w"], d["k_norm_w"], d["cos"],
                                        d["sin"], kc, vc, d["cu"], d["pos"], d["bt"], H,
                                        eps=c.eps)
    out = pk.pkv_decode(q_out, kc, vc, d["bt"], torch.from_numpy(lens).to(cuda_device),
                        1.0 / np.sqrt(D))
    torch.cuda.synchronize()
    assert_attention_close(out.float().cpu().numpy().astype(np.float64), ref, "qkv step + decode")
    assert pk.pkv_read_device_status() == 0
