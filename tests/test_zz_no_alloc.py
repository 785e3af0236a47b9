"""The split-K decode entry point that allocates nothing.

Some callers may not allocate device memory at all: a plugin or extension
whose host owns every allocation and hands it only the input and output
buffers, or a decode loop under a latency budget where cudaMalloc (which can
block and synchronize the device) is not allowed.  For them,
``pkv_decode_splitk_noalloc`` keeps the split-K partials in a static device
buffer built into the library instead of caller scratch.

The test calls it through the C ABI, one call after another on the same
stream, and checks every output element against the float64 oracle (the
attention tolerance of the other parity tests) and against
``pkv_decode_splitk`` with caller-owned scratch.  The calls cover forced
split counts, the heuristic (0) and a forced count above the table width
(launched as max_blocks_per_seq splits); each
call has a different shape or split count from the one before, so partials
left in the shared buffer by an earlier call would show if they were read.

The file name makes pytest collect it last.
"""

import numpy as np
import pytest

import oracle
from paged_kv_decode_08_gb300 import workloads as W
from tests.tolerance import assert_attention_close

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


def _noalloc_raw(pk, w, d, out, num_splits):
    """One call of the entry point through the raw C ABI."""
    return pk.lib.pkv_decode_splitk_noalloc(
        d["q"].data_ptr(), d["k_cache"].data_ptr(), d["v_cache"].data_ptr(),
        d["block_tables"].data_ptr(), d["context_lens"].data_ptr(), w.num_seqs,
        w.max_blocks_per_seq, w.num_blocks, float(w.scale), w.num_heads, w.num_kv_heads,
        w.head_dim, w.block_size, out.data_ptr(), num_splits,
        torch.cuda.current_stream().cuda_stream)


def _case(seed, H, Hkv, D, bs, lens):
    w = W.small_random(seed, num_seqs=len(lens), num_heads=H, num_kv_heads=Hkv, head_dim=D,
                       block_size=bs, lens=lens)
    kc, vc = W.host_pool(w)
    ref = oracle.decode(w.q, kc, vc, w.block_tables, w.context_lens, w.scale)
    return w, ref


def test_noalloc_matches_the_oracle_on_calls_in_a_row(cuda_device):
    from paged_kv_decode_08_gb300 import pagedkv as pk

    pk.pkv_read_device_status()
    a = _case(901, 32, 8, 128, 16, [4096, 1, 777, 2048, 3000, 16, 4095, 1500])
    b = _case(902, 28, 4, 64, 32, [100, 2000, 33, 1, 640])
    c = _case(903, 8, 2, 64, 16, [100, 37, 5])  # 7 table blocks: S = 64 runs as 7 splits
    calls = [(a, 16), (b, 3), (a, 0), (b, 0), (c, 64), (b, 7), (a, 16)]
    for (w, ref), S in calls:
        S_run, need = pk.pkv_decode_splitk_plan(w.num_seqs, w.num_heads, w.num_kv_heads,
                                                w.head_dim, w.max_blocks_per_seq, w.block_size,
                                                S)
        assert S_run != 1 and 0 < need <= pk.PKV_NOALLOC_SCRATCH_BYTES, (S, S_run, need)
        if S == 64:
            assert S_run == w.max_blocks_per_seq
        d = W.to_device(w, cuda_device)
        out = torch.full_like(d["q"], float("nan"))
        status = _noalloc_raw(pk, w, d, out, S)
        assert status == pk.PKV_OK, pk.last_error()
        caller = pk.pkv_decode_splitk(d["q"], d["k_cache"], d["v_cache"], d["block_tables"],
                                      d["context_lens"], w.scale, num_splits=S)
        torch.cuda.synchronize()
        got = out.float().cpu().numpy().astype(np.float64)
        assert np.all(np.isfinite(got))
        assert_attention_close(got, ref, f"no-alloc vs oracle, S={S}")
        assert_attention_close(got, caller.float().cpu().numpy().astype(np.float64),
                               f"no-alloc vs caller scratch, S={S}")
    assert pk.pkv_read_device_status() == 0


def test_noalloc_rejects_requests_beyond_its_buffer(cuda_device):
    from paged_kv_decode_08_gb300 import pagedkv as pk

    # 32 blocks per sequence and 16 splits: 64 x 32 x 16 x 128 f32 partials
    # (16.8 MB) do not fit the 8 MiB buffer.
    w = W.small_random(904, num_seqs=64, num_heads=32, num_kv_heads=8, head_dim=128,
                       block_size=16, lens=[512] * 64)
    d = W.to_device(w, cuda_device)
    out = torch.zeros_like(d["q"])
    assert w.max_blocks_per_seq == 32
    assert pk.pkv_splitk_scratch_bytes(64, 32, 128, 16) > pk.PKV_NOALLOC_SCRATCH_BYTES
    status = _noalloc_raw(pk, w, d, out, 16)
    assert status == pk.PKV_ERR_SCRATCH_TOO_SMALL
    assert "built-in buffer" in pk.last_error()
    torch.cuda.synchronize()
    assert torch.count_nonzero(out).item() == 0  # nothing was launched
