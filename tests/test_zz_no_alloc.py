"""The split-K decode entry point that allocates nothing.

Some callers may not allocate device memory at all: a plugin or extension
whose host owns every allocation and hands it only the input and output
buffers, or a decode loop under a latency budget where cudaMalloc (which can
block and synchronize the device) is not allowed.  For them,
``pkv_decode_splitk_noalloc`` keeps the split-K partials in a static device
buffer built into the library instead of caller scratch.

The test calls it through the C ABI and checks its output against
``pkv_decode_splitk`` with caller-owned scratch, within the attention
tolerance of the other parity tests, on two calls in a row: the second call
has a different shape and split count, so partials left behind by the first
call would show if they were read.

The file name makes pytest collect it last.
"""

import numpy as np
import pytest

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


def test_noalloc_matches_caller_scratch_on_two_calls_in_a_row(cuda_device):
    from paged_kv_decode_08_gb300 import pagedkv as pk

    pk.pkv_read_device_status()
    cases = [
        (W.small_random(901, num_seqs=8, num_heads=32, num_kv_heads=8, head_dim=128,
                        block_size=16, lens=[4096, 1, 777, 2048, 3000, 16, 4095, 1500]), 16),
        (W.small_random(902, num_seqs=5, num_heads=28, num_kv_heads=4, head_dim=64,
                        block_size=32, lens=[100, 2000, 33, 1, 640]), 3),
    ]
    for w, S in cases:
        need = pk.pkv_splitk_scratch_bytes(w.num_seqs, w.num_heads, w.head_dim, S)
        assert 0 < need <= pk.PKV_NOALLOC_SCRATCH_BYTES
        d = W.to_device(w, cuda_device)
        scratch = pk.alloc_scratch(d["q"], d["k_cache"], d["block_tables"], S)
        ref = torch.empty_like(d["q"])
        pk.pkv_decode_splitk(d["q"], d["k_cache"], d["v_cache"], d["block_tables"],
                             d["context_lens"], w.scale, num_splits=S, scratch=scratch, out=ref)
        out = torch.full_like(d["q"], float("nan"))
        status = _noalloc_raw(pk, w, d, out, S)
        assert status == pk.PKV_OK, pk.last_error()
        torch.cuda.synchronize()
        got = out.float().cpu().numpy().astype(np.float64)
        exp = ref.float().cpu().numpy().astype(np.float64)
        assert np.all(np.isfinite(got))
        assert_attention_close(got, exp, f"no-alloc vs caller scratch, S={S}")
    assert pk.pkv_read_device_status() == 0


def test_noalloc_rejects_requests_beyond_its_buffer(cuda_device):
    from paged_kv_decode_08_gb300 import pagedkv as pk

    # 32 blocks per sequence and 16 splits: 64 x 32 x 16 x 128 f32 partials
    # (16.8 MB) do not fit the 8 MiB buffer.
    w = W.small_random(903, num_seqs=64, num_heads=32, num_kv_heads=8, head_dim=128,
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
