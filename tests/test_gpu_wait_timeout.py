"""The failure path on the GPU, without a fault: a wait that nothing will
satisfy gives up after its 100 ms limit, flags PKV_DEV_WAIT_TIMEOUT and
returns; while the flag is set every decode and varlen call (combine kernels
and the tcgen05 varlen kernel included) writes nothing; reading the status clears it and the next calls
are correct again (the context stayed usable)."""

import time

import numpy as np
import pytest

import oracle
from paged_kv_decode_08_gb300 import workloads as W
from tests.tolerance import assert_attention_close

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def pk(cuda_device):
    from paged_kv_decode_08_gb300 import pagedkv

    pagedkv.pkv_read_device_status()
    return pagedkv


def test_wait_timeout_is_flagged_and_nothing_is_written_until_cleared(pk, cuda_device):
    w = W.small_random(301, num_seqs=3, num_heads=8, num_kv_heads=2, head_dim=128,
                       block_size=16, lens=[40, 300, 7])
    d = W.to_device(w, cuda_device)
    v = W.varlen_random(302, 8, 2, 128, 16, [3, 2], [50, 200])
    dv = W.to_device(v.base, cuda_device)
    vq = torch.from_numpy(v.q).to(cuda_device)
    cu = torch.from_numpy(v.cu_seqlens_q).to(cuda_device)
    pos = torch.from_numpy(v.pos_offsets).to(cuda_device)
    sentinel = 7.0
    try:
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        pk.pkv_selftest_wait_timeout()
        torch.cuda.synchronize()
        assert time.perf_counter() - t0 >= 0.09  # the wait ran to its limit

        outs = [torch.full_like(d["q"], sentinel) for _ in range(2)]
        pk.pkv_decode(d["q"], d["k_cache"], d["v_cache"], d["block_tables"], d["context_lens"],
                      w.scale, out=outs[0])
        pk.pkv_decode_splitk(d["q"], d["k_cache"], d["v_cache"], d["block_tables"],
                             d["context_lens"], w.scale, num_splits=3, out=outs[1])
        # varlen on both kernels (12 columns per CTA: the tcgen05 one when selected)
        vouts = [torch.full_like(vq, sentinel) for _ in range(4)]
        prev = pk.pkv_set_varlen_tensor_path(0)
        try:
            for path in (0, 1):
                pk.pkv_set_varlen_tensor_path(path)
                pk.pkv_varlen_attention(vq, dv["k_cache"], dv["v_cache"], cu, pos,
                                        dv["block_tables"], v.base.scale, max_q_len=3,
                                        out=vouts[2 * path])
                pk.pkv_varlen_attention_splitk(vq, dv["k_cache"], dv["v_cache"], cu, pos,
                                               dv["block_tables"], v.base.scale, max_q_len=3,
                                               num_splits=4, out=vouts[2 * path + 1])
        finally:
            pk.pkv_set_varlen_tensor_path(prev)
        torch.cuda.synchronize()
        for i, o in enumerate(outs + vouts):
            assert bool((o == sentinel).all()), f"call {i} wrote while the timeout flag was set"

        flags = pk.pkv_read_device_status()  # reads and clears
        assert flags & pk.PKV_DEV_WAIT_TIMEOUT

        kc, vc = W.host_pool(w)
        ref = oracle.decode(w.q, kc, vc, w.block_tables, w.context_lens, w.scale)
        for S in (1, 3):
            got = pk.pkv_decode_splitk(d["q"], d["k_cache"], d["v_cache"], d["block_tables"],
                                       d["context_lens"], w.scale, num_splits=S)
            torch.cuda.synchronize()
            assert_attention_close(got.float().cpu().numpy().astype(np.float64), ref,
                                   f"after clearing, S={S}")
        assert pk.pkv_read_device_status() == 0
    finally:
        torch.cuda.synchronize()
        pk.pkv_read_device_status()
