"""The C-ABI library on the host: it loads, exports every declared symbol,
rejects bad arguments before any CUDA call, and its host-side helpers (split
heuristic, scratch size, status strings) behave as documented.  No GPU."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pagedkv.h")


@pytest.fixture(scope="module")
def pk():
    from paged_kv_decode_08_gb300 import build

    build.build_library()
    from paged_kv_decode_08_gb300 import pagedkv

    return pagedkv


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pkv_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_expected_calls():
    names = declared_functions()
    for n in ["pkv_append", "pkv_decode", "pkv_decode_splitk", "pkv_append_decode",
              "pkv_varlen_attention", "pkv_splitk_scratch_bytes",
              "pkv_pick_num_splits", "pkv_status_string", "pkv_last_error",
              "pkv_read_device_status", "pkv_append_vllm_layout", "pkv_decode_vllm_layout",
              "pkv_varlen_attention_vllm_layout", "pkv_varlen_attention_splitk",
              "pkv_varlen_attention_splitk_vllm_layout", "pkv_varlen_pick_num_splits",
              "pkv_qkv_norm_rope_append", "pkv_qkv_norm_rope_append_decode",
              "pkv_selftest_wait_timeout", "pkv_decode_splitk_plan", "pkv_varlen_splitk_plan",
              "pkv_decode_splitk_noalloc", "pkv_set_varlen_tensor_path"]:
        assert n in names


def test_library_exports_every_declared_symbol(pk):
    lib = ctypes.CDLL(pk.LIB_PATH)
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_status_strings(pk):
    for code in (0, -1, -2, -3, -4, 99):
        s = pk.status_string(code)
        assert isinstance(s, str) and s
    assert pk.status_string(-3).startswith("split-K scratch")


def test_scratch_bytes(pk):
    assert pk.pkv_splitk_scratch_bytes(4, 32, 128, 1) == 0
    assert pk.pkv_splitk_scratch_bytes(0, 32, 128, 4) == 0
    n = pk.pkv_splitk_scratch_bytes(4, 32, 128, 64)
    rows = 4 * 32 * 64
    a = lambda x: (x + 255) // 256 * 256  # noqa: E731
    # a 256-byte header, then f32 partial outputs, maxima and sums
    assert n == 256 + a(rows * 128 * 4) + 2 * a(rows * 4)


@pytest.mark.parametrize("args,expect", [
    # (num_seqs, num_kv_heads, max_context_len, block_size, num_sms) -> splits
    ((2, 2, 48, 16, 152), 1),          # tiny: too short to split
    ((32, 8, 2048, 16, 152), 1),       # Llama-3-8B shape: 256 CTAs are nearest one wave of 304
    ((4, 8, 131072, 16, 152), 10),     # long context: fill 2 CTAs x 152 SMs
    ((256, 4, 16384, 32, 152), 8),     # ragged batch: saturated, cap 2048 tokens per CTA
    ((128, 16, 4352, 16, 152), 3),     # append+decode loop
    ((1, 1, 1 << 20, 16, 152), 64),    # capped at 64
    ((0, 8, 2048, 16, 152), 1),        # invalid -> 1
    ((1, 1, 100, 16, 152), 1),         # shorter than one split's minimum
])
def test_pick_num_splits_table(pk, args, expect):
    assert pk.pkv_pick_num_splits(*args) == expect


def test_decode_splitk_plan(pk):
    """The plan the decode calls follow: forced counts capped at the table
    width, single pass without scratch."""
    assert pk.pkv_decode_splitk_plan(4, 32, 8, 128, 8192, 16, 16) == (
        16, pk.pkv_splitk_scratch_bytes(4, 32, 128, 16))
    assert pk.pkv_decode_splitk_plan(3, 8, 2, 64, 7, 16, 64) == (
        7, pk.pkv_splitk_scratch_bytes(3, 8, 64, 7))
    assert pk.pkv_decode_splitk_plan(4, 32, 8, 128, 8192, 16, 1) == (1, 0)
    assert pk.pkv_decode_splitk_plan(0, 32, 8, 128, 8192, 16, 16) == (16, 0)
    for bad in (dict(num_splits=129), dict(num_splits=-1), dict(num_heads=30),
                dict(max_blocks_per_seq=0)):
        a = dict(num_seqs=4, num_heads=32, num_kv_heads=8, head_dim=128,
                 max_blocks_per_seq=8192, block_size=16, num_splits=4)
        a.update(bad)
        with pytest.raises(pk.PagedKVError) as e:
            pk.pkv_decode_splitk_plan(**a)
        assert e.value.status == pk.PKV_ERR_INVALID_ARG
    S, n = ctypes.c_int32(0), ctypes.c_size_t(0)
    assert pk.lib.pkv_decode_splitk_plan(4, 32, 8, 128, 8192, 16, 4, None, ctypes.byref(n)) == -1
    assert pk.lib.pkv_decode_splitk_plan(4, 32, 8, 128, 8192, 16, 4, ctypes.byref(S), None) == -1


def test_decode_splitk_plan_heuristic_needs_a_device(pk):
    """num_splits = 0 asks the current GPU for its SM count: without one the
    call reports a CUDA error instead of guessing."""
    import torch

    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    with pytest.raises(pk.PagedKVError) as e:
        pk.pkv_decode_splitk_plan(4, 32, 8, 128, 8192, 16, 0)
    assert e.value.status == pk.PKV_ERR_CUDA


def test_varlen_splitk_plan(pk):
    assert pk.pkv_varlen_splitk_plan(4, 16, 4, 32, 8, 128, 8192, 16, 10) == (
        10, pk.pkv_splitk_scratch_bytes(16, 32, 128, 10))
    assert pk.pkv_varlen_splitk_plan(4, 16, 4, 32, 8, 128, 3, 16, 64) == (
        3, pk.pkv_splitk_scratch_bytes(16, 32, 128, 3))
    assert pk.pkv_varlen_splitk_plan(4, 16, 4, 32, 8, 128, 8192, 16, 1) == (1, 0)
    assert pk.pkv_varlen_splitk_plan(4, 0, 0, 32, 8, 128, 8192, 16, 0) == (1, 0)
    with pytest.raises(pk.PagedKVError):
        pk.pkv_varlen_splitk_plan(4, 16, 4, 32, 8, 128, 8192, 16, -1)


def test_varlen_splitk_plan_prefill_sizes_forced(pk):
    """Chunked-prefill sizes (4 x 512 queries, group 4, head_dim 128) with a
    forced split count: that count (at most max_blocks_per_seq) and its
    scratch, with no device query; the pick for num_splits = 0 needs the GPU."""
    assert pk.pkv_varlen_splitk_plan(4, 2048, 512, 32, 8, 128, 160, 16, 3) == (
        3, pk.pkv_splitk_scratch_bytes(2048, 32, 128, 3))
    assert pk.pkv_varlen_splitk_plan(4, 2048, 512, 32, 8, 128, 2, 16, 5) == (
        2, pk.pkv_splitk_scratch_bytes(2048, 32, 128, 2))
    assert pk.pkv_varlen_splitk_plan(4, 2048, 512, 32, 8, 128, 160, 16, 1) == (1, 0)
    with pytest.raises(pk.PagedKVError) as e:
        pk.pkv_varlen_splitk_plan(4, 2048, 512, 32, 8, 128, 160, 16, 0)
    assert e.value.status == pk.PKV_ERR_CUDA


def test_pick_num_splits_never_leaves_a_split_empty_by_length(pk):
    for L in (256, 300, 512, 777, 4096, 65536):
        for base in (1, 4, 32, 300, 2000):
            s = pk.pkv_pick_num_splits(base, 1, L, 16, 152)
            assert 1 <= s <= 64
            assert s <= max(1, L // 256)


NULL = None
F16 = 0x10000  # a fake, 16-byte aligned address; validation rejects before any use


def _decode_args(**over):
    a = dict(q=F16, k=F16, v=F16, bt=F16, cl=F16, B=2, mbps=3, nb=8, scale=0.125, H=4, Hkv=2,
             D=64, bs=16, out=F16)
    a.update(over)
    return a


def _call_decode(pk, a):
    return pk.lib.pkv_decode(a["q"], a["k"], a["v"], a["bt"], a["cl"], a["B"], a["mbps"],
                             a["nb"], a["scale"], a["H"], a["Hkv"], a["D"], a["bs"], a["out"],
                             None)


@pytest.mark.parametrize("over,status", [
    (dict(q=None), -1),
    (dict(out=None), -1),
    (dict(H=6, Hkv=4), -1),          # not a multiple
    (dict(Hkv=0), -1),
    (dict(D=96), -2),
    (dict(bs=8), -2),
    (dict(H=18, Hkv=2), -2),         # group 9
    (dict(B=-1), -1),
    (dict(nb=1 << 28), -1),          # nb * bs overflows int32 slots
    (dict(k=F16 + 8), -1),           # misaligned cache
    (dict(q=F16 + 2), -1),           # misaligned q
    (dict(scale=float("inf")), -1),
    (dict(mbps=0), -1),
])
def test_decode_rejects_bad_arguments_before_cuda(pk, over, status):
    assert _call_decode(pk, _decode_args(**over)) == status
    assert pk.last_error()


def test_decode_with_no_sequences_is_a_no_op(pk):
    assert _call_decode(pk, _decode_args(B=0)) == 0


def test_splitk_rejects_bad_splits_and_small_scratch(pk):
    a = _decode_args(B=4, mbps=8192, nb=24576, H=32, Hkv=8, D=128, bs=16)
    f = pk.lib.pkv_decode_splitk
    args = [a["q"], a["k"], a["v"], a["bt"], a["cl"], a["B"], a["mbps"], a["nb"], a["scale"],
            a["H"], a["Hkv"], a["D"], a["bs"], a["out"]]
    assert f(*args, -2, F16, 1 << 30, None) == -1
    assert f(*args, 129, F16, 1 << 30, None) == -1
    assert f(*args, -1, F16, 1 << 30, None) == -1
    assert f(*args, 16, None, 0, None) == -3
    need = pk.pkv_splitk_scratch_bytes(4, 32, 128, 16)
    assert f(*args, 16, F16, need - 1, None) == -3
    assert "needs" in pk.last_error()


def test_append_rejects_bad_arguments(pk):
    f = pk.lib.pkv_append
    assert f(F16, F16, F16, -1, F16, F16, 8, 16, 2, 64, None) == -1
    assert f(None, F16, F16, 2, F16, F16, 8, 16, 2, 64, None) == -1
    assert f(F16, F16, F16, 2, F16, F16, 8, 16, 2, 80, None) == -2
    assert f(F16, F16, F16, 2, F16, F16, 8, 24, 2, 64, None) == -2
    assert f(F16 + 4, F16, F16, 2, F16, F16, 8, 16, 2, 64, None) == -1
    assert f(F16, F16, F16, 0, F16, F16, 8, 16, 2, 64, None) == 0


def test_noalloc_rejects_oversized_requests_before_any_cuda_call(pk):
    # 256 sequences x 32 heads x 64 splits x 128 dims of f32 partials: 268 MB,
    # far beyond the built-in buffer; rejected on the host, nothing launched.
    f = pk.lib.pkv_decode_splitk_noalloc
    st = f(F16, F16, F16, F16, F16, 256, 8192, 24576, 0.1, 32, 8, 128, 16, F16, 64, None)
    assert st == pk.PKV_ERR_SCRATCH_TOO_SMALL
    assert "built-in buffer" in pk.last_error()
    assert f(F16, F16, F16, F16, F16, 2, 3, 8, 0.1, 4, 2, 64, 16, F16, -2, None) == -1


def test_append_decode_rejects_bad_arguments(pk):
    f = pk.lib.pkv_append_decode
    ok = [F16, F16, F16, F16, F16, F16, F16, F16, 2, 3, 8, 0.125, 4, 2, 64, 16, F16, 0, None, 0,
          None]
    bad_k = list(ok)
    bad_k[0] = None
    assert f(*bad_k) == -1
    misaligned = list(ok)
    misaligned[1] = F16 + 4
    assert f(*misaligned) == -1
    bad_group = list(ok)
    bad_group[12] = 5  # 5 heads over 2 kv heads
    assert f(*bad_group) == -1
    assert f(*(ok[:8] + [0] + ok[9:])) == 0  # no sequences: nothing to do


def test_varlen_rejects_bad_arguments(pk):
    f = pk.lib.pkv_varlen_attention
    ok = [F16, F16, F16, F16, F16, F16, 2, 5, 4, 3, 8, 0.125, 4, 2, 64, 16, F16, None]
    cu_null = list(ok)
    cu_null[3] = None
    assert f(*cu_null) == -1
    neg = list(ok)
    neg[7] = -1
    assert f(*neg) == -1
    assert f(*(ok[:7] + [0] + ok[8:])) == 0  # no queries
    bad_d = list(ok)
    bad_d[14] = 96
    assert f(*bad_d) == -2


def test_vllm_layout_calls_reject_bad_arguments(pk):
    f = pk.lib.pkv_decode_vllm_layout
    ok = [F16, F16, F16, F16, F16, 2, 3, 8, 0.125, 4, 2, 64, 16, F16]
    assert f(*ok, -1, F16, 1 << 30, None) == -1   # no negative split counts
    assert f(*ok, -2, F16, 1 << 30, None) == -1
    assert f(*ok, 4, None, 0, None) == -3
    bad = list(ok)
    bad[11] = 96
    assert f(*bad, 1, None, 0, None) == -2
    assert f(*(ok[:5] + [0] + ok[6:]), 1, None, 0, None) == 0  # no sequences
    a = pk.lib.pkv_append_vllm_layout
    assert a(F16, F16, F16, -1, F16, F16, 8, 16, 2, 64, None) == -1
    assert a(F16, F16, F16, 2, F16, F16, 8, 24, 2, 64, None) == -2
    assert a(F16, F16, F16, 2, F16 + 4, F16, 8, 16, 2, 64, None) == -1
    assert a(F16, F16, F16, 0, F16, F16, 8, 16, 2, 64, None) == 0


def test_vllm_varlen_rejects_bad_arguments(pk):
    f = pk.lib.pkv_varlen_attention_vllm_layout
    ok = [F16, F16, F16, F16, F16, F16, 2, 5, 4, 3, 8, 0.125, 4, 2, 64, 16, F16, None]
    cu_null = list(ok)
    cu_null[3] = None
    assert f(*cu_null) == -1
    assert f(*(ok[:7] + [0] + ok[8:])) == 0  # no queries
    bad_bs = list(ok)
    bad_bs[15] = 24
    assert f(*bad_bs) == -2


@pytest.mark.parametrize("args,expect", [
    ((32, 32, 8, 4, 128, 16, 152), 1),      # speculative verification: one wave already
    ((4, 32, 8, 4, 8192, 16, 152), 10),     # long contexts: 32 CTAs -> nearest one wave
    ((1, 8, 8, 1, 4, 16, 152), 1),          # 64 tokens of capacity: a split keeps >= 256
    ((1, 32, 8, 4, 1 << 20, 16, 152), 38),  # 8 CTAs -> nearest one wave of 304
    ((1, 32, 8, 4, 1 << 20, 16, 1000), 64), # capped at 64
    ((0, 32, 8, 4, 128, 16, 152), 1),       # invalid -> 1
    ((2, 6, 4, 4, 128, 16, 152), 1),        # heads not a multiple of kv heads -> 1
])
def test_varlen_pick_num_splits_table(pk, args, expect):
    assert pk.pkv_varlen_pick_num_splits(*args) == expect


def test_varlen_splitk_rejects_bad_arguments(pk):
    f = pk.lib.pkv_varlen_attention_splitk
    ok = [F16, F16, F16, F16, F16, F16, 2, 5, 4, 3, 8, 0.125, 4, 2, 64, 16, F16]
    assert f(*ok, -1, F16, 1 << 30, None) == -1
    assert f(*ok, 129, F16, 1 << 30, None) == -1
    assert f(*ok, 4, None, 0, None) == -3         # 3 splits of 1 block need scratch
    assert f(*(ok[:7] + [0] + ok[8:]), 4, None, 0, None) == 0  # no queries
    g = pk.lib.pkv_varlen_attention_splitk_vllm_layout
    assert g(*ok, 4, None, 0, None) == -3


def test_header_compiles_as_c99_and_links(pk, tmp_path):
    """A plain C caller: the header is valid C99 without CUDA headers, and the
    library's host-only entry points answer through it."""
    import shutil
    import subprocess

    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    src = os.path.join(ROOT, "tests", "c_abi", "host_calls.c")
    exe = str(tmp_path / "host_calls")
    libdir = os.path.dirname(pk.LIB_PATH)
    build = subprocess.run([gcc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic",
                            "-I", os.path.join(ROOT, "include"), src, "-o", exe,
                            "-L", libdir, "-lpagedkv", "-Wl,-rpath," + libdir],
                           capture_output=True, text=True)
    assert build.returncode == 0, build.stderr
    run = subprocess.run([exe], capture_output=True, text=True, timeout=60)
    assert run.returncode == 0, run.stdout + run.stderr
    assert "all ok" in run.stdout


def test_qkv_norm_rope_rejects_bad_arguments(pk):
    """Every call here is rejected (or has no rows) before any CUDA call."""
    f = pk.lib.pkv_qkv_norm_rope_append
    # qkv, qw, kw, cos, sin, q_out, kc, vc, cu, pos, bt, B, T, MBPS, NB, H, Hkv, D, bs, max_pos, eps
    base = [F16, None, None, F16, F16, F16, F16, F16, F16, F16, F16, 2, 4, 3, 8, 4, 2, 64, 16,
            100, 1e-6]

    def call(**over):
        a = list(base)
        names = ["qkv", "qw", "kw", "cos", "sin", "qo", "kc", "vc", "cu", "pos", "bt", "B", "T",
                 "mbps", "nb", "H", "Hkv", "D", "bs", "max_pos", "eps"]
        for k, v in over.items():
            a[names.index(k)] = v
        return f(*a, None)

    assert call(qkv=None) == -1
    assert call(cos=None) == -1
    assert call(H=6, Hkv=4) == -1
    assert call(D=96) == -2
    assert call(bs=8) == -2
    assert call(max_pos=0) == -1
    assert call(eps=-1.0) == -1
    assert call(eps=float("nan")) == -1
    assert call(qkv=F16 + 2) == -1            # the kernel moves 16-byte words
    assert call(qkv=F16 + 8) == -1
    assert call(qo=F16 + 4) == -1
    assert call(kc=F16 + 4) == -1
    assert call(qw=F16 + 2) == -1
    assert call(cos=F16 + 2) == -1            # misaligned f32
    assert call(sin=F16 + 8) == -1
    assert call(T=0) == 0                      # no rows: nothing launched
    assert call(B=0) == 0


def test_qkv_norm_rope_append_decode_rejects_bad_arguments(pk):
    """Every call here is rejected (or has no sequences) before any CUDA call."""
    f = pk.lib.pkv_qkv_norm_rope_append_decode
    names = ["qkv", "qw", "kw", "cos", "sin", "max_pos", "eps", "kc", "vc", "bt", "cl", "B",
             "mbps", "nb", "scale", "H", "Hkv", "D", "bs", "out", "S", "scratch", "scratch_bytes"]
    base = [F16, None, None, F16, F16, 100, 1e-6, F16, F16, F16, F16, 2, 3, 8, 0.125, 8, 2, 128,
            16, F16, 0, None, 0]

    def call(**over):
        a = list(base)
        for k, v in over.items():
            a[names.index(k)] = v
        return f(*a, None)

    assert call(qkv=None) == -1
    assert call(cos=None) == -1
    assert call(sin=None) == -1
    assert call(out=None) == -1
    assert call(H=6, Hkv=4) == -1
    assert call(H=32, Hkv=2) == -2             # group 16
    assert call(D=96) == -2
    assert call(bs=8) == -2
    assert call(max_pos=0) == -1
    assert call(eps=-1.0) == -1
    assert call(eps=float("inf")) == -1
    assert call(scale=float("nan")) == -1
    assert call(qkv=F16 + 2) == -1            # half2 loads need 4-byte alignment
    assert call(kc=F16 + 4) == -1             # tensor copies need 16-byte pools
    assert call(qw=F16 + 1) == -1
    assert call(cos=F16 + 2) == -1
    assert call(S=-1) == -1                    # no negative split counts
    assert call(S=pk.PKV_MAX_SPLITS + 1) == -1
    assert call(B=0) == 0                      # no sequences: nothing launched
