"""Python binding of libpagedkv: the C-ABI calls under the same names.

Argument marshalling only: every step of the path runs in the CUDA library.
There is no fallback; if ``libpagedkv.so`` is missing or does not load, the
import fails with an error that says how to build it.

The tensor-level wrappers take torch CUDA tensors, check dtype, shape,
device and contiguity, and pass ``data_ptr()`` plus the current torch stream
(or the one given).  :data:`lib` exposes the raw ``ctypes`` functions for
callers that manage their own pointers.
"""

from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpagedkv.so")

PKV_OK = 0
PKV_ERR_INVALID_ARG = -1
PKV_ERR_UNSUPPORTED = -2
PKV_ERR_SCRATCH_TOO_SMALL = -3
PKV_ERR_CUDA = -4

PKV_DEV_BAD_SLOT = 0x1
PKV_DEV_BAD_BLOCK_ID = 0x2
PKV_DEV_BAD_CONTEXT_LEN = 0x4
PKV_DEV_WAIT_TIMEOUT = 0x8

PKV_MAX_SPLITS = 128
PKV_NOALLOC_SCRATCH_BYTES = 8 * 1024 * 1024


class PagedKVError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{message} (status {status})")
        self.status = status


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is not built; run `python -c 'import __graft_entry__ as g; g.build()'` "
            "or `python paged_kv_decode_08_gb300/build.py`")
    lib = ctypes.CDLL(LIB_PATH)
    vp, i32, sz, f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t, ctypes.c_float
    lib.pkv_append.argtypes = [vp, vp, vp, i32, vp, vp, i32, i32, i32, i32, vp]
    lib.pkv_append.restype = i32
    lib.pkv_decode.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, f32, i32, i32, i32, i32, vp, vp]
    lib.pkv_decode.restype = i32
    lib.pkv_decode_splitk.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, f32, i32, i32, i32, i32,
                                      vp, i32, vp, sz, vp]
    lib.pkv_decode_splitk.restype = i32
    lib.pkv_append_decode.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, f32, i32,
                                      i32, i32, i32, vp, i32, vp, sz, vp]
    lib.pkv_append_decode.restype = i32
    lib.pkv_varlen_attention.argtypes = [vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, f32, i32,
                                         i32, i32, i32, vp, vp]
    lib.pkv_varlen_attention.restype = i32
    lib.pkv_varlen_attention_vllm_layout.argtypes = lib.pkv_varlen_attention.argtypes
    lib.pkv_varlen_attention_vllm_layout.restype = i32
    split_args = lib.pkv_varlen_attention.argtypes[:-1] + [i32, vp, sz, vp]
    lib.pkv_varlen_attention_splitk.argtypes = split_args
    lib.pkv_varlen_attention_splitk.restype = i32
    lib.pkv_varlen_attention_splitk_vllm_layout.argtypes = split_args
    lib.pkv_varlen_attention_splitk_vllm_layout.restype = i32
    lib.pkv_set_varlen_tensor_path.argtypes = [i32]
    lib.pkv_set_varlen_tensor_path.restype = i32
    lib.pkv_decode_splitk_noalloc.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, f32, i32, i32,
                                              i32, i32, vp, i32, vp]
    lib.pkv_decode_splitk_noalloc.restype = i32
    lib.pkv_append_vllm_layout.argtypes = [vp, vp, vp, i32, vp, vp, i32, i32, i32, i32, vp]
    lib.pkv_append_vllm_layout.restype = i32
    lib.pkv_decode_vllm_layout.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, f32, i32, i32, i32,
                                           i32, vp, i32, vp, sz, vp]
    lib.pkv_decode_vllm_layout.restype = i32
    lib.pkv_varlen_pick_num_splits.argtypes = [i32, i32, i32, i32, i32, i32, i32]
    lib.pkv_varlen_pick_num_splits.restype = i32
    lib.pkv_splitk_scratch_bytes.argtypes = [i32, i32, i32, i32]
    lib.pkv_splitk_scratch_bytes.restype = sz
    lib.pkv_pick_num_splits.argtypes = [i32, i32, i32, i32, i32]
    lib.pkv_pick_num_splits.restype = i32
    lib.pkv_decode_splitk_plan.argtypes = [i32, i32, i32, i32, i32, i32, i32,
                                           ctypes.POINTER(i32), ctypes.POINTER(sz)]
    lib.pkv_decode_splitk_plan.restype = i32
    lib.pkv_varlen_splitk_plan.argtypes = [i32, i32, i32, i32, i32, i32, i32, i32, i32,
                                           ctypes.POINTER(i32), ctypes.POINTER(sz)]
    lib.pkv_varlen_splitk_plan.restype = i32
    lib.pkv_status_string.argtypes = [i32]
    lib.pkv_status_string.restype = ctypes.c_char_p
    lib.pkv_last_error.argtypes = []
    lib.pkv_last_error.restype = ctypes.c_char_p
    lib.pkv_qkv_norm_rope_append.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i32,
                                             i32, i32, i32, i32, i32, i32, i32, f32, vp]
    lib.pkv_qkv_norm_rope_append.restype = i32
    lib.pkv_qkv_norm_rope_append_decode.argtypes = [vp, vp, vp, vp, vp, i32, f32, vp, vp, vp, vp,
                                                    i32, i32, i32, f32, i32, i32, i32, i32, vp,
                                                    i32, vp, sz, vp]
    lib.pkv_qkv_norm_rope_append_decode.restype = i32
    lib.pkv_selftest_wait_timeout.argtypes = [vp]
    lib.pkv_selftest_wait_timeout.restype = i32
    lib.pkv_read_device_status.argtypes = [ctypes.POINTER(ctypes.c_int32), vp]
    lib.pkv_read_device_status.restype = i32
    return lib


lib = _load()


def _check(status: int, what: str):
    if status != PKV_OK:
        msg = lib.pkv_last_error().decode(errors="replace")
        raise PagedKVError(status, f"{what}: {lib.pkv_status_string(status).decode()}: {msg}")


def status_string(status: int) -> str:
    return lib.pkv_status_string(status).decode()


def last_error() -> str:
    return lib.pkv_last_error().decode(errors="replace")


def _stream_ptr(stream):
    import torch

    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _want(t, name, dtype, ndim=None, shape=None):
    import torch

    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got {tuple(t.shape)}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


def pkv_append(k, v, slot_mapping, k_cache, v_cache, stream=None):
    """Write ``k``/``v`` rows ``[T][Hkv][D]`` into the pools at ``slot_mapping``."""
    import torch

    _want(k_cache, "k_cache", torch.float16, 4)
    NB, Hkv, bs, D = k_cache.shape
    _want(v_cache, "v_cache", torch.float16, 4, k_cache.shape)
    _want(k, "k", torch.float16, 3)
    T = k.shape[0]
    _want(k, "k", torch.float16, 3, (T, Hkv, D))
    _want(v, "v", torch.float16, 3, (T, Hkv, D))
    _want(slot_mapping, "slot_mapping", torch.int32, 1, (T,))
    _check(lib.pkv_append(k.data_ptr(), v.data_ptr(), slot_mapping.data_ptr(), T,
                          k_cache.data_ptr(), v_cache.data_ptr(), NB, bs, Hkv, D,
                          _stream_ptr(stream)), "pkv_append")


def _decode_shapes(q, k_cache, v_cache, block_tables, context_lens, out):
    import torch

    _want(q, "q", torch.float16, 3)
    B, H, D = q.shape
    _want(k_cache, "k_cache", torch.float16, 4)
    NB, Hkv, bs, Dk = k_cache.shape
    if Dk != D:
        raise ValueError("k_cache head_dim differs from q")
    _want(v_cache, "v_cache", torch.float16, 4, k_cache.shape)
    _want(block_tables, "block_tables", torch.int32, 2)
    if block_tables.shape[0] != B:
        raise ValueError("block_tables must have num_seqs rows")
    _want(context_lens, "context_lens", torch.int32, 1, (B,))
    if out is None:
        out = torch.empty_like(q)
    _want(out, "out", torch.float16, 3, (B, H, D))
    return B, H, D, NB, Hkv, bs, block_tables.shape[1], out


def pkv_decode(q, k_cache, v_cache, block_tables, context_lens, scale, out=None, stream=None):
    """Single-pass paged decode; returns ``out`` ``[B][H][D]`` f16."""
    B, H, D, NB, Hkv, bs, mbps, out = _decode_shapes(q, k_cache, v_cache, block_tables,
                                                     context_lens, out)
    _check(lib.pkv_decode(q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
                          block_tables.data_ptr(), context_lens.data_ptr(), B, mbps, NB,
                          float(scale), H, Hkv, D, bs, out.data_ptr(), _stream_ptr(stream)),
           "pkv_decode")
    return out


def pkv_splitk_scratch_bytes(num_seqs, num_heads, head_dim, num_splits) -> int:
    return int(lib.pkv_splitk_scratch_bytes(num_seqs, num_heads, head_dim, num_splits))


def pkv_pick_num_splits(num_seqs, num_kv_heads, max_context_len, block_size, num_sms) -> int:
    return int(lib.pkv_pick_num_splits(num_seqs, num_kv_heads, max_context_len, block_size,
                                       num_sms))


def pkv_decode_splitk_plan(num_seqs, num_heads, num_kv_heads, head_dim, max_blocks_per_seq,
                           block_size, num_splits=0):
    """``(splits, scratch_bytes)`` the decode calls launch for these sizes (the
    library's own rule; ``num_splits`` 0 = the heuristic for the current GPU)."""
    S = ctypes.c_int32(0)
    n = ctypes.c_size_t(0)
    _check(lib.pkv_decode_splitk_plan(num_seqs, num_heads, num_kv_heads, head_dim,
                                      max_blocks_per_seq, block_size, int(num_splits),
                                      ctypes.byref(S), ctypes.byref(n)), "pkv_decode_splitk_plan")
    return int(S.value), int(n.value)


def pkv_varlen_splitk_plan(num_seqs, total_q, max_q_len, num_heads, num_kv_heads, head_dim,
                           max_blocks_per_seq, block_size, num_splits=0):
    """``(splits, scratch_bytes)`` the varlen split-K calls launch."""
    S = ctypes.c_int32(0)
    n = ctypes.c_size_t(0)
    _check(lib.pkv_varlen_splitk_plan(num_seqs, total_q, max_q_len, num_heads, num_kv_heads,
                                      head_dim, max_blocks_per_seq, block_size, int(num_splits),
                                      ctypes.byref(S), ctypes.byref(n)), "pkv_varlen_splitk_plan")
    return int(S.value), int(n.value)


def _pool_dims(k_cache):
    """(num_kv_heads, block_size) of a blocked [NB][Hkv][bs][D] or vLLM-layout
    [NB][Hkv][D/8][bs][8] K pool."""
    return k_cache.shape[1], (k_cache.shape[3] if k_cache.dim() == 5 else k_cache.shape[2])


def _decode_plan(q, k_cache, block_tables, num_splits, device=None):
    import torch

    Hkv, bs = _pool_dims(k_cache)
    with torch.cuda.device(device or q.device):
        return pkv_decode_splitk_plan(q.shape[0], q.shape[1], Hkv, q.shape[2],
                                      block_tables.shape[1], bs, num_splits)


def splits_for(q, k_cache, block_tables, num_splits=0, device=None) -> int:
    """The split count :func:`pkv_decode_splitk` launches for these tensors."""
    return _decode_plan(q, k_cache, block_tables, num_splits, device)[0]


def alloc_scratch(q, k_cache, block_tables, num_splits=0):
    """A scratch tensor (uint8, on q's device) of the size the library's plan
    gives for these tensors and ``num_splits`` (0 = the heuristic)."""
    import torch

    n = _decode_plan(q, k_cache, block_tables, num_splits)[1]
    return torch.empty(max(n, 16), dtype=torch.uint8, device=q.device)


def pkv_decode_splitk(q, k_cache, v_cache, block_tables, context_lens, scale, num_splits=0,
                      scratch=None, out=None, stream=None):
    """Split-K paged decode (``num_splits`` 0 = heuristic); returns ``out``."""
    import torch

    B, H, D, NB, Hkv, bs, mbps, out = _decode_shapes(q, k_cache, v_cache, block_tables,
                                                     context_lens, out)
    if scratch is None:
        scratch = alloc_scratch(q, k_cache, block_tables, num_splits)
    _want(scratch, "scratch", torch.uint8, 1)
    _check(lib.pkv_decode_splitk(q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
                                 block_tables.data_ptr(), context_lens.data_ptr(), B, mbps, NB,
                                 float(scale), H, Hkv, D, bs, out.data_ptr(), int(num_splits),
                                 scratch.data_ptr(), scratch.numel(), _stream_ptr(stream)),
           "pkv_decode_splitk")
    return out


def pkv_append_decode(k_new, v_new, slot_mapping, k_cache, v_cache, q, block_tables,
                      context_lens, scale, num_splits=0, scratch=None, out=None, stream=None):
    """One decode step: append row s of ``k_new``/``v_new`` (sequence s's newest
    token) at ``slot_mapping[s]`` and decode; returns ``out``."""
    import torch

    B, H, D, NB, Hkv, bs, mbps, out = _decode_shapes(q, k_cache, v_cache, block_tables,
                                                     context_lens, out)
    _want(k_new, "k_new", torch.float16, 3, (B, Hkv, D))
    _want(v_new, "v_new", torch.float16, 3, (B, Hkv, D))
    _want(slot_mapping, "slot_mapping", torch.int32, 1, (B,))
    if scratch is None:
        scratch = alloc_scratch(q, k_cache, block_tables, num_splits)
    _want(scratch, "scratch", torch.uint8, 1)
    _check(lib.pkv_append_decode(k_new.data_ptr(), v_new.data_ptr(), slot_mapping.data_ptr(),
                                 k_cache.data_ptr(), v_cache.data_ptr(), q.data_ptr(),
                                 block_tables.data_ptr(), context_lens.data_ptr(), B, mbps, NB,
                                 float(scale), H, Hkv, D, bs, out.data_ptr(), int(num_splits),
                                 scratch.data_ptr(), scratch.numel(), _stream_ptr(stream)),
           "pkv_append_decode")
    return out


def pkv_varlen_attention(q, k_cache, v_cache, cu_seqlens_q, pos_offsets, block_tables, scale,
                         max_q_len=None, out=None, stream=None):
    """Causal attention of several query tokens per sequence (token-major
    ``q [total_q][H][D]``, ``cu_seqlens_q [B+1]``, ``pos_offsets [B]``)."""
    return _varlen(q, k_cache, v_cache, cu_seqlens_q, pos_offsets, block_tables, scale,
                   max_q_len, out, stream, vllm=False)


def pkv_varlen_attention_vllm_layout(q, k_cache, v_cache, cu_seqlens_q, pos_offsets,
                                     block_tables, scale, max_q_len=None, out=None, stream=None):
    """:func:`pkv_varlen_attention` over vLLM-layout pools."""
    return _varlen(q, k_cache, v_cache, cu_seqlens_q, pos_offsets, block_tables, scale,
                   max_q_len, out, stream, vllm=True)


def pkv_varlen_attention_splitk(q, k_cache, v_cache, cu_seqlens_q, pos_offsets, block_tables,
                                scale, max_q_len=None, num_splits=0, scratch=None, out=None,
                                stream=None):
    """:func:`pkv_varlen_attention` with split-K (``num_splits`` 0 = heuristic).
    ``scratch`` (uint8) is allocated when not given."""
    return _varlen(q, k_cache, v_cache, cu_seqlens_q, pos_offsets, block_tables, scale,
                   max_q_len, out, stream, vllm=False, split=(num_splits, scratch))


def pkv_varlen_attention_splitk_vllm_layout(q, k_cache, v_cache, cu_seqlens_q, pos_offsets,
                                            block_tables, scale, max_q_len=None, num_splits=0,
                                            scratch=None, out=None, stream=None):
    """:func:`pkv_varlen_attention_splitk` over vLLM-layout pools."""
    return _varlen(q, k_cache, v_cache, cu_seqlens_q, pos_offsets, block_tables, scale,
                   max_q_len, out, stream, vllm=True, split=(num_splits, scratch))


def pkv_set_varlen_tensor_path(on) -> int:
    """Run varlen attention with more than 8 (query, head) columns per CTA
    on the tcgen05 kernel (``on`` = 1) or the mma.sync kernel (0, the
    initial setting); returns the previous setting."""
    prev = int(lib.pkv_set_varlen_tensor_path(int(on)))
    if prev < 0:
        raise ValueError(f"pkv_set_varlen_tensor_path: {on!r} is not 0 or 1")
    return prev


def pkv_varlen_pick_num_splits(num_seqs, num_heads, num_kv_heads, max_q_len,
                               max_blocks_per_seq, block_size, num_sms) -> int:
    return int(lib.pkv_varlen_pick_num_splits(num_seqs, num_heads, num_kv_heads, max_q_len,
                                              max_blocks_per_seq, block_size, num_sms))


def _varlen_plan(q, k_cache, block_tables, max_q_len, num_splits=0):
    import torch

    Hkv, bs = _pool_dims(k_cache)
    with torch.cuda.device(q.device):
        return pkv_varlen_splitk_plan(block_tables.shape[0], q.shape[0], int(max_q_len),
                                      q.shape[1], Hkv, q.shape[2], block_tables.shape[1], bs,
                                      num_splits)


def varlen_splits_for(q, k_cache, block_tables, max_q_len, num_splits=0):
    """The split count the varlen split-K call launches for these tensors."""
    return _varlen_plan(q, k_cache, block_tables, max_q_len, num_splits)[0]


def _varlen(q, k_cache, v_cache, cu_seqlens_q, pos_offsets, block_tables, scale, max_q_len, out,
            stream, vllm, split=None):
    import torch

    _want(q, "q", torch.float16, 3)
    total_q, H, D = q.shape
    if vllm:
        NB, Hkv, bs, Dk = _vllm_pools(k_cache, v_cache)
    else:
        _want(k_cache, "k_cache", torch.float16, 4)
        NB, Hkv, bs, Dk = k_cache.shape
        _want(v_cache, "v_cache", torch.float16, 4, k_cache.shape)
    if Dk != D:
        raise ValueError("k_cache head_dim differs from q")
    _want(block_tables, "block_tables", torch.int32, 2)
    B = block_tables.shape[0]
    _want(cu_seqlens_q, "cu_seqlens_q", torch.int32, 1, (B + 1,))
    _want(pos_offsets, "pos_offsets", torch.int32, 1, (B,))
    if out is None:
        out = torch.empty_like(q)
    _want(out, "out", torch.float16, 3, (total_q, H, D))
    if max_q_len is None:
        raise ValueError("max_q_len (a host-side bound) is required")
    args = [q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), cu_seqlens_q.data_ptr(),
            pos_offsets.data_ptr(), block_tables.data_ptr(), B, total_q, int(max_q_len),
            block_tables.shape[1], NB, float(scale), H, Hkv, D, bs, out.data_ptr()]
    if split is None:
        fn = lib.pkv_varlen_attention_vllm_layout if vllm else lib.pkv_varlen_attention
        name = "pkv_varlen_attention_vllm_layout" if vllm else "pkv_varlen_attention"
    else:
        num_splits, scratch = split
        if scratch is None:
            n = _varlen_plan(q, k_cache, block_tables, max_q_len, num_splits)[1]
            scratch = torch.empty(max(n, 16), dtype=torch.uint8, device=q.device)
        _want(scratch, "scratch", torch.uint8, 1)
        args += [int(num_splits), scratch.data_ptr(), scratch.numel()]
        fn = (lib.pkv_varlen_attention_splitk_vllm_layout if vllm
              else lib.pkv_varlen_attention_splitk)
        name = ("pkv_varlen_attention_splitk_vllm_layout" if vllm
                else "pkv_varlen_attention_splitk")
    _check(fn(*args, _stream_ptr(stream)), name)
    return out


def pkv_decode_splitk_noalloc(q, k_cache, v_cache, block_tables, context_lens, scale, out,
                              num_splits=0, stream=None):
    """Split-K decode that allocates nothing: the partials go to the library's
    built-in static device buffer (PKV_NOALLOC_SCRATCH_BYTES) instead of caller
    scratch, and ``out`` must be given.  For callers that may not allocate
    device memory; calls that can overlap on the GPU share that buffer and
    must not be issued."""
    if out is None:
        raise ValueError("pkv_decode_splitk_noalloc needs a caller-provided out")
    B, H, D, NB, Hkv, bs, mbps, out = _decode_shapes(q, k_cache, v_cache, block_tables,
                                                     context_lens, out)
    _check(lib.pkv_decode_splitk_noalloc(q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
                                         block_tables.data_ptr(), context_lens.data_ptr(), B,
                                         mbps, NB, float(scale), H, Hkv, D, bs, out.data_ptr(),
                                         int(num_splits), _stream_ptr(stream)),
           "pkv_decode_splitk_noalloc")
    return out


def _vllm_pools(k_cache, v_cache):
    """(NB, Hkv, bs, D) of vLLM-layout pools: K [NB][Hkv][D/8][bs][8], V [NB][Hkv][D][bs]."""
    import torch

    _want(k_cache, "k_cache", torch.float16, 5)
    NB, Hkv, D8, bs, x = k_cache.shape
    if x != 8:
        raise ValueError("vLLM-layout k_cache must end in 8 (16 bytes of f16)")
    _want(v_cache, "v_cache", torch.float16, 4, (NB, Hkv, D8 * 8, bs))
    return NB, Hkv, bs, D8 * 8


def pkv_append_vllm_layout(k, v, slot_mapping, k_cache, v_cache, stream=None):
    """:func:`pkv_append` into vLLM-layout pools."""
    import torch

    NB, Hkv, bs, D = _vllm_pools(k_cache, v_cache)
    _want(k, "k", torch.float16, 3)
    T = k.shape[0]
    _want(k, "k", torch.float16, 3, (T, Hkv, D))
    _want(v, "v", torch.float16, 3, (T, Hkv, D))
    _want(slot_mapping, "slot_mapping", torch.int32, 1, (T,))
    _check(lib.pkv_append_vllm_layout(k.data_ptr(), v.data_ptr(), slot_mapping.data_ptr(), T,
                                      k_cache.data_ptr(), v_cache.data_ptr(), NB, bs, Hkv, D,
                                      _stream_ptr(stream)), "pkv_append_vllm_layout")


def pkv_decode_vllm_layout(q, k_cache, v_cache, block_tables, context_lens, scale, num_splits=0,
                           scratch=None, out=None, stream=None):
    """:func:`pkv_decode_splitk` over vLLM-layout pools; returns ``out``."""
    import torch

    NB, Hkv, bs, D = _vllm_pools(k_cache, v_cache)
    _want(q, "q", torch.float16, 3)
    B, H, Dq = q.shape
    if Dq != D:
        raise ValueError("k_cache head_dim differs from q")
    _want(block_tables, "block_tables", torch.int32, 2)
    if block_tables.shape[0] != B:
        raise ValueError("block_tables must have num_seqs rows")
    _want(context_lens, "context_lens", torch.int32, 1, (B,))
    if out is None:
        out = torch.empty_like(q)
    _want(out, "out", torch.float16, 3, (B, H, D))
    mbps = block_tables.shape[1]
    if scratch is None:
        scratch = alloc_scratch(q, k_cache, block_tables, num_splits)
    _want(scratch, "scratch", torch.uint8, 1)
    _check(lib.pkv_decode_vllm_layout(q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
                                      block_tables.data_ptr(), context_lens.data_ptr(), B, mbps,
                                      NB, float(scale), H, Hkv, D, bs, out.data_ptr(),
                                      int(num_splits), scratch.data_ptr(), scratch.numel(),
                                      _stream_ptr(stream)), "pkv_decode_vllm_layout")
    return out


def pkv_qkv_norm_rope_append(qkv, q_norm_w, k_norm_w, cos_table, sin_table, k_cache, v_cache,
                             cu_seqlens_q, pos_offsets, block_tables, num_heads, eps=1e-6,
                             q_out=None, stream=None):
    """Split ``qkv [total_q][(H + 2 Hkv) D]``, RMS-norm query/key heads (weights
    may be None), rotate by the tables ``[max_pos][D/2]`` (f32), write the
    queries (returned, ``[total_q][H][D]``) and append keys/values to the pools."""
    import torch

    _want(k_cache, "k_cache", torch.float16, 4)
    NB, Hkv, bs, D = k_cache.shape
    _want(v_cache, "v_cache", torch.float16, 4, k_cache.shape)
    H = int(num_heads)
    _want(qkv, "qkv", torch.float16, 2)
    total_q = qkv.shape[0]
    _want(qkv, "qkv", torch.float16, 2, (total_q, (H + 2 * Hkv) * D))
    for name, w in (("q_norm_w", q_norm_w), ("k_norm_w", k_norm_w)):
        if w is not None:
            _want(w, name, torch.float16, 1, (D,))
    _want(cos_table, "cos_table", torch.float32, 2)
    max_pos = cos_table.shape[0]
    _want(cos_table, "cos_table", torch.float32, 2, (max_pos, D // 2))
    _want(sin_table, "sin_table", torch.float32, 2, (max_pos, D // 2))
    _want(block_tables, "block_tables", torch.int32, 2)
    B = block_tables.shape[0]
    _want(cu_seqlens_q, "cu_seqlens_q", torch.int32, 1, (B + 1,))
    _want(pos_offsets, "pos_offsets", torch.int32, 1, (B,))
    if q_out is None:
        q_out = torch.empty((total_q, H, D), dtype=torch.float16, device=qkv.device)
    _want(q_out, "q_out", torch.float16, 3, (total_q, H, D))
    ptr = lambda t: None if t is None else t.data_ptr()  # noqa: E731
    _check(lib.pkv_qkv_norm_rope_append(
        qkv.data_ptr(), ptr(q_norm_w), ptr(k_norm_w), cos_table.data_ptr(), sin_table.data_ptr(),
        q_out.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), cu_seqlens_q.data_ptr(),
        pos_offsets.data_ptr(), block_tables.data_ptr(), B, total_q, block_tables.shape[1], NB,
        H, Hkv, D, bs, max_pos, float(eps), _stream_ptr(stream)), "pkv_qkv_norm_rope_append")
    return q_out


def pkv_qkv_norm_rope_append_decode(qkv, q_norm_w, k_norm_w, cos_table, sin_table, k_cache,
                                    v_cache, block_tables, context_lens, num_heads, scale,
                                    eps=1e-6, num_splits=0, scratch=None, out=None, stream=None):
    """One decode attention step from each sequence's fused projection row
    ``qkv [B][(H + 2 Hkv) D]``: norm + rotary of its query and key heads at
    position ``context_lens[s] - 1``, append of the key and value rows, and the
    decode of :func:`pkv_decode_splitk` with the rotated queries; returns
    ``out [B][H][D]``."""
    import torch

    _want(k_cache, "k_cache", torch.float16, 4)
    NB, Hkv, bs, D = k_cache.shape
    _want(v_cache, "v_cache", torch.float16, 4, k_cache.shape)
    H = int(num_heads)
    _want(block_tables, "block_tables", torch.int32, 2)
    B, mbps = block_tables.shape
    _want(qkv, "qkv", torch.float16, 2, (B, (H + 2 * Hkv) * D))
    _want(context_lens, "context_lens", torch.int32, 1, (B,))
    for name, w in (("q_norm_w", q_norm_w), ("k_norm_w", k_norm_w)):
        if w is not None:
            _want(w, name, torch.float16, 1, (D,))
    _want(cos_table, "cos_table", torch.float32, 2)
    max_pos = cos_table.shape[0]
    _want(cos_table, "cos_table", torch.float32, 2, (max_pos, D // 2))
    _want(sin_table, "sin_table", torch.float32, 2, (max_pos, D // 2))
    if out is None:
        out = torch.empty((B, H, D), dtype=torch.float16, device=qkv.device)
    _want(out, "out", torch.float16, 3, (B, H, D))
    if scratch is None:
        scratch = alloc_scratch(out, k_cache, block_tables, num_splits)
    _want(scratch, "scratch", torch.uint8, 1)
    ptr = lambda t: None if t is None else t.data_ptr()  # noqa: E731
    _check(lib.pkv_qkv_norm_rope_append_decode(
        qkv.data_ptr(), ptr(q_norm_w), ptr(k_norm_w), cos_table.data_ptr(), sin_table.data_ptr(),
        max_pos, float(eps), k_cache.data_ptr(), v_cache.data_ptr(), block_tables.data_ptr(),
        context_lens.data_ptr(), B, mbps, NB, float(scale), H, Hkv, D, bs, out.data_ptr(),
        int(num_splits), scratch.data_ptr(), scratch.numel(), _stream_ptr(stream)),
        "pkv_qkv_norm_rope_append_decode")
    return out


def pkv_selftest_wait_timeout(stream=None):
    """Launch the failure-path diagnostic (sets PKV_DEV_WAIT_TIMEOUT after 100 ms)."""
    _check(lib.pkv_selftest_wait_timeout(_stream_ptr(stream)), "pkv_selftest_wait_timeout")


def pkv_read_device_status(stream=None) -> int:
    """Read and clear the device status word (synchronizes ``stream``)."""
    flags = ctypes.c_int32(0)
    _check(lib.pkv_read_device_status(ctypes.byref(flags), _stream_ptr(stream)),
           "pkv_read_device_status")
    return int(flags.value)
