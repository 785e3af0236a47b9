"""Seeded synthetic inputs for batched paged-KV decode attention.

This module only draws random numbers and assembles block tables, slot
mappings and cache pools.  It holds none of the attention arithmetic, so both
the CPU oracle (``oracle/``) and the CUDA path can be fed from it.

Shapes follow the five workloads the paged-decode pages describe:

* ``tiny``     B=2,   H=4,  Hkv=2, D=64,  bs=16, L={17,40}, 8-block pool
* ``llama8b``  B=32,  H=32, Hkv=8, D=128, bs=16, L~U[512,2048], 16384-block pool
* ``long``     B=4,   H=32, Hkv=8, D=128, bs=16, L={32K,64K,96K,128K}, one key x8
* ``ragged``   B=256, H=28, Hkv=4, D=128, bs=32, L lognormal(median 1024, sigma 1)
* ``loop``     B=128, H=Hkv=16, D=64, bs=16, 128 append+decode steps

Cache layout: ``[num_blocks][num_kv_heads][block_size][head_dim]`` f16, one
pool for K and one for V.  Block tables are ``int32 [B][max_blocks_per_seq]``;
entries past ``ceil(L/bs)`` hold the id of a *poison* block whose contents are
NaN.  Rows of a sequence's last block past its length are NaN too, so any read
outside a sequence's context turns an output into NaN.

Random numbers come from ``numpy.random.Generator(PCG64(seed))`` with seed
``20261202 + config index``; values are drawn in f32 and rounded to f16.
"""

from __future__ import annotations

import dataclasses
import math
from typing import List, Optional

import numpy as np

BASE_SEED = 20261202

CONFIG_NAMES = ("tiny", "llama8b", "long", "ragged", "loop")


def _rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def _normal_f16(rng: np.random.Generator, shape, std: float = 1.0) -> np.ndarray:
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    return x.astype(np.float16)


def _nan_f16(shape) -> np.ndarray:
    return np.full(shape, np.nan, dtype=np.float16)


@dataclasses.dataclass
class Workload:
    """One decode call: one query token per sequence over a paged KV pool.

    ``seq_k[s]`` / ``seq_v[s]`` are the contiguous ``[L_s][Hkv][D]`` f16 rows of
    sequence ``s`` *including* its newest token (position ``L_s - 1``).  The
    pool built by :func:`host_pool` scatters them through ``block_tables``.
    """

    name: str
    num_seqs: int
    num_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    max_blocks_per_seq: int
    scale: float
    context_lens: np.ndarray  # int32 [B]
    block_tables: np.ndarray  # int32 [B][MBPS]
    q: np.ndarray  # f16 [B][H][D]
    seq_k: List[np.ndarray]
    seq_v: List[np.ndarray]
    poison_block: int

    @property
    def group(self) -> int:
        return self.num_heads // self.num_kv_heads

    @property
    def total_tokens(self) -> int:
        return int(np.asarray(self.context_lens, dtype=np.int64).sum())

    @property
    def kv_bytes(self) -> int:
        """Algorithmic K+V bytes one decode call reads (each token once)."""
        return self.total_tokens * 2 * self.num_kv_heads * self.head_dim * 2

    def blocks_of(self, s: int) -> np.ndarray:
        n = -(-int(self.context_lens[s]) // self.block_size)
        return self.block_tables[s, :n]

    def last_token_append(self):
        """K/V rows and slots that append each sequence's newest token.

        Returns ``(k_new [B][Hkv][D], v_new, slot_mapping int32 [B])`` where the
        slot is ``physical_block * block_size + offset`` of position ``L_s-1``.
        Sequences with ``L_s == 0`` get slot ``-1`` (skip).
        """
        B, Hkv, D, bs = self.num_seqs, self.num_kv_heads, self.head_dim, self.block_size
        k_new = np.zeros((B, Hkv, D), np.float16)
        v_new = np.zeros((B, Hkv, D), np.float16)
        slots = np.full((B,), -1, np.int32)
        for s in range(B):
            L = int(self.context_lens[s])
            if L == 0:
                continue
            pos = L - 1
            k_new[s] = self.seq_k[s][pos]
            v_new[s] = self.seq_v[s][pos]
            slots[s] = int(self.block_tables[s, pos // bs]) * bs + pos % bs
        return k_new, v_new, slots


def _blocked(rows: np.ndarray, bs: int) -> np.ndarray:
    """``[L][Hkv][D]`` rows -> ``[nblk][Hkv][bs][D]`` tiles, NaN past ``L``."""
    L, Hkv, D = rows.shape
    nblk = -(-L // bs)
    padded = _nan_f16((nblk * bs, Hkv, D))
    padded[:L] = rows
    return np.ascontiguousarray(padded.reshape(nblk, bs, Hkv, D).transpose(0, 2, 1, 3))


def compact_blocks(w: Workload, upto_last: bool = False):
    """Used blocks as ``(ids int64 [n], k [n][Hkv][bs][D], v [...])``.

    With ``upto_last`` the newest token of every sequence (position ``L-1``) is
    left out (NaN), i.e. the pool as it stands before that token is appended.
    The poison block (all NaN) is included so a device pool built from this
    also carries it.
    """
    ids, ks, vs = [], [], []
    bs = w.block_size
    for s in range(w.num_seqs):
        L = int(w.context_lens[s])
        if L == 0:
            continue
        kb = _blocked(w.seq_k[s][:L], bs)
        vb = _blocked(w.seq_v[s][:L], bs)
        if upto_last:
            pos = L - 1
            kb[pos // bs, :, pos % bs, :] = np.nan
            vb[pos // bs, :, pos % bs, :] = np.nan
        ids.append(w.blocks_of(s).astype(np.int64))
        ks.append(kb)
        vs.append(vb)
    shape = (1, w.num_kv_heads, bs, w.head_dim)
    ids.append(np.array([w.poison_block], np.int64))
    ks.append(_nan_f16(shape))
    vs.append(_nan_f16(shape))
    return np.concatenate(ids), np.concatenate(ks), np.concatenate(vs)


def host_pool(w: Workload, upto_last: bool = False, fill: float = 0.0):
    """Full ``[NB][Hkv][bs][D]`` host pools (numpy f16).

    Blocks that no sequence uses hold ``fill``; with the default 0.0 the array
    comes from ``np.zeros`` and untouched pages are never materialised, so the
    200000-block pool of the ragged workload costs only what it uses.
    """
    shape = (w.num_blocks, w.num_kv_heads, w.block_size, w.head_dim)
    if fill == 0.0:
        kc = np.zeros(shape, np.float16)
        vc = np.zeros(shape, np.float16)
    else:
        kc = np.full(shape, fill, np.float16)
        vc = np.full(shape, fill, np.float16)
    ids, kb, vb = compact_blocks(w, upto_last=upto_last)
    kc[ids] = kb
    vc[ids] = vb
    return kc, vc


def _tables_from_perm(lens, bs, mbps, perm, poison):
    B = len(lens)
    tables = np.full((B, mbps), poison, np.int32)
    cur = 0
    for s, L in enumerate(lens):
        n = -(-int(L) // bs)
        tables[s, :n] = perm[cur : cur + n]
        cur += n
    return tables, cur


def _finish(name, rng, lens, H, Hkv, D, bs, NB, mbps, std=1.0, perm=None,
            sharp_key=False) -> Workload:
    lens = np.asarray(lens, np.int32)
    B = len(lens)
    if perm is None:
        perm = rng.permutation(NB).astype(np.int32)
    need = int(sum(-(-int(L) // bs) for L in lens))
    if need >= NB:
        raise ValueError(f"{name}: pool of {NB} blocks cannot hold {need} + poison")
    poison = int(perm[need])
    tables, used = _tables_from_perm(lens, bs, mbps, perm, poison)
    assert used == need
    q = _normal_f16(rng, (B, H, D), std)
    seq_k, seq_v = [], []
    for s in range(B):
        L = int(lens[s])
        k = _normal_f16(rng, (L, Hkv, D), std)
        v = _normal_f16(rng, (L, Hkv, D), std)
        if sharp_key and L > 0:
            pos = int(rng.integers(0, L))
            k[pos] = (k[pos].astype(np.float32) * 8.0).astype(np.float16)
        seq_k.append(k)
        seq_v.append(v)
    return Workload(name=name, num_seqs=B, num_heads=H, num_kv_heads=Hkv, head_dim=D,
                    block_size=bs, num_blocks=NB, max_blocks_per_seq=mbps,
                    scale=1.0 / math.sqrt(D), context_lens=lens, block_tables=tables,
                    q=q, seq_k=seq_k, seq_v=seq_v, poison_block=poison)


def tiny() -> Workload:
    """B=2, H=4, Hkv=2, D=64, bs=16, L={17,40}, 8 blocks by seeded permutation."""
    rng = _rng(BASE_SEED + 0)
    perm = rng.permutation(8).astype(np.int32)
    # seq 0 takes perm[0:2], seq 1 perm[2:5]; perm[5] is the poison block.
    return _finish("tiny", rng, [17, 40], H=4, Hkv=2, D=64, bs=16, NB=8, mbps=3,
                   perm=perm)


def llama8b() -> Workload:
    """Llama-3-8B attention shape: B=32, H=32, Hkv=8, D=128, bs=16."""
    rng = _rng(BASE_SEED + 1)
    lens = rng.integers(512, 2048, size=32, endpoint=True)
    return _finish("llama8b", rng, lens, H=32, Hkv=8, D=128, bs=16, NB=16384, mbps=128)


def long_context() -> Workload:
    """B=4, H=32, Hkv=8, D=128, bs=16, L = 32K/64K/96K/128K, one key x8 per seq."""
    rng = _rng(BASE_SEED + 2)
    lens = [32768, 65536, 98304, 131072]
    return _finish("long", rng, lens, H=32, Hkv=8, D=128, bs=16, NB=24576, mbps=8192,
                   sharp_key=True)


def ragged_lens(rng: np.random.Generator, B: int = 256) -> np.ndarray:
    z = rng.standard_normal(B)
    lens = np.clip(np.rint(np.exp(math.log(1024.0) + z)), 1, 16384).astype(np.int32)
    ones = rng.choice(B, size=8, replace=False)
    lens[ones] = 1
    return lens


def ragged() -> Workload:
    """B=256, H=28, Hkv=4 (G=7), D=128, bs=32, lognormal lengths, 200000 blocks."""
    rng = _rng(BASE_SEED + 3)
    lens = ragged_lens(rng)
    return _finish("ragged", rng, lens, H=28, Hkv=4, D=128, bs=32, NB=200000, mbps=512,
                   std=0.5)


def make(name: str) -> Workload:
    return {"tiny": tiny, "llama8b": llama8b, "long": long_context,
            "ragged": ragged}[name]()


def compact_pool(w: Workload, seed: int = BASE_SEED + 99, slack: int = 64) -> Workload:
    """The same workload over a smaller pool: the blocks its sequences use
    (and the poison block) renumbered by a seeded random permutation of
    ``used + slack`` ids, so the reads stay scattered but the pool holds only
    what the call reads (for profiling captures that save and restore device
    memory).  Values, lengths and the logical tables are unchanged."""
    ids, _, _ = compact_blocks(w)
    used = np.unique(ids)
    nb = len(used) + slack
    perm = _rng(seed).permutation(nb).astype(np.int32)
    remap = np.full(w.num_blocks, -1, np.int64)
    remap[used] = perm[:len(used)]
    tables = remap[w.block_tables].astype(np.int32)
    assert (tables >= 0).all()
    return dataclasses.replace(w, name=f"{w.name}-compact", num_blocks=nb, block_tables=tables,
                               poison_block=int(remap[w.poison_block]))


def widen_tables(w: Workload, factor: int) -> Workload:
    """The same workload with block tables ``factor`` times wider than its
    longest context needs (as a server sizes them for the model's maximum
    context); the extra entries point at the poison block."""
    mbps = w.max_blocks_per_seq * factor
    tables = np.full((w.num_seqs, mbps), w.poison_block, np.int32)
    tables[:, :w.max_blocks_per_seq] = w.block_tables
    return dataclasses.replace(w, name=f"{w.name}-x{factor}", max_blocks_per_seq=mbps,
                               block_tables=tables)


def small_random(seed: int, num_seqs: int, num_heads: int, num_kv_heads: int,
                 head_dim: int, block_size: int, lens, num_blocks: Optional[int] = None,
                 std: float = 1.0) -> Workload:
    """A seeded random case of any shape (used for tiny brute-force checks)."""
    rng = _rng(seed)
    need = sum(-(-int(L) // block_size) for L in lens)
    NB = num_blocks if num_blocks is not None else need + 3
    mbps = max(1, max(-(-int(L) // block_size) for L in lens))
    return _finish(f"random{seed}", rng, lens, H=num_heads, Hkv=num_kv_heads, D=head_dim,
                   bs=block_size, NB=NB, mbps=mbps, std=std)


# ---------------------------------------------------------------------------
# The append+decode loop: 128 steps, each appending one token per sequence
# (plus padding rows with slot -1) and then decoding over the grown context.
# ---------------------------------------------------------------------------


@dataclasses.dataclass
class LoopStep:
    k_new: np.ndarray  # f16 [T][Hkv][D]   (padding rows are NaN)
    v_new: np.ndarray
    slot_mapping: np.ndarray  # int32 [T]   (-1 on padding rows)
    q: np.ndarray  # f16 [B][H][D]
    context_lens: np.ndarray  # int32 [B], after this step's append
    block_tables: np.ndarray  # int32 [B][MBPS], after this step's allocation


class AppendDecodeLoop:
    """MHA H=Hkv=16, D=64, bs=16, B=128, start L~U[64,4096], 128 steps.

    The host keeps a seeded shuffled free list of physical blocks; a sequence
    that crosses into a new block pops one.  Each step appends T=142 rows: the
    128 real tokens plus 14 padding rows (slot -1, NaN K/V) at seeded places.
    """

    name = "loop"

    def __init__(self, steps: int = 128, seed: int = BASE_SEED + 4, num_seqs: int = 128,
                 num_heads: int = 16, head_dim: int = 64, block_size: int = 16,
                 num_blocks: int = 40000, max_blocks_per_seq: int = 272,
                 num_pad: int = 14, min_len: int = 64, max_len: int = 4096):
        self.steps = steps
        self.seed = seed
        self.num_seqs = B = num_seqs
        self.num_heads = self.num_kv_heads = num_heads
        self.head_dim = head_dim
        self.block_size = bs = block_size
        self.num_blocks = num_blocks
        self.max_blocks_per_seq = max_blocks_per_seq
        self.scale = 1.0 / math.sqrt(head_dim)
        self.num_pad = num_pad
        rng = _rng(seed)
        self.start_lens = rng.integers(min_len, max_len, size=B, endpoint=True).astype(np.int32)
        free = list(rng.permutation(num_blocks).astype(np.int32)[::-1])
        self.poison_block = int(free.pop(0))  # the last block of the shuffled list
        tables = np.full((B, max_blocks_per_seq), self.poison_block, np.int32)
        nalloc = np.zeros(B, np.int64)
        for s in range(B):
            n = -(-int(self.start_lens[s]) // bs)
            if n > max_blocks_per_seq:
                raise ValueError("start length exceeds max_blocks_per_seq")
            for j in range(n):
                if not free:
                    raise RuntimeError("free list exhausted")
                tables[s, j] = free.pop()
            nalloc[s] = n
        self.start_tables = tables.copy()
        # The allocation schedule of every step, fixed up front (integers only).
        self.tables = np.empty((steps, B, max_blocks_per_seq), np.int32)
        self.slots = np.empty((steps, B), np.int32)
        lens = self.start_lens.astype(np.int64).copy()
        for t in range(steps):
            for s in range(B):
                pos = int(lens[s])
                j = pos // bs
                if j >= nalloc[s]:
                    if j >= max_blocks_per_seq:
                        raise ValueError("sequence outgrew max_blocks_per_seq")
                    if not free:
                        raise RuntimeError("free list exhausted")
                    tables[s, j] = free.pop()
                    nalloc[s] = j + 1
                self.slots[t, s] = int(tables[s, j]) * bs + pos % bs
            lens += 1
            self.tables[t] = tables
        self.end_lens = lens.astype(np.int32)
        self.pad_rows = np.stack([
            np.sort(_rng(seed * 1000 + 7 + t).choice(B + num_pad, size=num_pad, replace=False))
            for t in range(steps)])
        # initial cache contents, one row per existing token
        self.init_k = [_normal_f16(rng, (int(L), num_heads, head_dim)) for L in self.start_lens]
        self.init_v = [_normal_f16(rng, (int(L), num_heads, head_dim)) for L in self.start_lens]

    @property
    def group(self) -> int:
        return 1

    def initial_workload(self) -> Workload:
        """The pool before step 0, as a :class:`Workload` (q unused)."""
        return Workload(name="loop-start", num_seqs=self.num_seqs, num_heads=self.num_heads,
                        num_kv_heads=self.num_kv_heads, head_dim=self.head_dim,
                        block_size=self.block_size, num_blocks=self.num_blocks,
                        max_blocks_per_seq=self.max_blocks_per_seq, scale=self.scale,
                        context_lens=self.start_lens.copy(), block_tables=self.start_tables.copy(),
                        q=np.zeros((self.num_seqs, self.num_heads, self.head_dim), np.float16),
                        seq_k=self.init_k, seq_v=self.init_v, poison_block=self.poison_block)

    def step(self, t: int) -> LoopStep:
        B, H, D = self.num_seqs, self.num_heads, self.head_dim
        rng = _rng(self.seed * 1000 + 100003 + t)
        q = _normal_f16(rng, (B, H, D))
        k_real = _normal_f16(rng, (B, H, D))
        v_real = _normal_f16(rng, (B, H, D))
        T = B + self.num_pad
        pad = np.zeros(T, bool)
        pad[self.pad_rows[t]] = True
        k_new = _nan_f16((T, H, D))
        v_new = _nan_f16((T, H, D))
        slots = np.full(T, -1, np.int32)
        real_idx = np.nonzero(~pad)[0]
        k_new[real_idx] = k_real
        v_new[real_idx] = v_real
        slots[real_idx] = self.slots[t]
        lens = (self.start_lens.astype(np.int64) + t + 1).astype(np.int32)
        return LoopStep(k_new=k_new, v_new=v_new, slot_mapping=slots, q=q,
                        context_lens=lens, block_tables=self.tables[t])

    @property
    def kv_bytes_per_step(self):
        """Algorithmic K+V bytes of every step's decode, as a list."""
        per_tok = 2 * self.num_kv_heads * self.head_dim * 2
        return [int((self.start_lens.astype(np.int64) + t + 1).sum()) * per_tok
                for t in range(self.steps)]


def to_device(w: Workload, device="cuda", upto_last: bool = False, poison_fill=True):
    """Device copies of a workload: pools, tables, lens and q as torch tensors.

    Unused pool blocks are NaN when ``poison_fill`` (so stray reads show), the
    used blocks come from :func:`compact_blocks`.
    """
    import torch

    shape = (w.num_blocks, w.num_kv_heads, w.block_size, w.head_dim)
    fill = float("nan") if poison_fill else 0.0
    kc = torch.full(shape, fill, dtype=torch.float16, device=device)
    vc = torch.full(shape, fill, dtype=torch.float16, device=device)
    ids, kb, vb = compact_blocks(w, upto_last=upto_last)
    idx = torch.from_numpy(ids).to(device)
    kc.index_copy_(0, idx, torch.from_numpy(kb).to(device))
    vc.index_copy_(0, idx, torch.from_numpy(vb).to(device))
    return {"k_cache": kc, "v_cache": vc, **_device_meta(w, device)}


def _device_meta(w: Workload, device):
    import torch

    return {
        "block_tables": torch.from_numpy(np.ascontiguousarray(w.block_tables)).to(device),
        "context_lens": torch.from_numpy(np.ascontiguousarray(w.context_lens)).to(device),
        "q": torch.from_numpy(np.ascontiguousarray(w.q)).to(device),
    }


def vllm_layout_tiles(kb: np.ndarray, vb: np.ndarray):
    """Blocked tiles ``[n][Hkv][bs][D]`` rearranged into the vLLM layout:
    K ``[n][Hkv][D/8][bs][8]``, V ``[n][Hkv][D][bs]`` (same values)."""
    n, Hkv, bs, D = kb.shape
    kv = np.ascontiguousarray(kb.reshape(n, Hkv, bs, D // 8, 8).transpose(0, 1, 3, 2, 4))
    vv = np.ascontiguousarray(vb.transpose(0, 1, 3, 2))
    return kv, vv


def host_pool_vllm(w: Workload, upto_last: bool = False, fill: float = 0.0):
    """:func:`host_pool` in the vLLM layout."""
    NB, Hkv, bs, D = w.num_blocks, w.num_kv_heads, w.block_size, w.head_dim
    make = np.zeros if fill == 0.0 else (lambda shp, dt: np.full(shp, fill, dt))
    kc = make((NB, Hkv, D // 8, bs, 8), np.float16)
    vc = make((NB, Hkv, D, bs), np.float16)
    ids, kb, vb = compact_blocks(w, upto_last=upto_last)
    kv, vv = vllm_layout_tiles(kb, vb)
    kc[ids] = kv
    vc[ids] = vv
    return kc, vc


def to_device_vllm(w: Workload, device="cuda", upto_last: bool = False, poison_fill=True):
    """:func:`to_device` with the pools in the vLLM layout."""
    import torch

    d = _device_meta(w, device)
    NB, Hkv, bs, D = w.num_blocks, w.num_kv_heads, w.block_size, w.head_dim
    fill = float("nan") if poison_fill else 0.0
    kc = torch.full((NB, Hkv, D // 8, bs, 8), fill, dtype=torch.float16, device=device)
    vc = torch.full((NB, Hkv, D, bs), fill, dtype=torch.float16, device=device)
    ids, kb, vb = compact_blocks(w, upto_last=upto_last)
    kv, vv = vllm_layout_tiles(kb, vb)
    idx = torch.from_numpy(ids).to(device)
    kc.index_copy_(0, idx, torch.from_numpy(kv).to(device))
    vc.index_copy_(0, idx, torch.from_numpy(vv).to(device))
    d["k_cache"] = kc
    d["v_cache"] = vc
    return d


@dataclasses.dataclass
class VarlenWorkload:
    """Multi-token queries over a paged context: sequence s has q_lens[s]
    query tokens at positions pos_offsets[s] .. pos_offsets[s]+q_lens[s]-1,
    and its cache holds pos_offsets[s] + q_lens[s] rows (the prefix and the
    new tokens' K/V, already written)."""

    base: Workload  # context_lens = pos_offsets + q_lens; q unused
    q: np.ndarray  # f16 [total_q][H][D]
    cu_seqlens_q: np.ndarray  # int32 [B+1]
    pos_offsets: np.ndarray  # int32 [B]

    @property
    def total_q(self) -> int:
        return int(self.cu_seqlens_q[-1])

    @property
    def max_q_len(self) -> int:
        return int(np.diff(self.cu_seqlens_q).max()) if len(self.cu_seqlens_q) > 1 else 0


def varlen_random(seed: int, num_heads: int, num_kv_heads: int, head_dim: int, block_size: int,
                  q_lens, prefix_lens, std: float = 1.0, num_blocks: Optional[int] = None
                  ) -> VarlenWorkload:
    """A seeded case: sequence s has prefix_lens[s] earlier tokens and
    q_lens[s] new query tokens."""
    q_lens = [int(x) for x in q_lens]
    prefix = [int(x) for x in prefix_lens]
    base = small_random(seed, num_seqs=len(q_lens), num_heads=num_heads,
                        num_kv_heads=num_kv_heads, head_dim=head_dim, block_size=block_size,
                        lens=[p + n for p, n in zip(prefix, q_lens)], num_blocks=num_blocks,
                        std=std)
    rng = _rng(seed * 7919 + 13)
    total_q = sum(q_lens)
    q = _normal_f16(rng, (total_q, num_heads, head_dim), std)
    cu = np.zeros(len(q_lens) + 1, np.int32)
    cu[1:] = np.cumsum(q_lens)
    return VarlenWorkload(base=base, q=q, cu_seqlens_q=cu,
                          pos_offsets=np.asarray(prefix, np.int32))


def spec_verify_long() -> VarlenWorkload:
    """Speculative-decode verification over long contexts (the long-context
    decode shape): B=4, H=32, Hkv=8, D=128, bs=16, 4 draft tokens per
    sequence after prefixes of 32768/65536/98304/131072 - 4 tokens."""
    prefix = [32768 - 4, 65536 - 4, 98304 - 4, 131072 - 4]
    return varlen_random(BASE_SEED + 6, 32, 8, 128, 16, [4] * 4, prefix, num_blocks=24576)


def prefill_chunk() -> VarlenWorkload:
    """Chunked prefill on the Llama-3-8B attention shape: B=4 sequences, 512
    new tokens each after a 2048-token prefix (H=32, Hkv=8, D=128, bs=16)."""
    return varlen_random(BASE_SEED + 7, 32, 8, 128, 16, [512] * 4, [2048] * 4)


def prefill_one() -> VarlenWorkload:
    """Chunked prefill of one sequence (the common serving case): 512 new
    tokens after a 2048-token prefix on the Llama-3-8B attention shape; its
    pairs of query tiles fill under half of the GPU without split-K."""
    return varlen_random(BASE_SEED + 8, 32, 8, 128, 16, [512], [2048])


def spec_verify() -> VarlenWorkload:
    """Speculative-decode verification on the Llama-3-8B attention shape:
    B=32, H=32, Hkv=8, D=128, bs=16, 4 draft tokens per sequence over a
    prefix ~U[512,2048]."""
    rng = _rng(BASE_SEED + 5)
    prefix = rng.integers(508, 2044, size=32, endpoint=True)
    return varlen_random(BASE_SEED + 5, 32, 8, 128, 16, [4] * 32, prefix,
                         num_blocks=16384)


# ---------------------------------------------------------------------------
# Inputs of the fused QKV split + norm + rotary + append step
# ---------------------------------------------------------------------------

@dataclasses.dataclass
class QkvCase:
    """Seeded inputs: fused projection rows, norm weights, rotary tables and a
    paged context for each sequence's new tokens (positions prefix .. prefix +
    q_len - 1).  The tables hold cos/sin of the standard rotary angles
    p * base^(-2i/D); they are inputs of the step, like the weights."""

    qkv: np.ndarray        # f16 [total_q][(H + 2 Hkv) D]
    q_norm_w: Optional[np.ndarray]  # f16 [D] or None
    k_norm_w: Optional[np.ndarray]
    cos: np.ndarray        # f32 [max_pos][D/2]
    sin: np.ndarray
    cu_seqlens_q: np.ndarray  # int32 [B+1]
    pos_offsets: np.ndarray   # int32 [B]
    block_tables: np.ndarray  # int32 [B][MBPS]
    num_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    eps: float = 1e-6


def qkv_case(seed: int, num_heads: int, num_kv_heads: int, head_dim: int, block_size: int,
             q_lens, prefix_lens, norm: bool = True, base: float = 10000.0,
             extra_blocks: int = 3) -> QkvCase:
    rng = _rng(seed)
    q_lens = [int(x) for x in q_lens]
    prefix = [int(x) for x in prefix_lens]
    B = len(q_lens)
    ends = [p + n for p, n in zip(prefix, q_lens)]
    nblk = [-(-e // block_size) for e in ends]
    NB = sum(nblk) + extra_blocks
    mbps = max(1, max(nblk))
    perm = rng.permutation(NB).astype(np.int32)
    tables = np.full((B, mbps), perm[-1], np.int32)
    cur = 0
    for s, n in enumerate(nblk):
        tables[s, :n] = perm[cur:cur + n]
        cur += n
    total_q = sum(q_lens)
    width = (num_heads + 2 * num_kv_heads) * head_dim
    qkv = _normal_f16(rng, (total_q, width), 1.0)
    qw = rng.uniform(0.5, 1.5, head_dim).astype(np.float16) if norm else None
    kw = rng.uniform(0.5, 1.5, head_dim).astype(np.float16) if norm else None
    max_pos = max(ends) + 1
    inv = base ** (-np.arange(head_dim // 2) * 2.0 / head_dim)
    ang = np.arange(max_pos)[:, None] * inv[None, :]
    cu = np.zeros(B + 1, np.int32)
    cu[1:] = np.cumsum(q_lens)
    return QkvCase(qkv=qkv, q_norm_w=qw, k_norm_w=kw, cos=np.cos(ang).astype(np.float32),
                   sin=np.sin(ang).astype(np.float32), cu_seqlens_q=cu,
                   pos_offsets=np.asarray(prefix, np.int32), block_tables=tables,
                   num_heads=num_heads, num_kv_heads=num_kv_heads, head_dim=head_dim,
                   block_size=block_size, num_blocks=NB)
