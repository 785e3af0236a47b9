// Kernels of libpagedkv (GB300, sm_103a):
//   append_kernel                 slot-mapped KV write
//   append_vllm_kernel            the same write into vLLM-layout pools
//   qkv_norm_rope_kernel          fused QKV split + RMS norm + rotary
//                                 embedding + paged append
//   paged_decode_kernel           decode: single pass, or split-K phase 1;
//                                 optionally with the step's append, or the
//                                 step's QKV norm + rotary + append, fused
//                                 in; blocked or vLLM-layout pools
//   splitk_combine_kernel         log-sum-exp merge of split-K partials (a
//                                 warp per output row)
//   varlen_combine_kernel         the same for varlen split-K partials
//   paged_varlen_kernel           several causal queries per sequence (one or
//                                 two mma n-tiles of 8 query-head columns);
//                                 single pass or split-K phase 1; blocked or
//                                 vLLM-layout pools
//   wait_timeout_probe_kernel     failure-path diagnostic (a bounded wait on a
//                                 barrier nothing arrives on)
//
// Decode design:
//  * One CTA per (sequence, KV head[, split]).  It covers the whole GQA group
//    of that KV head, so every K/V byte is read from HBM once.
//  * Each of the CTA's W warps owns a private ring of P shared-memory stages.
//    A stage holds the K and V tiles of one physical block for this KV head
//    (block_size x head_dim f16 each, contiguous in the pool).  Lane 0 of the
//    warp fetches them with TMA copies (one tensor copy per tile with the
//    128-byte swizzle; a bulk copy for vLLM-layout K tiles) that complete on
//    the stage's mbarrier.  Warp w takes the chunk's blocks w, w+WE, ...
//    where WE <= W warps are active (fewer for short sequences under the
//    fair-share depth, see DecodeParams::fair_depth).
//  * Scores use tensor cores with tokens on M and the group on N:
//      S^T[16 tok x 8 heads] = K[16 x D] . Q^T[D x 8]      (mma m16n8k16)
//      O^T[D x 8 heads]     += V^T[D x 16 tok] . P^T[16 x 8]
//    K/V fragments come from ldmatrix (V transposed), Q^T fragments stay in
//    registers, and P^T is P transposed in registers with movmatrix.  Groups
//    smaller than 8 leave unused columns (computed, never stored).
//  * Online softmax in f32 (base-2 exponent with scale*log2(e) folded in);
//    the running max is shared by the 8 lanes holding one head's column, the
//    running sum stays per lane until the end.
//  * At the end the W warp states are merged through shared memory; the
//    single-pass kernel writes f16 output, the split-K kernel writes the
//    unnormalised f32 partial output, max and sum for the combine kernel.
//  * Every kernel is launched with programmatic dependent launch: it lets the
//    next kernel start on entry and waits (griddepcontrol.wait) before its
//    first global-memory access.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <math_constants.h>
#include <stdint.h>

#include <type_traits>

#include "pagedkv.h"
#include "ptx.cuh"

namespace pkv {

// Per-GPU status word; kernels OR PKV_DEV_* bits into it.  (This header is
// compiled into exactly one translation unit.)
__device__ unsigned int g_device_status = 0;

constexpr unsigned int kDevBadSlot = 0x1u;
constexpr unsigned int kDevBadBlockId = 0x2u;
constexpr unsigned int kDevBadContextLen = 0x4u;
constexpr unsigned int kDevWaitTimeout = 0x8u;

// Split the q.K mma chain of a tile over two accumulators (build flag).
#ifndef PKV_QK_SPLIT
#define PKV_QK_SPLIT 1
#endif

// A tile copy that has not landed after this long is reported, not awaited
// (a real copy takes microseconds).
constexpr uint64_t kWaitLimitNs = 100000000ull;

// ---------------------------------------------------------------------------
// append
// ---------------------------------------------------------------------------

// One thread per 16-byte chunk of a (token, kv head) row; K and V together.
__global__ void __launch_bounds__(256)
append_kernel(const uint4* __restrict__ k, const uint4* __restrict__ v,
              const int32_t* __restrict__ slot_mapping, long long total_chunks,
              int chunks_per_row, int num_kv_heads, int block_size, long long num_slots,
              uint4* __restrict__ k_cache, uint4* __restrict__ v_cache) {
  pdl_launch_dependents();
  pdl_wait();
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total_chunks;
       i += stride) {
    const int ch = (int)(i % chunks_per_row);
    const long long row = i / chunks_per_row;  // token * num_kv_heads + head
    const int h = (int)(row % num_kv_heads);
    const long long t = row / num_kv_heads;
    const int slot = __ldg(slot_mapping + t);
    if (slot < 0) continue;
    if ((long long)slot >= num_slots) {
      if (h == 0 && ch == 0) atomicOr(&g_device_status, kDevBadSlot);
      continue;
    }
    const int blk = slot / block_size;
    const int off = slot - blk * block_size;
    const size_t dst = (((size_t)blk * num_kv_heads + h) * block_size + off) * chunks_per_row + ch;
    k_cache[dst] = __ldg(k + i);
    v_cache[dst] = __ldg(v + i);
  }
}

// The same write into vLLM-layout pools: K [NB][Hkv][D/8][bs][8] (a 16-byte
// chunk of 8 head-dim elements per token), V [NB][Hkv][D][bs] (tokens
// innermost).  One thread per 16-byte chunk of a (token, kv head) row: its
// K chunk lands whole, its V chunk as 8 two-byte writes, one per d.
__global__ void __launch_bounds__(256)
append_vllm_kernel(const uint4* __restrict__ k, const uint4* __restrict__ v,
                   const int32_t* __restrict__ slot_mapping, long long total_chunks,
                   int chunks_per_row, int num_kv_heads, int block_size, long long num_slots,
                   uint4* __restrict__ k_cache, __half* __restrict__ v_cache) {
  pdl_launch_dependents();
  pdl_wait();
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total_chunks;
       i += stride) {
    const int ch = (int)(i % chunks_per_row);
    const long long row = i / chunks_per_row;  // token * num_kv_heads + head
    const int h = (int)(row % num_kv_heads);
    const long long t = row / num_kv_heads;
    const int slot = __ldg(slot_mapping + t);
    if (slot < 0) continue;
    if ((long long)slot >= num_slots) {
      if (h == 0 && ch == 0) atomicOr(&g_device_status, kDevBadSlot);
      continue;
    }
    const int blk = slot / block_size;
    const int off = slot - blk * block_size;
    const size_t tile = (size_t)blk * num_kv_heads + h;
    k_cache[(tile * chunks_per_row + ch) * block_size + off] = __ldg(k + i);
    const uint4 vv = __ldg(v + i);
    const __half* vh = reinterpret_cast<const __half*>(&vv);
    __half* vdst = v_cache + (tile * chunks_per_row * 8 + (size_t)ch * 8) * block_size + off;
#pragma unroll
    for (int e = 0; e < 8; ++e) vdst[(size_t)e * block_size] = vh[e];
  }
}

// ---------------------------------------------------------------------------
// fused QKV split + per-head RMS norm + rotary embedding + paged append
// ---------------------------------------------------------------------------
//
// One CTA of four warps per (token, group of heads) (grid x, y), over the
// token's row [q heads | k heads | v heads]; the head layout is described at
// qkv_norm_rope_kernel.  Token row r of sequence
// s sits at position p = pos_offsets[s] + (r - cu_seqlens_q[s]), its rotary
// position and its cache row.  Query and key heads are RMS-normalised when a
// weight vector is given, then turned by the rotary angles of position p
// (rotate-half pairs (i, i + D/2), cos/sin tables [max_pos][D/2] f32); value
// heads are copied.  Queries go to q_out token-major, keys and values to the
// pools at slot block_tables[s][p / bs] * bs + p % bs.  A token whose
// sequence range or position is invalid is skipped and flagged; an invalid
// block id skips its key and value writes and is flagged.

struct QkvRopeParams {
  const __half* qkv;       // [total_q][(H + 2 Hkv) D]
  const __half* q_norm_w;  // [D] or null: no query norm
  const __half* k_norm_w;  // [D] or null: no key norm
  const float* cos_t;      // [max_pos][D/2]
  const float* sin_t;
  __half* q_out;  // [total_q][H][D]
  __half* k_cache;
  __half* v_cache;
  const int32_t* cu_seqlens_q;  // [B + 1]
  const int32_t* pos_offsets;   // [B]
  const int32_t* block_tables;  // [B][MBPS]
  int num_seqs;
  int total_q;
  int num_heads;
  int num_kv_heads;
  int max_blocks_per_seq;
  int num_blocks;
  int block_size;
  int max_pos;
  float eps;
};

// qkv_norm_rope_kernel layout: a head of D halves is spread over D/16 lanes;
// lane l of a head holds elements 8l .. 8l+7 and the same + D/2 (both
// halves of its eight rotate-half pairs) as two 16-byte words.  A warp
// covers 512/D heads per slot and NS slots; the CTA's four warps issue the
// loads of all their heads before any work, so the CTA keeps
// 4 * NS * 512/D heads' rows in flight (NS = 1..4, picked on the host so
// that the heads of a row fill the CTAs with the fewest idle slots; on the
// Llama-3-8B shape, 48 heads, one CTA of NS = 3 per row ran 35.4 us per
// 8192 tokens against 41.6, 44.0 and 40.9 us for NS = 1, 2, 4).
__host__ __device__ constexpr int qkv_heads_per_cta(int D, int NS) { return 4 * NS * (512 / D); }

__device__ __forceinline__ float2 h2f(uint32_t v) {
  return __half22float2(*reinterpret_cast<const __half2*>(&v));
}
__device__ __forceinline__ uint32_t f2h(float x, float y) {
  return pack_half2(__floats2half2_rn(x, y));
}

template <int D, int BS, int NS>
__global__ void __launch_bounds__(128) qkv_norm_rope_kernel(const QkvRopeParams p) {
  constexpr int LPH = D / 16;    // lanes per head
  constexpr int G = 32 / LPH;    // heads per warp and slot
  pdl_launch_dependents();
  pdl_wait();
  const int H = p.num_heads, Hkv = p.num_kv_heads;
  const int heads = H + 2 * Hkv;
  const int row = blockIdx.x;  // grid: x = token row, y = group of heads
  const int lane = threadIdx.x & 31;
  const int l = lane % LPH;
  const int h0 = blockIdx.y * qkv_heads_per_cta(D, NS) + (threadIdx.x >> 5) * (NS * G) + lane / LPH;

  // The row's loads depend on nothing but the block index: they go out
  // first (raw bits, so value rows are copied exactly), and the sequence
  // lookup runs while they are in flight.
  const __half* x_row = p.qkv + (size_t)row * heads * D + 8 * l;
  uint4 ra[NS], rb[NS];
#pragma unroll
  for (int k = 0; k < NS; ++k) {
    const int hh = min(h0 + k * G, heads - 1);  // duplicates past the end are never stored
    ra[k] = __ldg(reinterpret_cast<const uint4*>(x_row + hh * D));
    rb[k] = __ldg(reinterpret_cast<const uint4*>(x_row + hh * D + D / 2));
  }

  int lo = 0, hi = p.num_seqs - 1;  // last sequence whose first row is <= row
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(p.cu_seqlens_q + mid) <= row)
      lo = mid;
    else
      hi = mid - 1;
  }
  const int q_begin = __ldg(p.cu_seqlens_q + lo);
  const int q_end = __ldg(p.cu_seqlens_q + lo + 1);
  const int pos = __ldg(p.pos_offsets + lo) + (row - q_begin);
  const int cap = p.max_blocks_per_seq * BS;
  if (q_begin < 0 || q_end > p.total_q || row < q_begin || row >= q_end || pos < 0 ||
      pos >= p.max_pos || pos >= cap) {
    if (threadIdx.x == 0) atomicOr(&g_device_status, kDevBadContextLen);
    return;
  }
  const int blk = __ldg(p.block_tables + (size_t)lo * p.max_blocks_per_seq + pos / BS);
  // this lane's angles and weights (elements 8l .. 8l+7 and + D/2)
  const float4* cs4 = reinterpret_cast<const float4*>(p.cos_t + (size_t)pos * (D / 2) + 8 * l);
  const float4* sn4 = reinterpret_cast<const float4*>(p.sin_t + (size_t)pos * (D / 2) + 8 * l);
  const float4 c0 = __ldg(cs4), c1 = __ldg(cs4 + 1), s0 = __ldg(sn4), s1 = __ldg(sn4 + 1);
  const float cs[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
  const float sn[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
  const uint4 one = make_uint4(0x3c003c00u, 0x3c003c00u, 0x3c003c00u, 0x3c003c00u);
  const uint4 wqa = p.q_norm_w ? __ldg(reinterpret_cast<const uint4*>(p.q_norm_w + 8 * l)) : one;
  const uint4 wqb =
      p.q_norm_w ? __ldg(reinterpret_cast<const uint4*>(p.q_norm_w + D / 2 + 8 * l)) : one;
  const uint4 wka = p.k_norm_w ? __ldg(reinterpret_cast<const uint4*>(p.k_norm_w + 8 * l)) : one;
  const uint4 wkb =
      p.k_norm_w ? __ldg(reinterpret_cast<const uint4*>(p.k_norm_w + D / 2 + 8 * l)) : one;
  const bool blk_ok = blk >= 0 && blk < p.num_blocks;
  if (!blk_ok && threadIdx.x == 0) atomicOr(&g_device_status, kDevBadBlockId);
  const size_t slot_row = ((size_t)(blk_ok ? blk : 0) * Hkv * BS + pos % BS) * D + 8 * l;

#pragma unroll
  for (int k = 0; k < NS; ++k) {
    const int hh = h0 + k * G;
    const uint32_t xa[4] = {ra[k].x, ra[k].y, ra[k].z, ra[k].w};
    const uint32_t xb[4] = {rb[k].x, rb[k].y, rb[k].z, rb[k].w};
    float a[8], b[8];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 fa = h2f(xa[j]), fb = h2f(xb[j]);
      a[2 * j] = fa.x;
      a[2 * j + 1] = fa.y;
      b[2 * j] = fb.x;
      b[2 * j + 1] = fb.y;
    }
    // sum of squares over the head's LPH lanes (every lane takes part)
    float ss = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) ss += a[j] * a[j] + b[j] * b[j];
#pragma unroll
    for (int o = 1; o < LPH; o <<= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if (hh >= heads) continue;
    if (hh >= H + Hkv) {  // value head: copied into the pool, bit for bit
      if (blk_ok) {
        __half* dst = p.v_cache + slot_row + (size_t)(hh - H - Hkv) * BS * D;
        *reinterpret_cast<uint4*>(dst) = ra[k];
        *reinterpret_cast<uint4*>(dst + D / 2) = rb[k];
      }
      continue;
    }
    const bool is_q = hh < H;
    __half* dst;
    if (is_q) {
      dst = p.q_out + ((size_t)row * H + hh) * D + 8 * l;
    } else {
      if (!blk_ok) continue;
      dst = p.k_cache + slot_row + (size_t)(hh - H) * BS * D;
    }
    if (is_q ? p.q_norm_w != nullptr : p.k_norm_w != nullptr) {
      const float rr = rsqrtf(ss / (float)D + p.eps);
      const uint4 wa4 = is_q ? wqa : wka, wb4 = is_q ? wqb : wkb;
      const uint32_t wa[4] = {wa4.x, wa4.y, wa4.z, wa4.w};
      const uint32_t wb[4] = {wb4.x, wb4.y, wb4.z, wb4.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float2 fa = h2f(wa[j]), fb = h2f(wb[j]);
        a[2 * j] = a[2 * j] * rr * fa.x;
        a[2 * j + 1] = a[2 * j + 1] * rr * fa.y;
        b[2 * j] = b[2 * j] * rr * fb.x;
        b[2 * j + 1] = b[2 * j + 1] * rr * fb.y;
      }
    }
    uint32_t oa[4], ob[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int e = 2 * j, f = 2 * j + 1;
      oa[j] = f2h(a[e] * cs[e] - b[e] * sn[e], a[f] * cs[f] - b[f] * sn[f]);
      ob[j] = f2h(b[e] * cs[e] + a[e] * sn[e], b[f] * cs[f] + a[f] * sn[f]);
    }
    *reinterpret_cast<uint4*>(dst) = make_uint4(oa[0], oa[1], oa[2], oa[3]);
    *reinterpret_cast<uint4*>(dst + D / 2) = make_uint4(ob[0], ob[1], ob[2], ob[3]);
  }
}

// ---------------------------------------------------------------------------
// decode
// ---------------------------------------------------------------------------

struct DecodeParams {
  const __half* q;              // [B][H][D]
  const int32_t* block_tables;  // [B][MBPS]
  const int32_t* context_lens;  // [B]
  __half* out;                  // [B][H][D]             (single pass)
  float* part_out;              // [B][H][S][D]          (split-K)
  float* part_m;                // [B][H][S]  base-2 running max
  float* part_l;                // [B][H][S]  running sum
  int num_seqs;
  int num_heads;
  int num_kv_heads;
  int group;
  int max_blocks_per_seq;
  int num_blocks;
  int num_splits;  // S (1 for single pass)
  // Split-K chunks are cut on the device from the longest context of the
  // call: chunk = max(min_chunk_blocks, ceil(ceil(Lmax / BS) / S)) blocks,
  // so tables sized for a larger maximum context than the call holds still
  // spread the work over every split.
  int min_chunk_blocks;
  // The host's guess of the chunk, ceil(max_blocks_per_seq / S): when it is
  // right the first table entry of a chunk is loaded before Lmax is known.
  int chunk_hint;
  int* split_header;  // split-K: where phase 1 leaves the chunk size for the combine
  float scale_log2;   // scale * log2(e)
  // Fair-share depth (set when the whole grid is resident at once): a CTA
  // keeps copies in flight in proportion to its share of the longest chunk
  // in the call.  HBM serves outstanding requests about evenly, so every CTA
  // then progresses at the same fraction of its work and they end together.
  int fair_depth;
  // Fused append (pkv_append_decode; FUSE kernels only): token s is sequence s's
  // newest position context_lens[s] - 1, written at new_slots[s] (< 0: none).
  const __half* k_new;  // [B][Hkv][D]
  const __half* v_new;
  const int32_t* new_slots;  // [B]
  __half* k_cache;           // the pools, for the row writes
  __half* v_cache;
  // Fused QKV step (pkv_qkv_rope_append_decode; QKV kernels only): sequence
  // s's newest token (position context_lens[s] - 1) comes as its fused
  // projection row; the kernel norms and rotates its query and key heads
  // (as qkv_norm_rope_kernel does), attends with the queries and appends
  // the key and value rows.
  const __half* qkv;       // [B][(H + 2 Hkv) D]
  const __half* q_norm_w;  // [D] or null
  const __half* k_norm_w;  // [D] or null
  const float* cos_t;      // [max_pos][D/2]
  const float* sin_t;
  int max_pos;
  float eps;
};

template <int D, int BS, int W, int P>
struct DecodeShape {
  static constexpr int kTileBytes = BS * D * 2;  // one K (or V) tile
  static constexpr int kStageBytes = 2 * kTileBytes;
  static constexpr int kRingBytes = W * P * kStageBytes;
  static constexpr int kBarrierBytes = W * P * 8;
  static constexpr int kSmemBytes = 1024 + kRingBytes + kBarrierBytes;  // +1024: alignment slack
  static constexpr int kMT = BS / 16;     // 16-token slices per tile
  static constexpr int kKS = D / 16;      // 16-wide slices of head_dim
  static constexpr int kHalves = D / 64;  // 128-byte lines per row
  static constexpr int kRedFloats = 16 + 8 * D;  // per warp: m[8], l[8], o[8][D]
  static_assert(kTileBytes % 1024 == 0, "tiles must keep 1024-byte alignment for the swizzle");
  static_assert(W * kRedFloats * 4 <= kRingBytes, "the merge area reuses the ring");
};

// Byte offset of element (row, d) inside a tile stored as [D/64][BS][64] f16
// with the TMA 128-byte swizzle (16-byte chunk index XOR row % 8).
template <int BS>
__device__ __forceinline__ uint32_t swz(int row, int d) {
  const int line = (d >> 6) * BS + row;
  const int chunk = ((d & 63) >> 3) ^ (row & 7);
  return (uint32_t)(line * 128 + chunk * 16 + (d & 7) * 2);
}

// vLLM-layout tiles in shared memory.  K [D/8][BS][8] arrives unchanged
// (16-byte chunk (d/8, row) at (d/8 * BS + row) * 16; eight consecutive rows
// of one chunk column are 128 contiguous bytes, so ldmatrix is conflict-free
// without a swizzle).  V^T [D][BS] arrives through TMA as 128-byte lines
// (128 / (2 BS) rows of d per line) with the 128-byte swizzle (16-byte chunk
// index XOR line % 8); the 8 rows d..d+7 of one ldmatrix then fall on 8
// distinct bank groups for BS 16 and 32 alike.
template <int BS>
__device__ __forceinline__ uint32_t vllm_k_off(int row, int d) {
  return (uint32_t)(((d >> 3) * BS + row) * 16 + (d & 7) * 2);
}

template <int BS>
__device__ __forceinline__ uint32_t vllm_vt_off(int d, int tok) {
  const uint32_t off = (uint32_t)(d * BS * 2 + tok * 2);
  return off ^ (((off >> 7) & 7u) << 4);
}

// One warp's online-softmax state.  Lane (r = lane/4, c = lane%4) holds the
// O^T fragments of rows d = 16*i + r (+8) for query heads 2c and 2c+1, the
// running max of those two heads (shared by the 8 lanes of a column) and its
// own share of their running sums.
template <int D>
struct WarpState {
  float acc[D / 16][4];
  float m0, m1, l0, l1;

  __device__ __forceinline__ void reset() {
#pragma unroll
    for (int i = 0; i < D / 16; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
    m0 = m1 = -CUDART_INF_F;
    l0 = l1 = 0.f;
  }

  // Completes the running sums across the 8 lanes of each head column.
  __device__ __forceinline__ void finish_sums() {
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      l0 += __shfl_xor_sync(0xffffffffu, l0, o);
      l1 += __shfl_xor_sync(0xffffffffu, l1, o);
    }
  }

  // Writes m[8], l[8] and o[heads][D] (heads 0..heads-1 of the group) at `dst`.
  __device__ __forceinline__ void store(float* dst, int lane, int heads) const {
    const int r = lane >> 2, c = lane & 3;
    if (r == 0) {
      dst[2 * c] = m0;
      dst[2 * c + 1] = m1;
      dst[8 + 2 * c] = l0;
      dst[8 + 2 * c + 1] = l1;
    }
    float* o = dst + 16;
#pragma unroll
    for (int i = 0; i < D / 16; ++i) {
      const int d = i * 16 + r;
      if (2 * c < heads) {
        o[(2 * c) * D + d] = acc[i][0];
        o[(2 * c) * D + d + 8] = acc[i][2];
      }
      if (2 * c + 1 < heads) {
        o[(2 * c + 1) * D + d] = acc[i][1];
        o[(2 * c + 1) * D + d + 8] = acc[i][3];
      }
    }
  }
};

// The pair layout of one head (or weight vector) of D halves: lane holds
// elements PL*lane .. +PL and the same + D/2 (PL = D/64), so that each lane
// has both halves of its rotate-half pairs.  `lo` / `hi` pack them: PL = 2,
// one half2 word each; PL = 1, one half in the low bits.  Plain loads (the
// source may be global or shared memory).
template <int D>
__device__ __forceinline__ void load_pairs(const __half* x, int lane, uint32_t& lo, uint32_t& hi) {
  constexpr int PL = D / 64;
  const int i0 = PL * lane;
  if (PL == 2) {
    lo = *reinterpret_cast<const uint32_t*>(x + i0);
    hi = *reinterpret_cast<const uint32_t*>(x + i0 + D / 2);
  } else {
    lo = *reinterpret_cast<const unsigned short*>(x + i0);
    hi = *reinterpret_cast<const unsigned short*>(x + i0 + D / 2);
  }
}

template <int D>
__device__ __forceinline__ void unpack_pairs(uint32_t v, float (&f)[D / 64]) {
  if (D / 64 == 2) {
    const float2 t = __half22float2(*reinterpret_cast<const __half2*>(&v));
    f[0] = t.x;
    f[D / 64 - 1] = t.y;
  } else {
    f[0] = __half2float(__ushort_as_half((unsigned short)v));
  }
}

// The rotary angles of one position for the lane's pairs.
template <int D>
__device__ __forceinline__ void load_angles(const float* cs_row, const float* sn_row, int lane,
                                            float (&c)[D / 64], float (&sn)[D / 64]) {
#pragma unroll
  for (int j = 0; j < D / 64; ++j) {
    c[j] = __ldg(cs_row + (D / 64) * lane + j);
    sn[j] = __ldg(sn_row + (D / 64) * lane + j);
  }
}

// One query or key head in the pair layout, RMS-normed over its D elements
// when `has_w` (weights in the pair layout) and turned by the lane's rotary
// angles (rotate-half pairs (i, i + D/2)); f32, rounded once to f16; the
// result in the pair layout.  All lanes of the warp take part.
template <int D>
__device__ __forceinline__ void norm_rotate_pairs(uint32_t xlo, uint32_t xhi, bool has_w,
                                                  uint32_t wlo, uint32_t whi,
                                                  const float (&c)[D / 64],
                                                  const float (&sn)[D / 64], float eps,
                                                  uint32_t& lo, uint32_t& hi) {
  constexpr int PL = D / 64;
  float a[PL], b[PL];
  unpack_pairs<D>(xlo, a);
  unpack_pairs<D>(xhi, b);
  if (has_w) {
    float ss = 0.f;
#pragma unroll
    for (int j = 0; j < PL; ++j) ss += a[j] * a[j] + b[j] * b[j];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    const float rr = rsqrtf(ss / (float)D + eps);
    float wa[PL], wb[PL];
    unpack_pairs<D>(wlo, wa);
    unpack_pairs<D>(whi, wb);
#pragma unroll
    for (int j = 0; j < PL; ++j) {
      a[j] = a[j] * rr * wa[j];
      b[j] = b[j] * rr * wb[j];
    }
  }
  float oa[PL], ob[PL];
#pragma unroll
  for (int j = 0; j < PL; ++j) {
    oa[j] = a[j] * c[j] - b[j] * sn[j];
    ob[j] = b[j] * c[j] + a[j] * sn[j];
  }
  if (PL == 2) {
    lo = pack_half2(__floats2half2_rn(oa[0], oa[PL - 1]));
    hi = pack_half2(__floats2half2_rn(ob[0], ob[PL - 1]));
  } else {
    lo = (uint32_t)__half_as_ushort(__float2half_rn(oa[0]));
    hi = (uint32_t)__half_as_ushort(__float2half_rn(ob[0]));
  }
}

// Stores a head in the pair layout (see load_pairs) at `dst` (global or shared).
template <int D>
__device__ __forceinline__ void store_pairs(__half* dst, int lane, uint32_t lo, uint32_t hi) {
  constexpr int PL = D / 64;
  const int i0 = PL * lane;
  if (PL == 2) {
    *reinterpret_cast<uint32_t*>(dst + i0) = lo;
    *reinterpret_cast<uint32_t*>(dst + i0 + D / 2) = hi;
  } else {
    dst[i0] = __ushort_as_half((unsigned short)lo);
    dst[i0 + D / 2] = __ushort_as_half((unsigned short)hi);
  }
}

// Q^T fragments from query heads held in shared memory [8][D] (heads at or
// past `group` are zero), same layout as load_q_frags.
template <int D>
__device__ __forceinline__ void load_q_frags_smem(uint32_t (&qf)[D / 16][2], const __half* sq,
                                                  int group, int lane) {
  const int r = lane >> 2, c = lane & 3;
  const bool live = r < group;
  const uint32_t* qrow = reinterpret_cast<const uint32_t*>(sq + (live ? r : 0) * D);
#pragma unroll
  for (int ks = 0; ks < D / 16; ++ks) {
    qf[ks][0] = live ? qrow[ks * 8 + c] : 0u;
    qf[ks][1] = live ? qrow[ks * 8 + 4 + c] : 0u;
  }
}

// Q^T fragments (B operand): column n = lane/4 is query head `head0 + n`;
// columns at or past `group` are zero.
template <int D>
__device__ __forceinline__ void load_q_frags(uint32_t (&qf)[D / 16][2], const __half* q,
                                             size_t head0, int group, int lane) {
  const int r = lane >> 2, c = lane & 3;
  const bool live = r < group;
  const uint32_t* qrow = reinterpret_cast<const uint32_t*>(q + (head0 + (live ? r : 0)) * D);
#pragma unroll
  for (int ks = 0; ks < D / 16; ++ks) {
    qf[ks][0] = live ? __ldg(qrow + ks * 8 + c) : 0u;
    qf[ks][1] = live ? __ldg(qrow + ks * 8 + 4 + c) : 0u;
  }
}

// Folds one K/V tile (already in shared memory at kb / vb) into NT warp
// states, one per 8-column n-tile of queries (each K and V fragment read
// from shared memory serves all NT tiles).  Token t0 is the tile's first
// position; positions at or past tok_end are masked, and with COLMASK each
// lane's two columns of n-tile nt also stop at lim[nt][0] / lim[nt][1].
// VLLM: the tiles are in the vLLM layout (see vllm_k_off / vllm_vt_off)
// instead of the swizzled [D/64][BS][64].
template <int D, int BS, int NT, bool COLMASK, bool VLLM>
__device__ __forceinline__ void consume_tiles(uint32_t kb, uint32_t vb, int t0, int tok_end,
                                              const uint32_t (&qf)[NT][D / 16][2],
                                              float scale_log2, WarpState<D> (&st)[NT], int lane,
                                              const int (&lim)[NT][2]) {
  constexpr int MT = BS / 16;
  constexpr int KS = D / 16;
  constexpr int HALVES = D / 64;
  const int r = lane >> 2;
  const int n_valid = min(BS, tok_end - t0);
  if (n_valid < BS) {
    // Rows past the context may hold anything (even NaN); P is 0 there, but
    // 0 * NaN is NaN, so clear those V rows before P.V.
    if (VLLM) {
      // V^T: the tokens are columns; clear them chunk by chunk (8 tokens)
      const int c0 = n_valid >> 3;
      const int n_chunks = (BS / 8 - c0) * D;
      for (int x = lane; x < n_chunks; x += 32) {
        const int d = x % D;
        const int ch = c0 + x / D;
        const uint32_t a = vb + vllm_vt_off<BS>(d, ch * 8);
        uint32_t w[4];
        asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3])
                     : "r"(a));
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int tk = ch * 8 + 2 * e;  // tokens tk (low half) and tk + 1
          if (tk >= n_valid) w[e] = 0u;
          else if (tk + 1 >= n_valid) w[e] &= 0xffffu;
        }
        asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(w[0]), "r"(w[1]),
                     "r"(w[2]), "r"(w[3])
                     : "memory");
      }
    } else {
      const int n_chunks = (BS - n_valid) * HALVES * 8;
      for (int x = lane; x < n_chunks; x += 32) {
        const int row = n_valid + x / (HALVES * 8);
        const int rest = x % (HALVES * 8);
        const int line = (rest >> 3) * BS + row;
        const uint32_t a = vb + line * 128 + (rest & 7) * 16;
        asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(a), "r"(0) : "memory");
      }
    }
    __syncwarp();
  }

  // S^T = K . Q^T for every 16-token slice of the tile and every n-tile (two
  // accumulators per slice halve the dependent mma chain).
  float sc[MT][NT][4];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt) {
    float s2[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      s2[nt][0] = s2[nt][1] = s2[nt][2] = s2[nt][3] = 0.f;
      sc[mt][nt][0] = sc[mt][nt][1] = sc[mt][nt][2] = sc[mt][nt][3] = 0.f;
    }
    const int row = mt * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      uint32_t a[4];
      if (VLLM)
        ldsm_x4(kb + vllm_k_off<BS>(row, ks * 16 + (lane >> 4) * 8), a);
      else
        ldsm_x4(kb + swz<BS>(row, ks * 16 + (lane >> 4) * 8), a);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        if (PKV_QK_SPLIT && (ks & 1))
          mma_16816(s2[nt], a, qf[nt][ks][0], qf[nt][ks][1]);
        else
          mma_16816(sc[mt][nt], a, qf[nt][ks][0], qf[nt][ks][1]);
      }
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) sc[mt][nt][e] += s2[nt][e];
  }

#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    WarpState<D>& w = st[nt];
    // scale, mask rows past the context, tile max per column
    float x0 = -CUDART_INF_F, x1 = -CUDART_INF_F;
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int tok = t0 + mt * 16 + r + (e >> 1) * 8;
        const float v = sc[mt][nt][e] * scale_log2;
        // COLMASK: each column (query) has its own causal limit
        const int lm = COLMASK ? lim[nt][e & 1] : tok_end;
        sc[mt][nt][e] = tok < lm ? v : -CUDART_INF_F;
      }
      x0 = fmaxf(x0, fmaxf(sc[mt][nt][0], sc[mt][nt][2]));
      x1 = fmaxf(x1, fmaxf(sc[mt][nt][1], sc[mt][nt][3]));
    }
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      x0 = fmaxf(x0, __shfl_xor_sync(0xffffffffu, x0, o));
      x1 = fmaxf(x1, __shfl_xor_sync(0xffffffffu, x1, o));
    }
    float mn0 = fmaxf(w.m0, x0);
    float mn1 = fmaxf(w.m1, x1);
    float al0 = exp2f(w.m0 - mn0);  // 0 on the first tile (m = -inf)
    float al1 = exp2f(w.m1 - mn1);
    w.m0 = mn0;
    w.m1 = mn1;
    if (COLMASK) {
      // a column with nothing valid so far keeps m = -inf: no rescale, P = 0
      if (mn0 == -CUDART_INF_F) { al0 = 1.f; mn0 = 0.f; }
      if (mn1 == -CUDART_INF_F) { al1 = 1.f; mn1 = 0.f; }
    }

    // P = exp2(S - m), rounded to f16 for the tensor cores; the running sum
    // adds the same rounded values so numerator and denominator agree.  P^T
    // overwrites the scores of this n-tile (as two packed registers).
    float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
      const __half2 h01 =
          __floats2half2_rn(exp2f(sc[mt][nt][0] - mn0), exp2f(sc[mt][nt][1] - mn1));
      const __half2 h23 =
          __floats2half2_rn(exp2f(sc[mt][nt][2] - mn0), exp2f(sc[mt][nt][3] - mn1));
      const float2 f01 = __half22float2(h01);
      const float2 f23 = __half22float2(h23);
      ps0 += f01.x + f23.x;
      ps1 += f01.y + f23.y;
      sc[mt][nt][0] = __uint_as_float(movmatrix_trans(pack_half2(h01)));
      sc[mt][nt][1] = __uint_as_float(movmatrix_trans(pack_half2(h23)));
    }
    w.l0 = w.l0 * al0 + ps0;
    w.l1 = w.l1 * al1 + ps1;
#pragma unroll
    for (int i = 0; i < KS; ++i) {
      w.acc[i][0] *= al0;
      w.acc[i][1] *= al1;
      w.acc[i][2] *= al0;
      w.acc[i][3] *= al1;
    }
  }

  // O^T += V^T . P^T (V^T fragments: matrix lane/8 covers d rows +8*(bit 0),
  // token columns +8*(bit 1))
#pragma unroll
  for (int mt = 0; mt < MT; ++mt) {
    const int row = mt * 16 + (lane & 7) + (lane >> 4) * 8;
#pragma unroll
    for (int i = 0; i < KS; ++i) {
      uint32_t a[4];
      if (VLLM)
        ldsm_x4(vb + vllm_vt_off<BS>(i * 16 + ((lane >> 3) & 1) * 8 + (lane & 7),
                                     mt * 16 + (lane >> 4) * 8),
                a);
      else
        ldsm_x4_trans(vb + swz<BS>(row, i * 16 + ((lane >> 3) & 1) * 8), a);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
        mma_16816(st[nt].acc[i], a, __float_as_uint(sc[mt][nt][0]),
                  __float_as_uint(sc[mt][nt][1]));
    }
  }
}

// One n-tile (the decode kernels: the 8 columns are the GQA group).
template <int D, int BS, bool COLMASK = false, bool VLLM = false>
__device__ __forceinline__ void consume_tile(uint32_t kb, uint32_t vb, int t0, int tok_end,
                                             const uint32_t (&qf)[D / 16][2], float scale_log2,
                                             WarpState<D>& st, int lane, int lim0 = 0,
                                             int lim1 = 0) {
  const int lim[1][2] = {{lim0, lim1}};
  consume_tiles<D, BS, 1, COLMASK, VLLM>(
      kb, vb, t0, tok_end, reinterpret_cast<const uint32_t(&)[1][D / 16][2]>(qf), scale_log2,
      reinterpret_cast<WarpState<D>(&)[1]>(st), lane, lim);
}

// Log-sum-exp merge of W warp states stored with WarpState::store (stride
// `stride` floats per warp) for head h, element d.
template <int W, int D>
__device__ __forceinline__ void merge_warps(const float* red, int stride, int h, int d, float& M,
                                            float& num, float& den) {
  M = -CUDART_INF_F;
#pragma unroll
  for (int w = 0; w < W; ++w) M = fmaxf(M, red[w * stride + h]);
  num = 0.f;
  den = 0.f;
#pragma unroll
  for (int w = 0; w < W; ++w) {
    const float mw = red[w * stride + h];
    const float f = (mw == -CUDART_INF_F) ? 0.f : exp2f(mw - M);
    num += f * red[w * stride + 16 + h * D + d];
    den += f * red[w * stride + 8 + h];
  }
}

// Starts the TMA copies of the K and V tiles of (physical block, kv head)
// into the stage at `kdst` (V follows K), completing on `bar`.  Blocked
// pools: one tensor box of TR = 16 rows per tile, from row `row0` of the
// block (landing as [D/64][16][64], swizzled).  VLLM: a whole block (TR =
// block size); K is one contiguous bulk copy from `kpool`, V one 3-D tensor
// copy.
template <int D, int TR, bool VLLM = false>
__device__ __forceinline__ void issue_tile_copy(uint32_t kdst, uint32_t bar, int tile, int row0,
                                                const CUtensorMap* kmap, const CUtensorMap* vmap,
                                                const __half* kpool = nullptr) {
  constexpr int TB = TR * D * 2;
  mbar_arrive_expect_tx(bar, 2 * TB);
  if (VLLM) {
    bulk_load(kdst, kpool + (size_t)tile * (TR * D), TB, bar);
    tma_load_3d(kdst + TB, vmap, bar, 0, 0, tile);
  } else {
    tma_load_4d(kdst, kmap, bar, 0, row0, 0, tile);
    tma_load_4d(kdst + TB, vmap, bar, 0, row0, 0, tile);
  }
}

// Staging in 16-row sub-tiles for blocked pools (build flag; see the kernel).
#ifndef PKV_SUBTILE
#define PKV_SUBTILE 1
#endif
constexpr bool kSubtile = PKV_SUBTILE != 0;

// VLLM: the pools are in the vLLM layout (p.k_cache is the K pool; kmap is
// unused); no fused append.  Single pass: one CTA per (sequence, KV head).
// Split-K phase 1: one CTA per (sequence, KV head, chunk); a chunk past the
// sequence's end exits at once, a (sequence, KV head) whose context fits one
// chunk is finished here (f16 output, the combine skips it), and the others
// leave f32 partials per chunk for the combine.
template <int D, int BS, int W, int P, bool SPLIT, bool FUSE, bool VLLM = false, bool QKV = false>
__global__ void __launch_bounds__(W * 32)
paged_decode_kernel(const __grid_constant__ CUtensorMap kmap,
                    const __grid_constant__ CUtensorMap vmap, const DecodeParams p) {
  static_assert(!(FUSE && VLLM), "the fused append writes the blocked layout only");
  static_assert(!(QKV && (FUSE || VLLM)), "the fused QKV step is its own variant");
  // Staging tiles hold TR rows of one (block, KV head).  A blocked pool is
  // read in 16-row sub-tiles, SUB per block, so every block size keeps the
  // same stage size and ring depth; the vLLM layout stages whole blocks.
  // Tile indices below count these sub-tiles.
  constexpr int TR = (VLLM || !kSubtile) ? BS : 16;
  constexpr int SUB = BS / TR;
  using Shape = DecodeShape<D, TR, W, P>;
  constexpr int KS = Shape::kKS;
  constexpr int TB = Shape::kTileBytes;
  constexpr int PL = D / 64;
  constexpr int HPL = D / 32;  // halves per lane of one row

  extern __shared__ uint8_t smem_raw[];
  __shared__ int s_failed;
  __shared__ int s_max[W];
  __shared__ __align__(16) __half s_q[QKV ? 8 * D : 2];   // QKV: the group's rotated queries
  __shared__ __align__(16) __half s_kv[QKV ? 2 * D : 2];  // QKV: the new key and value rows
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t ring = smem_addr(smem);
  const uint32_t bars = ring + Shape::kRingBytes;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int Hkv = p.num_kv_heads;

  pdl_launch_dependents();
  // Barrier set-up touches no global memory: before the dependency wait.
  if (threadIdx.x == 0) s_failed = 0;
  const uint32_t my_bars = bars + warp * P * 8;
  if (lane == 0) {
#pragma unroll
    for (int i = 0; i < P; ++i) mbar_init(my_bars + 8 * i, 1);
    fence_mbar_init();
  }
  pdl_wait();

  const int cap = p.max_blocks_per_seq * BS;
  // The CTA's work: sequence s, KV head g and (split) chunk `piece`.  Every
  // independent global load of the prologue goes out together: the status
  // word, the length, the warp's first block-table entry (its first tile is
  // the chunk's tile `warp` whatever the fair share decides; the entry is in
  // bounds and only used if the tile exists; split kernels load it under
  // the host's chunk guess), the fused slot, (QKV) the raw projection-row
  // heads, and every length (the longest context sets the split chunks and
  // the fair share).
  int item = blockIdx.x;
  const int piece = SPLIT ? item % p.num_splits : 0;
  if (SPLIT) item /= p.num_splits;
  const int g = item % Hkv;
  const int s = item / Hkv;
  const int32_t* table = p.block_tables + (size_t)s * p.max_blocks_per_seq;
  const unsigned int status = *reinterpret_cast<volatile unsigned int*>(&g_device_status);
  // QKV: the warp's query heads (warp, warp + W) of the projection row, the
  // norm weights, and in warp W-1 the KV head's key and value heads.
  uint32_t xq[2][2] = {{0u, 0u}, {0u, 0u}}, wq[2] = {0u, 0u};
  uint32_t xk[2] = {0u, 0u}, xv[2] = {0u, 0u}, wk[2] = {0u, 0u};
  if (QKV) {
    const int H = p.num_heads;
    const __half* row = p.qkv + (size_t)s * (H + 2 * Hkv) * D;
#pragma unroll
    for (int j = 0; j < 2; ++j)
      if (warp + j * W < p.group)
        load_pairs<D>(row + (size_t)(g * p.group + warp + j * W) * D, lane, xq[j][0], xq[j][1]);
    if (p.q_norm_w && warp < p.group) load_pairs<D>(p.q_norm_w, lane, wq[0], wq[1]);
    if (warp == W - 1) {
      load_pairs<D>(row + (size_t)(H + g) * D, lane, xk[0], xk[1]);
      load_pairs<D>(row + (size_t)(H + Hkv + g) * D, lane, xv[0], xv[1]);
      if (p.k_norm_w) load_pairs<D>(p.k_norm_w, lane, wk[0], wk[1]);
    }
  }
  int L = __ldg(p.context_lens + s);
  const int j0_guess = (SPLIT ? piece * p.chunk_hint * SUB : 0) + warp;  // in tiles
  const int phys0_guess =
      (lane == 0 && j0_guess / SUB < p.max_blocks_per_seq) ? __ldg(table + j0_guess / SUB) : -1;
  const int slot_new = FUSE ? __ldg(p.new_slots + s) : -1;
  const bool need_max = SPLIT || p.fair_depth;
  if (need_max) {
    int mx = 0;
    for (int i = threadIdx.x; i < p.num_seqs; i += W * 32) {
      int Li = __ldg(p.context_lens + i);
      if (SPLIT && blockIdx.x == 0 && (Li < 0 || Li > cap)) atomicOr(&g_device_status, kDevBadContextLen);
      Li = Li < 0 ? 0 : (Li > cap ? cap : Li);
      mx = max(mx, (Li + BS - 1) / BS);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if (lane == 0) s_max[warp] = mx;
  }

  // After a lost copy has been flagged, later CTAs do no work (and write
  // nothing) until the host reads and clears the status word.  The decision
  // is made for the whole CTA at once.  (The barrier also publishes s_max.)
  if (__syncthreads_or(status & kDevWaitTimeout)) return;
  int nblk_max = 0;  // the call's longest context, in blocks
  if (need_max) {
#pragma unroll
    for (int w = 0; w < W; ++w) nblk_max = max(nblk_max, s_max[w]);
  }
  const int chunk = SPLIT ? max(p.min_chunk_blocks, (nblk_max + p.num_splits - 1) / p.num_splits)
                          : p.max_blocks_per_seq;

  if (SPLIT && blockIdx.x == 0 && threadIdx.x == 0) *p.split_header = chunk;  // for the combine

  if (L < 0 || L > cap) {  // (split kernels flag it once, in CTA 0's scan)
    if (!SPLIT && threadIdx.x == 0) atomicOr(&g_device_status, kDevBadContextLen);
    L = L < 0 ? 0 : cap;
  }
  int tok_begin = 0;
  int tok_end = L;
  int n_pieces = 1;  // chunks of this sequence (1: this CTA writes the output)
  if (SPLIT) {
    const int nb = (L + BS - 1) / BS;
    n_pieces = (nb + chunk - 1) / chunk;
    if ((long long)piece * chunk >= nb) return;  // past the sequence's end
    tok_begin = piece * chunk * BS;
    tok_end = (int)min((long long)L, (long long)tok_begin + (long long)chunk * BS);
  }
  // QKV: a newest position without rotary angles is flagged; the sequence
  // then attends with zero queries and appends nothing (its output is
  // written but meaningless).
  const bool qkv_bad = QKV && L > p.max_pos;
  if (qkv_bad && threadIdx.x == 0) atomicOr(&g_device_status, kDevBadContextLen);
  float ang_c[PL], ang_s[PL];  // QKV: the rotary angles of position L-1
  if (QKV && !qkv_bad && L > 0 && (warp < p.group || warp == W - 1))
    load_angles<D>(p.cos_t + (size_t)(L - 1) * (D / 2), p.sin_t + (size_t)(L - 1) * (D / 2),
                   lane, ang_c, ang_s);
  const int sub_begin = tok_begin / TR;  // the chunk's first tile
  const int n_tiles = (tok_end - tok_begin + TR - 1) / TR;
  // the first tile's table entry: the prologue's guess when it was right
  const int phys0 = (!SPLIT || piece == 0 || chunk == p.chunk_hint)
                        ? phys0_guess
                        : ((lane == 0 && (sub_begin + warp) / SUB < p.max_blocks_per_seq)
                               ? __ldg(table + (sub_begin + warp) / SUB)
                               : -1);

  // Warps that take tiles: all W, or (fair share) W scaled by this chunk's
  // tiles over the longest chunk of the call.
  int WE = W;
  if (p.fair_depth) {
    const int mx = (SPLIT ? min(nblk_max, chunk) : nblk_max) * SUB;
    if (mx > 0) WE = max(1, min(W, (W * n_tiles + mx - 1) / mx));
  }
  const int my_tiles = (warp < WE && n_tiles > warp) ? (n_tiles - warp + WE - 1) / WE : 0;

  // Fused append: the CTA whose chunk holds position L-1 writes this KV
  // head's new row into the pools and, for its own attention, patches the
  // row into that tile in shared memory once the tile's copy has landed (so
  // it never depends on the global write being visible to its TMA reads).
  // A slot other than that position's is neither written nor used: flagged.
  int fuse_li = -1;  // local tile index of the new row, in its owner warp
  int fuse_row = 0;  // its row in that tile
  int kv_phys = -1;  // QKV: the new row's block when this CTA holds it
  int kv_prow = 0;   // and its row in the block
  uint32_t kn[HPL / 2], vn[HPL / 2];
  if ((FUSE || QKV) && !qkv_bad && L > 0 && L - 1 >= tok_begin && L - 1 < tok_end &&
      (QKV || slot_new >= 0)) {
    const int pos = L - 1;
    const int phys = __ldg(table + pos / BS);
    const bool ok =
        phys >= 0 && phys < p.num_blocks && (QKV || slot_new == phys * BS + pos % BS);
    if (!ok) {
      if (threadIdx.x == 0) atomicOr(&g_device_status, kDevBadSlot);
    } else {
      const int idx = pos / TR - sub_begin;  // tile within the chunk
      fuse_row = pos % TR;
      if (QKV) {
        // the row is computed after the first copies are issued (below)
        kv_phys = phys;
        kv_prow = pos % BS;
        if (warp == idx % WE) fuse_li = idx / WE;
      } else if (warp == idx % WE) {
        fuse_li = idx / WE;
        const size_t src = ((size_t)s * Hkv + g) * D + lane * HPL;
        const size_t dst = (((size_t)phys * Hkv + g) * BS + pos % BS) * D + lane * HPL;
#pragma unroll
        for (int x = 0; x < HPL / 2; ++x) {
          kn[x] = __ldg(reinterpret_cast<const uint32_t*>(p.k_new + src) + x);
          vn[x] = __ldg(reinterpret_cast<const uint32_t*>(p.v_new + src) + x);
          reinterpret_cast<uint32_t*>(p.k_cache + dst)[x] = kn[x];
          reinterpret_cast<uint32_t*>(p.v_cache + dst)[x] = vn[x];
        }
      }
    }
  }

  auto k_stage = [&](int stage) { return ring + (warp * P + stage) * Shape::kStageBytes; };

  // Lane 0: start the copies of this warp's local tile `li` into its stage
  // (tile 0's entry was loaded in the prologue).
  auto issue = [&](int li) {
    const int stage = li % P;
    const int j = sub_begin + warp + li * WE;
    const int phys = (li == 0) ? phys0 : __ldg(table + j / SUB);
    const uint32_t bar = my_bars + 8 * stage;
    if (phys >= 0 && phys < p.num_blocks) {
      issue_tile_copy<D, TR, VLLM>(k_stage(stage), bar, phys * Hkv + g, (j % SUB) * TR, &kmap,
                                   &vmap, p.k_cache);
    } else {
      atomicOr(&g_device_status, kDevBadBlockId);
      mbar_arrive(bar);
    }
  };

  if (lane == 0) {
    const int n0 = my_tiles < P ? my_tiles : P;
    for (int li = 0; li < n0; ++li) issue(li);
  }

  uint32_t qf[KS][2];
  uint32_t qk_lo = 0, qk_hi = 0, qv_lo = 0, qv_hi = 0;  // QKV: the new key / value row
  if (QKV) {
    // With the first copies in flight: the group's queries (norm + rotary
    // at position L-1) into shared memory; warp W-1 turns the new key row,
    // writes key and value rows to the pools and leaves them in shared
    // memory for the warp whose tile holds them.
    if (L > 0 && !qkv_bad) {
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int h = warp + j * W;
        if (h < p.group) {
          uint32_t lo, hi;
          norm_rotate_pairs<D>(xq[j][0], xq[j][1], p.q_norm_w != nullptr, wq[0], wq[1], ang_c,
                               ang_s, p.eps, lo, hi);
          store_pairs<D>(s_q + h * D, lane, lo, hi);
        }
      }
      if (warp == W - 1 && kv_phys >= 0) {
        uint32_t lo, hi;
        norm_rotate_pairs<D>(xk[0], xk[1], p.k_norm_w != nullptr, wk[0], wk[1], ang_c, ang_s,
                             p.eps, lo, hi);
        const size_t dst = (((size_t)kv_phys * Hkv + g) * BS + kv_prow) * D;
        store_pairs<D>(p.k_cache + dst, lane, lo, hi);
        store_pairs<D>(p.v_cache + dst, lane, xv[0], xv[1]);
        store_pairs<D>(s_kv, lane, lo, hi);
        store_pairs<D>(s_kv + (QKV ? D : 0), lane, xv[0], xv[1]);
      }
    } else {
      for (int i = threadIdx.x; i < 8 * D / 2; i += W * 32)
        reinterpret_cast<uint32_t*>(s_q)[i] = 0u;
    }
    __syncthreads();
    load_q_frags_smem<D>(qf, s_q, p.group, lane);
    if (fuse_li >= 0) {
      load_pairs<D>(s_kv, lane, qk_lo, qk_hi);
      load_pairs<D>(s_kv + (QKV ? D : 0), lane, qv_lo, qv_hi);
    }
  } else {
    load_q_frags<D>(qf, p.q, (size_t)s * p.num_heads + (size_t)g * p.group, p.group, lane);
  }

  WarpState<D> st;
  st.reset();
  bool failed = false;
  int li = 0;

  for (; li < my_tiles; ++li) {
    const int stage = li % P;
    const uint32_t bar = my_bars + 8 * stage;
    if (!mbar_wait_bounded(bar, (li / P) & 1, kWaitLimitNs)) {
      failed = true;
      break;
    }
    const int j = sub_begin + warp + li * WE;
    const int phys = __ldg(table + j / SUB);
    if (phys >= 0 && phys < p.num_blocks) {
      const uint32_t kb = k_stage(stage);
      if (QKV && li == fuse_li) {
        // the new row of this tile is the one computed above, not the copy
        const int i0 = PL * lane;
        if (PL == 2) {
          asm volatile("st.shared.u32 [%0], %1;" ::"r"(kb + swz<TR>(fuse_row, i0)), "r"(qk_lo) : "memory");
          asm volatile("st.shared.u32 [%0], %1;" ::"r"(kb + swz<TR>(fuse_row, i0 + D / 2)), "r"(qk_hi) : "memory");
          asm volatile("st.shared.u32 [%0], %1;" ::"r"(kb + TB + swz<TR>(fuse_row, i0)), "r"(qv_lo) : "memory");
          asm volatile("st.shared.u32 [%0], %1;" ::"r"(kb + TB + swz<TR>(fuse_row, i0 + D / 2)), "r"(qv_hi) : "memory");
        } else {
          asm volatile("st.shared.u16 [%0], %1;" ::"r"(kb + swz<TR>(fuse_row, i0)), "h"((unsigned short)qk_lo) : "memory");
          asm volatile("st.shared.u16 [%0], %1;" ::"r"(kb + swz<TR>(fuse_row, i0 + D / 2)), "h"((unsigned short)qk_hi) : "memory");
          asm volatile("st.shared.u16 [%0], %1;" ::"r"(kb + TB + swz<TR>(fuse_row, i0)), "h"((unsigned short)qv_lo) : "memory");
          asm volatile("st.shared.u16 [%0], %1;" ::"r"(kb + TB + swz<TR>(fuse_row, i0 + D / 2)), "h"((unsigned short)qv_hi) : "memory");
        }
        __syncwarp();
      }
      if (FUSE && li == fuse_li) {
        // the new row of this tile comes from the step's k/v, not the copy
#pragma unroll
        for (int x = 0; x < HPL / 2; ++x) {
          const int d = lane * HPL + 2 * x;
          asm volatile("st.shared.u32 [%0], %1;" ::"r"(kb + swz<TR>(fuse_row, d)), "r"(kn[x]) : "memory");
          asm volatile("st.shared.u32 [%0], %1;" ::"r"(kb + TB + swz<TR>(fuse_row, d)), "r"(vn[x]) : "memory");
        }
        __syncwarp();
      }
      consume_tile<D, TR, false, VLLM>(kb, kb + TB, j * TR, tok_end, qf, p.scale_log2, st, lane);
    }
    __syncwarp();
    if (lane == 0 && li + P < my_tiles) {
      fence_proxy_async_smem();
      issue(li + P);
    }
  }

  if (failed) {
    // Let the copies this warp still has in flight land before the CTA may
    // exit (bounded as well), then report.
    if (lane == 0) atomicOr(&g_device_status, kDevWaitTimeout);
    const int last = min(li + P, my_tiles);
    for (int lj = li; lj < last; ++lj)
      (void)mbar_wait_bounded(my_bars + 8 * (lj % P), (lj / P) & 1, kWaitLimitNs);
    if (lane == 0) atomicOr(&s_failed, 1);
  }

  st.finish_sums();
  __syncthreads();  // every warp is done with its ring
  if (s_failed) return;

  // merge the W warp states through shared memory (reusing the ring)
  float* red = reinterpret_cast<float*>(smem);
  st.store(red + warp * Shape::kRedFloats, lane, 8);
  __syncthreads();

  const int G = p.group;
  const size_t qh0 = (size_t)s * p.num_heads + (size_t)g * G;
  if (SPLIT && n_pieces > 1) {  // this chunk's partials, for the combine
    for (int idx = threadIdx.x; idx < G * D; idx += W * 32) {
      const int h = idx / D;
      const int d = idx - h * D;
      float M, num, den;
      merge_warps<W, D>(red, Shape::kRedFloats, h, d, M, num, den);
      const size_t slot = (qh0 + h) * p.num_splits + piece;
      p.part_out[slot * D + d] = num;
      if (d == 0) {
        p.part_m[slot] = M;
        p.part_l[slot] = den;
      }
    }
  } else {  // the whole context: the f16 output
    for (int idx = threadIdx.x; idx < G * D; idx += W * 32) {
      const int h = idx / D;
      const int d = idx - h * D;
      float M, num, den;
      merge_warps<W, D>(red, Shape::kRedFloats, h, d, M, num, den);
      p.out[(qh0 + h) * D + d] = __float2half_rn(den > 0.f ? num / den : 0.f);
    }
  }
}

// ---------------------------------------------------------------------------
// multi-token queries (varlen, causal)
// ---------------------------------------------------------------------------
//
// One CTA per (sequence, KV head, chunk of QC queries), QC = max(1, 8 NT / G):
// the 8 NT columns of the mma n-tiles are the (query, head) pairs of the
// chunk, column n = (query n / G, head n % G).  Query t of sequence s sits
// at position pos_offsets[s] + t and sees positions up to and including it:
// each column masks with its own limit.  The chunk reads the context up to
// its last query's position, once for all its columns.  VLLM: the pools are
// in the vLLM layout (p.k_pool is the K pool; kmap is unused).

struct VarlenParams {
  const __half* q;              // [total_q][H][D]
  const int32_t* cu_seqlens_q;  // [B + 1]
  const int32_t* pos_offsets;   // [B]
  const int32_t* block_tables;  // [B][MBPS]
  __half* out;                  // [total_q][H][D]
  int total_q;
  int num_heads;
  int num_kv_heads;
  int group;
  int qc;          // queries per CTA
  int num_chunks;  // chunks per (sequence, KV head) in the grid
  int num_seqs;
  int fair_depth;  // the grid is resident at once: scale in-flight depth
  const __half* k_pool;  // the K pool (vLLM layout: tiles are bulk-copied from it)
  // split-K (SPLIT kernels): f32 partials per (query token, head, split);
  // each split takes chunk = max(min_chunk_blocks, ceil(n / S)) blocks of
  // context, n the most blocks any chunk of queries reads in the call (cut
  // on the device, as the decode kernel cuts its chunks)
  float* part_out;  // [total_q][H][S][D]
  float* part_m;    // [total_q][H][S]  base-2 running max
  float* part_l;    // [total_q][H][S]  running sum
  int num_splits;
  int min_chunk_blocks;
  int max_blocks_per_seq;
  int num_blocks;
  float scale_log2;
};

template <int D, int BS, int W, int P, int NT, bool VLLM, bool SPLIT>
__global__ void __launch_bounds__(W * 32)
paged_varlen_kernel(const __grid_constant__ CUtensorMap kmap,
                    const __grid_constant__ CUtensorMap vmap, const VarlenParams p) {
  // staging tiles as in the decode kernel: 16-row sub-tiles of blocked pools
  constexpr int TR = (VLLM || !kSubtile) ? BS : 16;
  constexpr int SUB = BS / TR;
  using Shape = DecodeShape<D, TR, W, P>;
  static_assert(W * NT * Shape::kRedFloats * 4 <= Shape::kRingBytes,
                "the merge area reuses the ring");
  constexpr int KS = Shape::kKS;
  constexpr int TB = Shape::kTileBytes;

  extern __shared__ uint8_t smem_raw[];
  __shared__ int s_failed;
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t ring = smem_addr(smem);
  const uint32_t bars = ring + Shape::kRingBytes;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int r = lane >> 2, c = lane & 3;

  int item = blockIdx.x;
  const int split = SPLIT ? item % p.num_splits : 0;
  if (SPLIT) item /= p.num_splits;
  const int qc_idx = item % p.num_chunks;
  item /= p.num_chunks;
  const int g = item % p.num_kv_heads;
  const int s = item / p.num_kv_heads;
  const int G = p.group;

  pdl_launch_dependents();
  if (threadIdx.x == 0) s_failed = 0;
  const uint32_t my_bars = bars + warp * P * 8;
  if (lane == 0) {
#pragma unroll
    for (int i = 0; i < P; ++i) mbar_init(my_bars + 8 * i, 1);
    fence_mbar_init();
  }
  pdl_wait();

  const unsigned int status = *reinterpret_cast<volatile unsigned int*>(&g_device_status);
  const int cap = p.max_blocks_per_seq * BS;
  const int q_begin = __ldg(p.cu_seqlens_q + s);
  const int q_end = __ldg(p.cu_seqlens_q + s + 1);
  int pos0 = __ldg(p.pos_offsets + s);
  // the longest context any chunk of the call reads, in tiles (sets the
  // split chunks and, as in the decode kernel, the fair share)
  __shared__ int s_max[W];
  const bool need_max = SPLIT || p.fair_depth;
  if (need_max) {
    int mx = 0;
    for (int i = threadIdx.x; i < p.num_seqs; i += W * 32) {
      int last = __ldg(p.pos_offsets + i) + __ldg(p.cu_seqlens_q + i + 1) -
                 __ldg(p.cu_seqlens_q + i);
      last = last < 0 ? 0 : (last > cap ? cap : last);
      mx = max(mx, (last + BS - 1) / BS);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if (lane == 0) s_max[warp] = mx;
  }
  if (__syncthreads_or(status & kDevWaitTimeout)) return;  // also publishes s_max
  int nblk_max = 0;
  if (need_max) {
#pragma unroll
    for (int w = 0; w < W; ++w) nblk_max = max(nblk_max, s_max[w]);
  }
  const int chunk = SPLIT ? max(p.min_chunk_blocks, (nblk_max + p.num_splits - 1) / p.num_splits)
                          : p.max_blocks_per_seq;

  // bad query ranges or positions are flagged and skipped / clamped
  if (q_begin < 0 || q_end < q_begin || q_end > p.total_q) {
    if (threadIdx.x == 0) atomicOr(&g_device_status, kDevBadContextLen);
    return;
  }
  const int q_len = q_end - q_begin;
  if (qc_idx == p.num_chunks - 1 && q_len > p.num_chunks * p.qc && threadIdx.x == 0)
    atomicOr(&g_device_status, kDevBadContextLen);  // more queries than the grid covers
  const int t0 = qc_idx * p.qc;
  if (t0 >= q_len) return;
  const int nq = min(p.qc, q_len - t0);
  if (pos0 < 0 || pos0 + q_len > cap) {
    if (threadIdx.x == 0) atomicOr(&g_device_status, kDevBadContextLen);
    pos0 = pos0 < 0 ? 0 : max(0, cap - q_len);
  }
  // positions this chunk of queries reads; with SPLIT, this CTA's slice of
  // them (a split starting at or past the end is never written nor read)
  const int chunk_end = min(cap, pos0 + t0 + nq);
  const int ncols = nq * G;  // (query, head) columns of this chunk
  int tok_begin = 0;
  int tok_end = chunk_end;
  if (SPLIT) {
    if ((long long)split * chunk * BS >= chunk_end) {
      // Empty split: max -inf and sum 0 for every column, so the combine can
      // read every split (it gives these weight 0).
      for (int n = threadIdx.x; n < ncols; n += W * 32) {
        const size_t row = (size_t)(q_begin + t0 + n / G) * p.num_heads + (size_t)g * G + n % G;
        p.part_m[row * p.num_splits + split] = -CUDART_INF_F;
        p.part_l[row * p.num_splits + split] = 0.f;
      }
      return;
    }
    tok_begin = split * chunk * BS;
    tok_end = (int)min((long long)chunk_end, (long long)tok_begin + (long long)chunk * BS);
  }
  const int sub_begin = tok_begin / TR;  // the CTA's first tile
  const int n_tiles = (tok_end - tok_begin + TR - 1) / TR;
  const int32_t* table = p.block_tables + (size_t)s * p.max_blocks_per_seq;
  int WE = W;  // warps that take tiles (fewer for short chunks under the fair share)
  if (p.fair_depth) {
    const int mx = (SPLIT ? min(nblk_max, chunk) : nblk_max) * SUB;
    if (mx > 0) WE = max(1, min(W, (W * n_tiles + mx - 1) / mx));
  }
  const int my_tiles = (warp < WE && n_tiles > warp) ? (n_tiles - warp + WE - 1) / WE : 0;

  auto k_stage = [&](int stage) { return ring + (warp * P + stage) * Shape::kStageBytes; };
  auto issue = [&](int li) {
    const int stage = li % P;
    const int j = sub_begin + warp + li * WE;
    const int phys = __ldg(table + j / SUB);
    const uint32_t bar = my_bars + 8 * stage;
    if (phys >= 0 && phys < p.num_blocks) {
      issue_tile_copy<D, TR, VLLM>(k_stage(stage), bar, phys * p.num_kv_heads + g, (j % SUB) * TR,
                                   &kmap, &vmap, p.k_pool);
    } else {
      atomicOr(&g_device_status, kDevBadBlockId);
      mbar_arrive(bar);
    }
  };
  if (lane == 0) {
    const int n0 = my_tiles < P ? my_tiles : P;
    for (int li = 0; li < n0; ++li) issue(li);
  }

  // column n = (query t0 + n / G, head n % G) while n < nq * G; n-tile nt
  // holds columns 8 nt .. 8 nt + 7 (this lane's B fragment: column 8 nt + r)
  uint32_t qf[NT][KS][2];
  int lim[NT][2];
  WarpState<D> st[NT];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int n = nt * 8 + r;
    const bool live = n < ncols;
    const size_t row = (size_t)(q_begin + t0 + (live ? n / G : 0)) * p.num_heads +
                       (size_t)g * G + (live ? n % G : 0);
    const uint32_t* qrow = reinterpret_cast<const uint32_t*>(p.q + row * D);
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      qf[nt][ks][0] = live ? __ldg(qrow + ks * 8 + c) : 0u;
      qf[nt][ks][1] = live ? __ldg(qrow + ks * 8 + 4 + c) : 0u;
    }
    // this lane's columns 8 nt + 2c and 8 nt + 2c + 1: their causal limits
    const int n0 = nt * 8 + 2 * c;
    lim[nt][0] = (n0 < ncols) ? pos0 + t0 + n0 / G + 1 : tok_end;
    lim[nt][1] = (n0 + 1 < ncols) ? pos0 + t0 + (n0 + 1) / G + 1 : tok_end;
    st[nt].reset();
  }
  bool failed = false;
  int li = 0;
  for (; li < my_tiles; ++li) {
    const int stage = li % P;
    if (!mbar_wait_bounded(my_bars + 8 * stage, (li / P) & 1, kWaitLimitNs)) {
      failed = true;
      break;
    }
    const int j = sub_begin + warp + li * WE;
    const int phys = __ldg(table + j / SUB);
    if (phys >= 0 && phys < p.num_blocks) {
      const uint32_t kb = k_stage(stage);
      consume_tiles<D, TR, NT, true, VLLM>(kb, kb + TB, j * TR, tok_end, qf, p.scale_log2, st,
                                           lane, lim);
    }
    __syncwarp();
    if (lane == 0 && li + P < my_tiles) {
      fence_proxy_async_smem();
      issue(li + P);
    }
  }
  if (failed) {
    if (lane == 0) atomicOr(&g_device_status, kDevWaitTimeout);
    const int last = min(li + P, my_tiles);
    for (int lj = li; lj < last; ++lj)
      (void)mbar_wait_bounded(my_bars + 8 * (lj % P), (lj / P) & 1, kWaitLimitNs);
    if (lane == 0) atomicOr(&s_failed, 1);
  }

#pragma unroll
  for (int nt = 0; nt < NT; ++nt) st[nt].finish_sums();
  __syncthreads();  // every warp is done with its ring
  if (s_failed) return;
  float* red = reinterpret_cast<float*>(smem);
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) st[nt].store(red + (warp * NT + nt) * Shape::kRedFloats, lane, 8);
  __syncthreads();
  for (int idx = threadIdx.x; idx < ncols * D; idx += W * 32) {
    const int n = idx / D;
    const int d = idx - n * D;
    float M, num, den;
    merge_warps<W, D>(red + (n / 8) * Shape::kRedFloats, NT * Shape::kRedFloats, n % 8, d, M,
                      num, den);
    const size_t row = (size_t)(q_begin + t0 + n / G) * p.num_heads + (size_t)g * G + n % G;
    if (SPLIT) {
      const size_t slot = row * p.num_splits + split;
      p.part_out[slot * D + d] = num;
      if (d == 0) {
        p.part_m[slot] = M;
        p.part_l[slot] = den;
      }
    } else {
      p.out[row * D + d] = __float2half_rn(den > 0.f ? num / den : 0.f);
    }
  }
}

// ---------------------------------------------------------------------------
// split-K combine
// ---------------------------------------------------------------------------

struct CombineParams {
  const float* part_out;
  const float* part_m;
  const float* part_l;
  const int32_t* context_lens;
  const int* split_header;  // the chunk size (blocks) phase 1 used
  __half* out;
  int num_rows;  // num_seqs * num_heads
  int num_heads;
  int num_splits;
  int block_size;
  int cap_tokens;  // max_blocks_per_seq * block_size
};

// Rows (output head vectors) merged per combine CTA: one warp each.
constexpr int kCombineWarps = 4;
// Split maxima and sums a lane holds (k = lane + 32 i); with
// PKV_MAX_SPLITS = 128 every split of a row is loaded in one round.
constexpr int kCombineSlots = (PKV_MAX_SPLITS + 31) / 32;
// Partial outputs a lane loads per round (each D/32 floats).
constexpr int kCombineBatch = 16;

// Lane `lane` loads the maxima and sums of splits lane, lane + 32, ... below
// num_splits (independent loads, issued together).
__device__ __forceinline__ void load_split_stats(const float* pm, const float* pl, int num_splits,
                                                 int lane, float (&mk)[kCombineSlots],
                                                 float (&lk)[kCombineSlots]) {
#pragma unroll
  for (int i = 0; i < kCombineSlots; ++i) {
    const int k = lane + 32 * i;
    mk[i] = k < num_splits ? __ldg(pm + k) : -CUDART_INF_F;
    lk[i] = k < num_splits ? __ldg(pl + k) : 0.f;
  }
}

// The log-sum-exp merge of one output row of D elements from its first n
// split partials, by one warp, given the split maxima and sums the lanes
// loaded (load_split_stats): M = max m_k, w_k = 2^(m_k - M) (0 for a split
// with max -inf, which holds no position of the row), den = sum w_k l_k;
// then each lane sums its D/32 elements of the weighted partial outputs with
// up to kCombineBatch independent vector loads in flight.  Splits at or past
// n are never read; a zero-weight split's partial is read but not used (it
// may never have been written).
template <int D>
__device__ __forceinline__ void merge_row_warp(const float (&mk)[kCombineSlots],
                                               const float (&lk)[kCombineSlots], const float* po,
                                               int n, __half* out_row, float* s_w) {
  constexpr int E = D / 32;  // elements per lane
  const int lane = threadIdx.x & 31;
  float M = -CUDART_INF_F;
#pragma unroll
  for (int i = 0; i < kCombineSlots; ++i)
    if (lane + 32 * i < n) M = fmaxf(M, mk[i]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  float den = 0.f;
#pragma unroll
  for (int i = 0; i < kCombineSlots; ++i) {
    const int k = lane + 32 * i;
    if (k < n) {
      const float w = (mk[i] == -CUDART_INF_F) ? 0.f : exp2f(mk[i] - M);
      s_w[k] = w;
      if (w != 0.f) den += w * lk[i];
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
  __syncwarp();
  float acc[E];
#pragma unroll
  for (int e = 0; e < E; ++e) acc[e] = 0.f;
  const float* base = po + lane * E;
  for (int kk = 0; kk < n; kk += kCombineBatch) {
    const int m = min(kCombineBatch, n - kk);
    float v[kCombineBatch][E];
#pragma unroll
    for (int x = 0; x < kCombineBatch; ++x) {
      if (x < m) {  // in bounds: loaded whatever the weight
        const float* src = base + (size_t)(kk + x) * D;
        if constexpr (E == 4) {
          const float4 t = __ldg(reinterpret_cast<const float4*>(src));
          v[x][0] = t.x;
          v[x][1] = t.y;
          v[x][2] = t.z;
          v[x][3] = t.w;
        } else {
          const float2 t = __ldg(reinterpret_cast<const float2*>(src));
          v[x][0] = t.x;
          v[x][1] = t.y;
        }
      }
    }
#pragma unroll
    for (int x = 0; x < kCombineBatch; ++x) {
      const float w = x < m ? s_w[kk + x] : 0.f;
      if (w != 0.f) {  // (a varlen split with no position of the row wrote no partial)
#pragma unroll
        for (int e = 0; e < E; ++e) acc[e] += w * v[x][e];
      }
    }
  }
  const float inv = den > 0.f ? 1.f / den : 0.f;
  __half2 h[E / 2];
#pragma unroll
  for (int e = 0; e < E / 2; ++e)
    h[e] = __floats2half2_rn(den > 0.f ? acc[2 * e] * inv : 0.f,
                             den > 0.f ? acc[2 * e + 1] * inv : 0.f);
  if constexpr (E == 4)
    *reinterpret_cast<uint2*>(out_row + lane * E) = make_uint2(pack_half2(h[0]), pack_half2(h[1]));
  else
    *reinterpret_cast<uint32_t*>(out_row + lane * E) = pack_half2(h[0]);
}

// Decode split-K: one warp per (sequence, query head) row.  The row's chunk
// count n follows from its length and the chunk size phase 1 used: n = 1 was
// finished by phase 1 (f16 output written), n = 0 (empty context) is zeros,
// n > 1 merges the n partials phase 1 wrote.  The chunk size, the length and
// every split's maximum and sum are loaded in one round (the maxima and sums
// past n are read but never used), the partials in the next.
template <int D>
__global__ void __launch_bounds__(kCombineWarps * 32) splitk_combine_kernel(const CombineParams p) {
  __shared__ float s_w[kCombineWarps][PKV_MAX_SPLITS];
  pdl_launch_dependents();
  pdl_wait();
  // after a lost copy has been flagged, decode calls write nothing (the
  // partials were not written either); uniform for the CTA
  if (*reinterpret_cast<volatile unsigned int*>(&g_device_status) & kDevWaitTimeout) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row = blockIdx.x * kCombineWarps + warp;
  if (row >= p.num_rows) return;
  const int s = row / p.num_heads;
  const int chunk_raw = *reinterpret_cast<const volatile int*>(p.split_header);
  int L = __ldg(p.context_lens + s);
  float mk[kCombineSlots], lk[kCombineSlots];
  load_split_stats(p.part_m + (size_t)row * p.num_splits, p.part_l + (size_t)row * p.num_splits,
                   p.num_splits, lane, mk, lk);
  const int chunk = max(1, chunk_raw);
  L = L < 0 ? 0 : (L > p.cap_tokens ? p.cap_tokens : L);
  const int nb = (L + p.block_size - 1) / p.block_size;
  const int n = min(p.num_splits, (nb + chunk - 1) / chunk);
  __half* out_row = p.out + (size_t)row * D;
  if (n == 1) return;
  if (n == 0) {
    constexpr int E = D / 32;
#pragma unroll
    for (int e = 0; e < E; ++e) out_row[lane * E + e] = __float2half_rn(0.f);
    return;
  }
  merge_row_warp<D>(mk, lk, p.part_out + (size_t)row * p.num_splits * D, n, out_row, s_w[warp]);
}

// Varlen split-K: one warp per (query token, head) row.  The token's
// sequence is found by binary search in cu_seqlens_q; phase 1 wrote every
// split of every query it covered (max -inf and sum 0 where the split holds
// none of the query's positions).  Rows phase 1 skipped (bad query ranges,
// queries past the grid; both flagged there) are written as zeros.
struct VarlenCombineParams {
  const float* part_out;
  const float* part_m;
  const float* part_l;
  const int32_t* cu_seqlens_q;
  __half* out;
  int num_seqs;
  int total_q;
  int num_heads;
  int num_splits;
  int covered_q;  // queries per sequence the phase-1 grid covers
};

template <int D>
__global__ void __launch_bounds__(kCombineWarps * 32)
varlen_combine_kernel(const VarlenCombineParams p) {
  __shared__ float s_w[kCombineWarps][PKV_MAX_SPLITS];
  pdl_launch_dependents();
  pdl_wait();
  if (*reinterpret_cast<volatile unsigned int*>(&g_device_status) & kDevWaitTimeout) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rh = blockIdx.x * kCombineWarps + warp;  // row * H + head
  if (rh >= p.total_q * p.num_heads) return;
  const int row = rh / p.num_heads;
  float mk[kCombineSlots], lk[kCombineSlots];  // in flight during the search
  load_split_stats(p.part_m + (size_t)rh * p.num_splits, p.part_l + (size_t)rh * p.num_splits,
                   p.num_splits, lane, mk, lk);
  int lo = 0, hi = p.num_seqs - 1;  // last sequence whose first row is <= row
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(p.cu_seqlens_q + mid) <= row)
      lo = mid;
    else
      hi = mid - 1;
  }
  const int q_begin = __ldg(p.cu_seqlens_q + lo);
  const int q_end = __ldg(p.cu_seqlens_q + lo + 1);
  const int t = row - q_begin;
  __half* out_row = p.out + (size_t)rh * D;
  if (q_begin < 0 || q_end < q_begin || q_end > p.total_q || t < 0 || t >= q_end - q_begin ||
      t >= p.covered_q) {
    constexpr int E = D / 32;
#pragma unroll
    for (int e = 0; e < E; ++e) out_row[lane * E + e] = __float2half_rn(0.f);
    return;
  }
  merge_row_warp<D>(mk, lk, p.part_out + (size_t)rh * p.num_splits * D, p.num_splits, out_row,
                    s_w[warp]);
}

// Diagnostic: one warp waits on an mbarrier that nothing arrives on.  The
// bounded wait gives up after kWaitLimitNs and the kernel flags
// kDevWaitTimeout, as a decode kernel does when a tile copy is lost; no copy,
// no global access but the flag.
__global__ void __launch_bounds__(32) wait_timeout_probe_kernel() {
  __shared__ __align__(8) uint64_t bar;
  const uint32_t b = smem_addr(&bar);
  if (threadIdx.x == 0) {
    mbar_init(b, 1);
    fence_mbar_init();
  }
  __syncwarp();
  const bool landed = mbar_wait_bounded(b, 0, kWaitLimitNs);
  if (!__any_sync(0xffffffffu, !landed)) return;
  if (threadIdx.x == 0) atomicOr(&g_device_status, kDevWaitTimeout);
}

}  // namespace pkv
