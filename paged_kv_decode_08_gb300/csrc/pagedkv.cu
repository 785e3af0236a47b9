// libpagedkv: the C-ABI entry points declared in include/pagedkv.h.
//
// Host side of every call: validate the arguments (before any CUDA call),
// build the TMA tensor maps of the two cache pools, pick the kernel
// instantiation for (head_dim, block_size) and launch on the caller's stream.
// Nothing here allocates device memory or reads device memory on the host
// (pkv_read_device_status excepted).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <utility>

#include "kernels.cuh"
#include "pagedkv.h"
#include "prefill_tc.cuh"
#include "varlen_tc.cuh"

// Warps per decode CTA and the shared-memory ring they split (KB); the
// defaults (6 warps, 96 KB: two resident CTAs per SM) won a sweep of warps x
// ring x CTAs per SM on all five workloads.  Overridable at build time.
#ifndef PKV_DECODE_WARPS
#define PKV_DECODE_WARPS 6
#endif
#ifndef PKV_DECODE_RING_KB
#define PKV_DECODE_RING_KB 96
#endif
#ifndef PKV_CTAS_PER_SM
#define PKV_CTAS_PER_SM 2
#endif
// The initial setting of pkv_set_varlen_tensor_path: varlen attention with
// more than 8 (query, head) columns per CTA on the tcgen05 kernel (blocked
// pools, head_dim 128) when 1, on the mma.sync kernel when 0.
#ifndef PKV_VARLEN_TC
#define PKV_VARLEN_TC 0
#endif
// Varlen attention (blocked pools, head_dim 128, no split) on the tcgen05
// prefill kernel once a sequence brings at least 128 (query, head) rows.
#ifndef PKV_PREFILL_TC
#define PKV_PREFILL_TC 1
#endif



namespace pkv {
namespace {

// Resident decode CTAs per SM the kernels are sized for.
constexpr int kCtasPerSm = PKV_CTAS_PER_SM;
// With the base grid already filling the GPU, a CTA keeps at most this many
// tokens, so one long context does not leave a long serial tail.
constexpr int kSaturatedChunkTokens = 2048;
// Below this a split's fixed costs outweigh its work.
constexpr int kMinSplitTokens = 256;
constexpr int kMaxAutoSplits = 64;
// The heuristic's smallest split of a chunked-prefill call (four 128-token
// spans: below that a split's fixed cost outweighs what it spreads).
constexpr int kMinPrefillSplitTokens = 512;

thread_local char t_last_error[512] = "";

pkv_status fail(pkv_status st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(t_last_error, sizeof(t_last_error), fmt, ap);
  va_end(ap);
  return st;
}

pkv_status cuda_fail(cudaError_t e, const char* what) {
  return fail(PKV_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Launches with programmatic stream serialization: the kernel's CTAs may
// start while the previous kernel in the stream finishes; every kernel here
// waits for it (griddepcontrol.wait) before touching global memory.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, int block, size_t smem,
                       cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3((unsigned)block, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

int current_device_sms(int* sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  static std::atomic<int> cache[64];
  if (dev >= 0 && dev < 64) {
    const int v = cache[dev].load(std::memory_order_relaxed);
    if (v > 0) {
      *sms = v;
      return 0;
    }
  }
  int v = 0;
  if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0)
    return -1;
  if (dev >= 0 && dev < 64) cache[dev].store(v, std::memory_order_relaxed);
  *sms = v;
  return 0;
}

// The pool as a 4-D tensor {64 elements, block_size rows, head_dim/64
// halves, num_blocks*num_kv_heads tiles} (innermost first; the row stride,
// head_dim * 2 bytes, is larger than the half stride, 128 bytes).  A box is
// 16 rows of one tile, 64 x 16 x head_dim/64 x 1 (the whole tile at block
// size 16, either half at 32, chosen by the row coordinate), landing as
// head_dim/64 runs of 16 128-byte lines with the 128-byte swizzle (one
// request per 16 rows measured slightly faster than one per 64-element half).
pkv_status encode_cache_map(CUtensorMap* map, const void* base, int num_blocks, int num_kv_heads,
                            int block_size, int head_dim, bool half_box = false) {
  auto encode = tensor_map_encoder();
  if (!encode) return fail(PKV_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  const cuuint64_t dims[4] = {64, (cuuint64_t)block_size, (cuuint64_t)(head_dim / 64),
                              (cuuint64_t)num_blocks * (cuuint64_t)num_kv_heads};
  const cuuint64_t strides[3] = {(cuuint64_t)head_dim * 2, 128,
                                 (cuuint64_t)block_size * head_dim * 2};
  const cuuint32_t box[4] = {64, (kSubtile || half_box) ? 16u : (cuuint32_t)block_size,
                             half_box ? 1u : (cuuint32_t)(head_dim / 64), 1};
  const cuuint32_t estride[4] = {1, 1, 1, 1};
  const CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4, const_cast<void*>(base), dims,
                            strides, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(PKV_ERR_CUDA, "cuTensorMapEncodeTiled failed (CUresult %d)", (int)r);
  return PKV_OK;
}

// The vLLM-layout V pool as a 3-D tensor {64 elements, head_dim*block_size/64
// lines, num_blocks*num_kv_heads tiles}: each V^T tile [head_dim][block_size]
// read as 128-byte lines.  A box is one whole tile, landing with the 128-byte
// swizzle.
pkv_status encode_vllm_v_map(CUtensorMap* map, const void* base, int num_blocks,
                             int num_kv_heads, int block_size, int head_dim) {
  auto encode = tensor_map_encoder();
  if (!encode) return fail(PKV_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  const int lines = head_dim * block_size / 64;
  const cuuint64_t dims[3] = {64, (cuuint64_t)lines,
                              (cuuint64_t)num_blocks * (cuuint64_t)num_kv_heads};
  const cuuint64_t strides[2] = {128, (cuuint64_t)block_size * head_dim * 2};
  const cuuint32_t box[3] = {64, (cuuint32_t)lines, 1};
  const cuuint32_t estride[3] = {1, 1, 1};
  const CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void*>(base), dims,
                            strides, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(PKV_ERR_CUDA, "cuTensorMapEncodeTiled failed (CUresult %d)", (int)r);
  return PKV_OK;
}

// Encoded tensor maps are kept per (pool address, shape, kind): a decode
// loop calls with the same pools every step, and a map depends on nothing
// else, so an entry never goes stale (a pool freed and another allocated at
// the same address with the same shape has the same map).  A small table,
// replaced round robin, shared by all threads under a mutex.
struct MapKey {
  const void* base;
  int num_blocks, num_kv_heads, block_size, head_dim, kind;
  bool operator==(const MapKey& o) const {
    return base == o.base && num_blocks == o.num_blocks && num_kv_heads == o.num_kv_heads &&
           block_size == o.block_size && head_dim == o.head_dim && kind == o.kind;
  }
};
constexpr int kMapCacheEntries = 32;
struct MapCache {
  std::mutex mu;
  MapKey key[kMapCacheEntries] = {};
  CUtensorMap map[kMapCacheEntries];
  int used = 0, next = 0;
};
MapCache g_maps;

// kind 0: a blocked-layout pool (K or V), 16 rows x head_dim per box;
// kind 1: a vLLM-layout V pool; kind 2: a blocked-layout pool, 16 rows x one
// 64-element half per box.
pkv_status cached_map(CUtensorMap* map, int kind, const void* base, int num_blocks,
                      int num_kv_heads, int block_size, int head_dim) {
  const MapKey k{base, num_blocks, num_kv_heads, block_size, head_dim, kind};
  {
    std::lock_guard<std::mutex> lock(g_maps.mu);
    for (int i = 0; i < g_maps.used; ++i)
      if (g_maps.key[i] == k) {
        *map = g_maps.map[i];
        return PKV_OK;
      }
  }
  const pkv_status st =
      kind == 1 ? encode_vllm_v_map(map, base, num_blocks, num_kv_heads, block_size, head_dim)
                : encode_cache_map(map, base, num_blocks, num_kv_heads, block_size, head_dim,
                                   kind == 2);
  if (st != PKV_OK) return st;
  std::lock_guard<std::mutex> lock(g_maps.mu);
  const int i = g_maps.used < kMapCacheEntries ? g_maps.used++ : g_maps.next;
  if (g_maps.used == kMapCacheEntries) g_maps.next = (i + 1) % kMapCacheEntries;
  g_maps.key[i] = k;
  g_maps.map[i] = *map;
  return PKV_OK;
}

pkv_status make_cache_map(CUtensorMap* map, const void* base, int num_blocks, int num_kv_heads,
                          int block_size, int head_dim) {
  return cached_map(map, 0, base, num_blocks, num_kv_heads, block_size, head_dim);
}

pkv_status make_vllm_v_map(CUtensorMap* map, const void* base, int num_blocks, int num_kv_heads,
                           int block_size, int head_dim) {
  return cached_map(map, 1, base, num_blocks, num_kv_heads, block_size, head_dim);
}

pkv_status make_half_box_map(CUtensorMap* map, const void* base, int num_blocks, int num_kv_heads,
                             int block_size, int head_dim) {
  return cached_map(map, 2, base, num_blocks, num_kv_heads, block_size, head_dim);
}

struct DecodeArgs {
  const void* q;
  const void* k_cache;
  const void* v_cache;
  const int32_t* block_tables;
  const int32_t* context_lens;
  int num_seqs, max_blocks_per_seq, num_blocks;
  float scale;
  int num_heads, num_kv_heads, head_dim, block_size;
  void* out;
  bool vllm = false;  // pools in the vLLM layout
};

pkv_status validate_decode(const DecodeArgs& a) {
  if (a.num_seqs < 0) return fail(PKV_ERR_INVALID_ARG, "num_seqs < 0");
  if (!a.q || !a.k_cache || !a.v_cache || !a.block_tables || !a.context_lens || !a.out)
    return fail(PKV_ERR_INVALID_ARG, "a required pointer is NULL");
  if (a.num_heads <= 0 || a.num_kv_heads <= 0 || a.num_heads % a.num_kv_heads != 0)
    return fail(PKV_ERR_INVALID_ARG, "num_heads (%d) must be a positive multiple of num_kv_heads (%d)",
                a.num_heads, a.num_kv_heads);
  if (a.max_blocks_per_seq <= 0 || a.num_blocks <= 0 || a.head_dim <= 0 || a.block_size <= 0)
    return fail(PKV_ERR_INVALID_ARG, "sizes must be positive");
  if (!std::isfinite(a.scale)) return fail(PKV_ERR_INVALID_ARG, "scale is not finite");
  if (a.head_dim != 64 && a.head_dim != 128)
    return fail(PKV_ERR_UNSUPPORTED, "head_dim %d (built: 64, 128)", a.head_dim);
  if (a.block_size != 16 && a.block_size != 32)
    return fail(PKV_ERR_UNSUPPORTED, "block_size %d (built: 16, 32)", a.block_size);
  if (a.num_heads / a.num_kv_heads > 8)
    return fail(PKV_ERR_UNSUPPORTED, "group %d (built: 1..8)", a.num_heads / a.num_kv_heads);
  if ((long long)a.num_blocks * a.block_size >= (1ll << 31) ||
      (long long)a.num_blocks * a.num_kv_heads >= (1ll << 31))
    return fail(PKV_ERR_INVALID_ARG, "num_blocks too large for 32-bit slots");
  if ((long long)a.max_blocks_per_seq * a.block_size >= (1ll << 31))
    return fail(PKV_ERR_INVALID_ARG, "max_blocks_per_seq * block_size overflows");
  if ((long long)a.num_seqs * a.num_heads >= (1ll << 31))
    return fail(PKV_ERR_INVALID_ARG, "num_seqs * num_heads too large");
  if (!aligned(a.k_cache, 16) || !aligned(a.v_cache, 16))
    return fail(PKV_ERR_INVALID_ARG, "k_cache and v_cache must be 16-byte aligned");
  if (!aligned(a.q, 4) || !aligned(a.out, 4))
    return fail(PKV_ERR_INVALID_ARG, "q and out must be 4-byte aligned");
  if (!aligned(a.block_tables, 4) || !aligned(a.context_lens, 4))
    return fail(PKV_ERR_INVALID_ARG, "block_tables and context_lens must be 4-byte aligned");
  return PKV_OK;
}

// Warps and ring stages for staging tiles of TR rows (16 for blocked pools,
// the block size for vLLM-layout pools).
template <int D, int TR>
struct Tuning {
  static constexpr int W = PKV_DECODE_WARPS;
  static constexpr int kStage = 2 * TR * D * 2;
  static constexpr int P = (PKV_DECODE_RING_KB * 1024) / (W * kStage) > 0
                               ? (PKV_DECODE_RING_KB * 1024) / (W * kStage)
                               : 1;
};

template <int D, int BS, bool SPLIT, bool FUSE, bool VLLM, bool QKV = false>
pkv_status launch_decode(const DecodeArgs& a, const DecodeParams& prm, cudaStream_t stream,
                         int grid) {
  constexpr int TR = (VLLM || !kSubtile) ? BS : 16;
  constexpr int W = Tuning<D, TR>::W;
  constexpr int P = Tuning<D, TR>::P;
  using Shape = DecodeShape<D, TR, W, P>;
  auto kernel = paged_decode_kernel<D, BS, W, P, SPLIT, FUSE, VLLM, QKV>;

  static std::atomic<unsigned long long> attr_set{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  const unsigned long long bit = 1ull << (dev & 63);
  if (!(attr_set.load(std::memory_order_relaxed) & bit)) {
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, Shape::kSmemBytes);
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(decode)");
    attr_set.fetch_or(bit, std::memory_order_relaxed);
  }

  CUtensorMap kmap, vmap;
  pkv_status st;
  DecodeParams prm2 = prm;
  if (VLLM) {
    // K tiles are bulk-copied from the pool pointer; kmap only fills the slot
    st = make_vllm_v_map(&vmap, a.v_cache, a.num_blocks, a.num_kv_heads, BS, D);
    if (st != PKV_OK) return st;
    kmap = vmap;
    prm2.k_cache = static_cast<__half*>(const_cast<void*>(a.k_cache));
  } else {
    st = make_cache_map(&kmap, a.k_cache, a.num_blocks, a.num_kv_heads, BS, D);
    if (st != PKV_OK) return st;
    st = make_cache_map(&vmap, a.v_cache, a.num_blocks, a.num_kv_heads, BS, D);
    if (st != PKV_OK) return st;
  }

  // fair-share depth only pays when every CTA of the grid is resident at once
  int sms = 0;
  prm2.fair_depth = (current_device_sms(&sms) == 0 && grid <= sms * kCtasPerSm) ? 1 : 0;
  e = launch_pdl(kernel, grid, W * 32, Shape::kSmemBytes, stream, kmap, vmap, prm2);
  if (e != cudaSuccess) return cuda_fail(e, SPLIT ? "split-K phase 1 launch" : "decode launch");
  return PKV_OK;
}

template <bool SPLIT, bool FUSE, bool VLLM, bool QKV = false>
pkv_status dispatch_decode_f(const DecodeArgs& a, const DecodeParams& prm, cudaStream_t stream,
                             int grid) {
  if (a.head_dim == 128 && a.block_size == 16)
    return launch_decode<128, 16, SPLIT, FUSE, VLLM, QKV>(a, prm, stream, grid);
  if (a.head_dim == 128 && a.block_size == 32)
    return launch_decode<128, 32, SPLIT, FUSE, VLLM, QKV>(a, prm, stream, grid);
  if (a.head_dim == 64 && a.block_size == 16)
    return launch_decode<64, 16, SPLIT, FUSE, VLLM, QKV>(a, prm, stream, grid);
  if (a.head_dim == 64 && a.block_size == 32)
    return launch_decode<64, 32, SPLIT, FUSE, VLLM, QKV>(a, prm, stream, grid);
  return fail(PKV_ERR_UNSUPPORTED, "head_dim %d / block_size %d", a.head_dim, a.block_size);
}

// Kernels with the fused append, the fused QKV step or the vLLM layout only
// where a call asks for it, so plain decode kernels carry none of that code.
template <bool SPLIT>
pkv_status dispatch_decode(const DecodeArgs& a, const DecodeParams& prm, cudaStream_t stream,
                           int grid) {
  if (prm.qkv) return dispatch_decode_f<SPLIT, false, false, true>(a, prm, stream, grid);
  if (a.vllm) {
    if (prm.new_slots) return fail(PKV_ERR_UNSUPPORTED, "no fused append on the vLLM layout");
    return dispatch_decode_f<SPLIT, false, true>(a, prm, stream, grid);
  }
  return prm.new_slots ? dispatch_decode_f<SPLIT, true, false>(a, prm, stream, grid)
                       : dispatch_decode_f<SPLIT, false, false>(a, prm, stream, grid);
}

DecodeParams base_params(const DecodeArgs& a) {
  DecodeParams p{};
  p.q = static_cast<const __half*>(a.q);
  p.block_tables = a.block_tables;
  p.context_lens = a.context_lens;
  p.out = static_cast<__half*>(a.out);
  p.num_seqs = a.num_seqs;
  p.num_heads = a.num_heads;
  p.num_kv_heads = a.num_kv_heads;
  p.group = a.num_heads / a.num_kv_heads;
  p.max_blocks_per_seq = a.max_blocks_per_seq;
  p.num_blocks = a.num_blocks;
  p.num_splits = 1;
  p.min_chunk_blocks = 1;
  p.chunk_hint = a.max_blocks_per_seq;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  return p;
}

template <int D, int BS, int NT, bool VLLM, bool SPLIT>
pkv_status launch_varlen(const DecodeArgs& a, const VarlenParams& vp, cudaStream_t stream,
                         int grid) {
  constexpr int TR = (VLLM || !kSubtile) ? BS : 16;
  constexpr int W = Tuning<D, TR>::W;
  constexpr int P = Tuning<D, TR>::P;
  using Shape = DecodeShape<D, TR, W, P>;
  auto kernel = paged_varlen_kernel<D, BS, W, P, NT, VLLM, SPLIT>;
  static std::atomic<unsigned long long> attr_set{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  const unsigned long long bit = 1ull << (dev & 63);
  if (!(attr_set.load(std::memory_order_relaxed) & bit)) {
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, Shape::kSmemBytes);
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(varlen)");
    attr_set.fetch_or(bit, std::memory_order_relaxed);
  }
  CUtensorMap kmap, vmap;
  pkv_status st;
  VarlenParams vp2 = vp;
  if (VLLM) {
    // K tiles are bulk-copied from the pool pointer; kmap only fills the slot
    st = make_vllm_v_map(&vmap, a.v_cache, a.num_blocks, a.num_kv_heads, BS, D);
    if (st != PKV_OK) return st;
    kmap = vmap;
    vp2.k_pool = static_cast<const __half*>(a.k_cache);
  } else {
    st = make_cache_map(&kmap, a.k_cache, a.num_blocks, a.num_kv_heads, BS, D);
    if (st != PKV_OK) return st;
    st = make_cache_map(&vmap, a.v_cache, a.num_blocks, a.num_kv_heads, BS, D);
    if (st != PKV_OK) return st;
  }
  int sms = 0;
  vp2.fair_depth = (current_device_sms(&sms) == 0 && grid <= sms * kCtasPerSm) ? 1 : 0;
  e = launch_pdl(kernel, grid, W * 32, Shape::kSmemBytes, stream, kmap, vmap, vp2);
  if (e != cudaSuccess) return cuda_fail(e, "varlen attention launch");
  return PKV_OK;
}

template <int BS, bool SPLIT>
pkv_status launch_varlen_tc(const DecodeArgs& a, const VarlenParams& vp, cudaStream_t stream,
                            int grid) {
  using Sh = TcVarlenShape<128>;
  auto kernel = paged_varlen_tc_kernel<128, BS, SPLIT>;
  static std::atomic<unsigned long long> attr_set{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  const unsigned long long bit = 1ull << (dev & 63);
  if (!(attr_set.load(std::memory_order_relaxed) & bit)) {
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, Sh::kSmemBytes);
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(varlen tc)");
    attr_set.fetch_or(bit, std::memory_order_relaxed);
  }
  CUtensorMap kmap, vmap;
  pkv_status st = make_half_box_map(&kmap, a.k_cache, a.num_blocks, a.num_kv_heads, BS, 128);
  if (st != PKV_OK) return st;
  st = make_half_box_map(&vmap, a.v_cache, a.num_blocks, a.num_kv_heads, BS, 128);
  if (st != PKV_OK) return st;
  e = launch_pdl(kernel, grid, Sh::kThreads, Sh::kSmemBytes, stream, kmap, vmap, vp);
  if (e != cudaSuccess) return cuda_fail(e, "varlen attention (tcgen05) launch");
  return PKV_OK;
}

std::atomic<int> g_varlen_tc{PKV_VARLEN_TC};

template <int BS, bool SPLIT>
pkv_status launch_prefill_tc(const DecodeArgs& a, const VarlenParams& vp, cudaStream_t stream,
                             int grid) {
  using Sh = TcPrefillShape;
  auto kernel = paged_prefill_tc_kernel<BS, SPLIT>;
  static std::atomic<unsigned long long> attr_set{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  const unsigned long long bit = 1ull << (dev & 63);
  if (!(attr_set.load(std::memory_order_relaxed) & bit)) {
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, Sh::kSmemBytes);
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(prefill tc)");
    attr_set.fetch_or(bit, std::memory_order_relaxed);
  }
  CUtensorMap kmap, vmap;
  pkv_status st = make_half_box_map(&kmap, a.k_cache, a.num_blocks, a.num_kv_heads, BS, 128);
  if (st != PKV_OK) return st;
  st = make_half_box_map(&vmap, a.v_cache, a.num_blocks, a.num_kv_heads, BS, 128);
  if (st != PKV_OK) return st;
  e = launch_pdl(kernel, grid, Sh::kThreads, Sh::kSmemBytes, stream, kmap, vmap, vp);
  if (e != cudaSuccess) return cuda_fail(e, "varlen attention (tcgen05 prefill) launch");
  return PKV_OK;
}

template <bool SPLIT>
pkv_status dispatch_varlen(const DecodeArgs& a, const VarlenParams& vp, cudaStream_t cs, int grid,
                           int NT, bool vllm) {
  if (g_varlen_tc.load(std::memory_order_relaxed) && !vllm && NT == 2 && a.head_dim == 128)
    return a.block_size == 16 ? launch_varlen_tc<16, SPLIT>(a, vp, cs, grid)
                              : launch_varlen_tc<32, SPLIT>(a, vp, cs, grid);
#define PKV_VARLEN_CASE(D_, BS_)                                                              \
  if (a.head_dim == D_ && a.block_size == BS_) {                                              \
    if (NT == 2)                                                                              \
      return vllm ? launch_varlen<D_, BS_, 2, true, SPLIT>(a, vp, cs, grid)                   \
                  : launch_varlen<D_, BS_, 2, false, SPLIT>(a, vp, cs, grid);                 \
    return vllm ? launch_varlen<D_, BS_, 1, true, SPLIT>(a, vp, cs, grid)                     \
                : launch_varlen<D_, BS_, 1, false, SPLIT>(a, vp, cs, grid);                   \
  }
  PKV_VARLEN_CASE(128, 16)
  PKV_VARLEN_CASE(128, 32)
  PKV_VARLEN_CASE(64, 16)
  PKV_VARLEN_CASE(64, 32)
#undef PKV_VARLEN_CASE
  return fail(PKV_ERR_UNSUPPORTED, "head_dim %d / block_size %d", a.head_dim, a.block_size);
}

// The fused append of pkv_append_decode (slots set), or the fused QKV step
// of pkv_qkv_norm_rope_append_decode (qkv set); all null: neither.
struct FuseArgs {
  const void* k_new = nullptr;
  const void* v_new = nullptr;
  const int32_t* slots = nullptr;
  void* k_cache = nullptr;
  void* v_cache = nullptr;
  const void* qkv = nullptr;
  const void* q_norm_w = nullptr;
  const void* k_norm_w = nullptr;
  const float* cos_t = nullptr;
  const float* sin_t = nullptr;
  int max_pos = 0;
  float eps = 0.f;
};

void apply_fuse(DecodeParams& p, const FuseArgs* f) {
  if (!f) return;
  p.k_new = static_cast<const __half*>(f->k_new);
  p.v_new = static_cast<const __half*>(f->v_new);
  p.new_slots = f->slots;
  p.k_cache = static_cast<__half*>(f->k_cache);
  p.v_cache = static_cast<__half*>(f->v_cache);
  p.qkv = static_cast<const __half*>(f->qkv);
  p.q_norm_w = static_cast<const __half*>(f->q_norm_w);
  p.k_norm_w = static_cast<const __half*>(f->k_norm_w);
  p.cos_t = f->cos_t;
  p.sin_t = f->sin_t;
  p.max_pos = f->max_pos;
  p.eps = f->eps;
}

pkv_status single_pass(const DecodeArgs& a, cudaStream_t stream, const FuseArgs* fuse = nullptr) {
  const long long grid = (long long)a.num_seqs * a.num_kv_heads;
  if (grid >= (1ll << 31)) return fail(PKV_ERR_INVALID_ARG, "grid too large");
  DecodeParams prm = base_params(a);
  apply_fuse(prm, fuse);
  return dispatch_decode<false>(a, prm, stream, (int)grid);
}

// pkv_append and pkv_append_vllm_layout: the same checks and grid, a kernel
// per layout.
pkv_status append_impl(const void* k, const void* v, const int32_t* slot_mapping,
                       int num_tokens, void* k_cache, void* v_cache, int num_blocks,
                       int block_size, int num_kv_heads, int head_dim, cudaStream_t stream,
                       bool vllm) {
  if (num_tokens < 0) return fail(PKV_ERR_INVALID_ARG, "num_tokens < 0");
  if (!k || !v || !slot_mapping || !k_cache || !v_cache)
    return fail(PKV_ERR_INVALID_ARG, "a required pointer is NULL");
  if (num_blocks <= 0 || block_size <= 0 || num_kv_heads <= 0 || head_dim <= 0)
    return fail(PKV_ERR_INVALID_ARG, "sizes must be positive");
  if (head_dim != 64 && head_dim != 128)
    return fail(PKV_ERR_UNSUPPORTED, "head_dim %d (built: 64, 128)", head_dim);
  if (block_size != 16 && block_size != 32)
    return fail(PKV_ERR_UNSUPPORTED, "block_size %d (built: 16, 32)", block_size);
  if ((long long)num_blocks * block_size >= (1ll << 31))
    return fail(PKV_ERR_INVALID_ARG, "num_blocks too large for 32-bit slots");
  if (!aligned(k, 16) || !aligned(v, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16))
    return fail(PKV_ERR_INVALID_ARG, "k, v, k_cache and v_cache must be 16-byte aligned");
  if (!aligned(slot_mapping, 4)) return fail(PKV_ERR_INVALID_ARG, "slot_mapping must be 4-byte aligned");
  if (num_tokens == 0) return PKV_OK;

  const int chunks_per_row = head_dim / 8;
  const long long total = (long long)num_tokens * num_kv_heads * chunks_per_row;
  long long blocks = (total + 255) / 256;
  if (blocks > 65536) blocks = 65536;  // grid-stride beyond this
  const long long num_slots = (long long)num_blocks * block_size;
  const cudaError_t e =
      vllm ? launch_pdl(append_vllm_kernel, (int)blocks, 256, 0, stream,
                        static_cast<const uint4*>(k), static_cast<const uint4*>(v), slot_mapping,
                        total, chunks_per_row, num_kv_heads, block_size, num_slots,
                        static_cast<uint4*>(k_cache), static_cast<__half*>(v_cache))
           : launch_pdl(append_kernel, (int)blocks, 256, 0, stream, static_cast<const uint4*>(k),
                        static_cast<const uint4*>(v), slot_mapping, total, chunks_per_row,
                        num_kv_heads, block_size, num_slots, static_cast<uint4*>(k_cache),
                        static_cast<uint4*>(v_cache));
  if (e != cudaSuccess) return cuda_fail(e, "append launch");
  return PKV_OK;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Split-K scratch: a 256-byte header (the chunk size phase 1 used, for the
// combine), then f32 part_out [rows][D], part_m [rows], part_l [rows] with
// rows = (num_seqs or total_q) * num_heads * S, each 256-byte aligned.
constexpr size_t kScratchHeaderBytes = 256;

struct SplitScratch {
  int* header;
  float* part_out;
  float* part_m;
  float* part_l;
};

SplitScratch carve_scratch(void* scratch, size_t rows, int head_dim) {
  uint8_t* b = static_cast<uint8_t*>(scratch);
  SplitScratch sc;
  sc.header = reinterpret_cast<int*>(b);
  b += kScratchHeaderBytes;
  sc.part_out = reinterpret_cast<float*>(b);
  b += align256(rows * head_dim * sizeof(float));
  sc.part_m = reinterpret_cast<float*>(b);
  b += align256(rows * sizeof(float));
  sc.part_l = reinterpret_cast<float*>(b);
  return sc;
}

// The split-K combine for head_dim D (one warp per output row).
template <typename Params>
cudaError_t launch_combine(void (*k64)(Params), void (*k128)(Params), int head_dim,
                           long long rows, cudaStream_t cs, const Params& cp) {
  const long long grid = (rows + kCombineWarps - 1) / kCombineWarps;
  return launch_pdl(head_dim == 128 ? k128 : k64, (int)grid, kCombineWarps * 32, 0, cs, cp);
}

}  // namespace
}  // namespace pkv

using namespace pkv;

extern "C" {

const char* pkv_status_string(pkv_status status) {
  switch (status) {
    case PKV_OK: return "ok";
    case PKV_ERR_INVALID_ARG: return "invalid argument";
    case PKV_ERR_UNSUPPORTED: return "unsupported configuration";
    case PKV_ERR_SCRATCH_TOO_SMALL: return "split-K scratch missing or too small";
    case PKV_ERR_CUDA: return "CUDA error";
    default: return "unknown status";
  }
}

const char* pkv_last_error(void) { return t_last_error; }

size_t pkv_splitk_scratch_bytes(int32_t num_seqs, int32_t num_heads, int32_t head_dim,
                                int32_t num_splits) {
  if (num_seqs <= 0 || num_heads <= 0 || head_dim <= 0 || num_splits <= 1) return 0;
  const size_t rows = (size_t)num_seqs * num_heads * num_splits;
  return kScratchHeaderBytes + align256(rows * head_dim * sizeof(float)) +
         2 * align256(rows * sizeof(float));
}

int32_t pkv_pick_num_splits(int32_t num_seqs, int32_t num_kv_heads, int32_t max_context_len,
                            int32_t block_size, int32_t num_sms) {
  if (num_seqs <= 0 || num_kv_heads <= 0 || max_context_len <= 0 || block_size <= 0 ||
      num_sms <= 0)
    return 1;
  const long long base = (long long)num_seqs * num_kv_heads;
  const long long slots = (long long)num_sms * kCtasPerSm;
  long long s;
  if (base >= slots) {
    s = (max_context_len + kSaturatedChunkTokens - 1) / kSaturatedChunkTokens;
  } else {
    s = (2 * slots + base) / (2 * base);  // nearest to one wave of split CTAs
  }
  const long long by_len = max_context_len / kMinSplitTokens;
  const long long max_blocks = (max_context_len + block_size - 1) / block_size;
  if (s > by_len) s = by_len;
  if (s > max_blocks) s = max_blocks;
  if (s > kMaxAutoSplits) s = kMaxAutoSplits;
  if (s < 1) s = 1;
  return (int32_t)s;
}

int32_t pkv_set_varlen_tensor_path(int32_t on) {
  if (on != 0 && on != 1) return -1;
  return pkv::g_varlen_tc.exchange(on);
}

int32_t pkv_varlen_pick_num_splits(int32_t num_seqs, int32_t num_heads, int32_t num_kv_heads,
                                   int32_t max_q_len, int32_t max_blocks_per_seq,
                                   int32_t block_size, int32_t num_sms) {
  if (num_seqs <= 0 || num_heads <= 0 || num_kv_heads <= 0 || num_heads % num_kv_heads != 0 ||
      max_q_len <= 0 || max_blocks_per_seq <= 0 || block_size <= 0 || num_sms <= 0)
    return 1;
  const int G = num_heads / num_kv_heads;
  const int nt = (long long)max_q_len * G > 8 ? 2 : 1;
  const int qc = G >= 8 * nt ? 1 : 8 * nt / G;
  const long long grid = (long long)num_seqs * num_kv_heads * ((max_q_len + qc - 1) / qc);
  const long long slots = (long long)num_sms * kCtasPerSm;
  // below one wave, the split count that brings the grid nearest one wave
  long long s = grid >= slots ? 1 : (2 * slots + grid) / (2 * grid);
  const long long cap_tokens = (long long)max_blocks_per_seq * block_size;
  if (s > cap_tokens / kMinSplitTokens) s = cap_tokens / kMinSplitTokens;
  if (s > max_blocks_per_seq) s = max_blocks_per_seq;
  if (s > kMaxAutoSplits) s = kMaxAutoSplits;
  return s < 1 ? 1 : (int32_t)s;
}

pkv_status pkv_append(const void* k, const void* v, const int32_t* slot_mapping,
                      int32_t num_tokens, void* k_cache, void* v_cache, int32_t num_blocks,
                      int32_t block_size, int32_t num_kv_heads, int32_t head_dim, void* stream) {
  return append_impl(k, v, slot_mapping, num_tokens, k_cache, v_cache, num_blocks, block_size,
                     num_kv_heads, head_dim, static_cast<cudaStream_t>(stream), false);
}

pkv_status pkv_append_vllm_layout(const void* k, const void* v, const int32_t* slot_mapping,
                                  int32_t num_tokens, void* k_cache, void* v_cache,
                                  int32_t num_blocks, int32_t block_size, int32_t num_kv_heads,
                                  int32_t head_dim, void* stream) {
  return append_impl(k, v, slot_mapping, num_tokens, k_cache, v_cache, num_blocks, block_size,
                     num_kv_heads, head_dim, static_cast<cudaStream_t>(stream), true);
}

pkv_status pkv_decode(const void* q, const void* k_cache, const void* v_cache,
                      const int32_t* block_tables, const int32_t* context_lens, int32_t num_seqs,
                      int32_t max_blocks_per_seq, int32_t num_blocks, float scale,
                      int32_t num_heads, int32_t num_kv_heads, int32_t head_dim,
                      int32_t block_size, void* out, void* stream) {
  const DecodeArgs a{q, k_cache, v_cache, block_tables, context_lens, num_seqs,
                     max_blocks_per_seq, num_blocks, scale, num_heads, num_kv_heads,
                     head_dim, block_size, out};
  pkv_status st = validate_decode(a);
  if (st != PKV_OK) return st;
  if (num_seqs == 0) return PKV_OK;
  return single_pass(a, static_cast<cudaStream_t>(stream));
}

}  // extern "C"

namespace pkv {
namespace {

// The split count a decode call launches for `num_splits` (0 = the
// heuristic for the current GPU): 1 (single pass) or 2..PKV_MAX_SPLITS.
// More splits than table blocks cannot all hold work, so the count is capped
// at max_blocks_per_seq.
pkv_status resolve_decode_splits(int num_seqs, int num_kv_heads, int max_blocks_per_seq,
                                 int block_size, int num_splits, int* S_out) {
  if (num_splits < 0 || num_splits > PKV_MAX_SPLITS)
    return fail(PKV_ERR_INVALID_ARG, "num_splits %d outside 0..%d", num_splits, PKV_MAX_SPLITS);
  int S = num_splits;
  if (S == 0) {
    int sms = 0;
    if (current_device_sms(&sms) != 0) return fail(PKV_ERR_CUDA, "cannot query the SM count");
    S = pkv_pick_num_splits(num_seqs, num_kv_heads, max_blocks_per_seq * block_size, block_size,
                            sms);
  }
  *S_out = S < 1 ? 1 : (S > max_blocks_per_seq ? max_blocks_per_seq : S);
  return PKV_OK;
}

// Whether a varlen call of these sizes is chunked prefill (the tcgen05
// prefill kernel on blocked pools; the split count below for either layout,
// so that the plan does not depend on the layout).
bool prefill_shaped(int num_heads, int num_kv_heads, int max_q_len, int head_dim) {
  return PKV_PREFILL_TC && head_dim == TcPrefillShape::D && num_kv_heads > 0 &&
         (long long)max_q_len * (num_heads / num_kv_heads) >= TcPrefillShape::kRows;
}

// Split count of a chunked-prefill call: below one wave of one CTA per SM,
// the count that brings the grid of tile pairs nearest one wave, each split
// keeping at least kMinPrefillSplitTokens of the table's capacity.
int prefill_pick_num_splits(int num_seqs, int num_heads, int num_kv_heads, int max_q_len,
                            int max_blocks_per_seq, int block_size, int num_sms) {
  const int G = num_heads / num_kv_heads;
  const int qc = TcPrefillShape::kTiles * (TcPrefillShape::kRows / G);
  const long long pairs = (long long)num_seqs * num_kv_heads * ((max_q_len + qc - 1) / qc);
  long long s = pairs >= num_sms ? 1 : (2LL * num_sms + pairs) / (2 * pairs);
  const long long cap_tokens = (long long)max_blocks_per_seq * block_size;
  if (s > cap_tokens / kMinPrefillSplitTokens) s = cap_tokens / kMinPrefillSplitTokens;
  if (s > kMaxAutoSplits) s = kMaxAutoSplits;
  return s < 1 ? 1 : (int)s;
}

// The same for varlen split-K (0 = pkv_varlen_pick_num_splits, or the
// prefill rule above for chunked-prefill sizes).
pkv_status resolve_varlen_splits(int num_seqs, int num_heads, int num_kv_heads, int max_q_len,
                                 int max_blocks_per_seq, int block_size, int head_dim,
                                 int num_splits, int* S_out) {
  if (num_splits < 0 || num_splits > PKV_MAX_SPLITS)
    return fail(PKV_ERR_INVALID_ARG, "num_splits %d outside 0..%d", num_splits, PKV_MAX_SPLITS);
  int S = num_splits;
  if (S == 0) {
    int sms = 0;
    if (current_device_sms(&sms) != 0) return fail(PKV_ERR_CUDA, "cannot query the SM count");
    S = prefill_shaped(num_heads, num_kv_heads, max_q_len, head_dim)
            ? prefill_pick_num_splits(num_seqs, num_heads, num_kv_heads, max_q_len,
                                      max_blocks_per_seq, block_size, sms)
            : pkv_varlen_pick_num_splits(num_seqs, num_heads, num_kv_heads, max_q_len,
                                         max_blocks_per_seq, block_size, sms);
  }
  *S_out = S < 1 ? 1 : (S > max_blocks_per_seq ? max_blocks_per_seq : S);
  return PKV_OK;
}

// The body of pkv_decode_splitk and pkv_append_decode (arguments validated).
pkv_status decode_impl(const DecodeArgs& a, int num_splits, void* scratch, size_t scratch_bytes,
                       cudaStream_t cs, const FuseArgs* fuse) {
  pkv_status st = PKV_OK;
  const int num_seqs = a.num_seqs, num_kv_heads = a.num_kv_heads, num_heads = a.num_heads;
  const int max_blocks_per_seq = a.max_blocks_per_seq, block_size = a.block_size;
  const int head_dim = a.head_dim;
  if (num_splits < 0 || num_splits > PKV_MAX_SPLITS)
    return fail(PKV_ERR_INVALID_ARG, "num_splits %d outside 0..%d", num_splits, PKV_MAX_SPLITS);
  if (num_seqs == 0) return PKV_OK;

  int S = 0;
  st = resolve_decode_splits(num_seqs, num_kv_heads, max_blocks_per_seq, block_size, num_splits, &S);
  if (st != PKV_OK) return st;
  const int S_eff = S;
  if (S_eff <= 1) return single_pass(a, cs, fuse);

  const size_t need = pkv_splitk_scratch_bytes(num_seqs, num_heads, head_dim, S_eff);
  if (!scratch || scratch_bytes < need)
    return fail(PKV_ERR_SCRATCH_TOO_SMALL, "split-K with %d splits needs %zu scratch bytes, got %zu",
                S_eff, need, scratch ? scratch_bytes : (size_t)0);
  if (!aligned(scratch, 16)) return fail(PKV_ERR_INVALID_ARG, "scratch must be 16-byte aligned");
  const long long grid1 = (long long)num_seqs * num_kv_heads * S_eff;
  if (grid1 >= (1ll << 31)) return fail(PKV_ERR_INVALID_ARG, "grid too large");

  const size_t rows = (size_t)num_seqs * num_heads * S_eff;
  const SplitScratch sc = carve_scratch(scratch, rows, head_dim);
  DecodeParams prm = base_params(a);
  apply_fuse(prm, fuse);
  prm.num_splits = S_eff;
  // the heuristic keeps a split at >= kMinSplitTokens; forced counts cut the
  // longest context into exactly S chunks
  prm.min_chunk_blocks = num_splits == 0 ? (kMinSplitTokens + block_size - 1) / block_size : 1;
  prm.chunk_hint = (max_blocks_per_seq + S_eff - 1) / S_eff;
  prm.split_header = sc.header;
  prm.part_out = sc.part_out;
  prm.part_m = sc.part_m;
  prm.part_l = sc.part_l;
  st = dispatch_decode<true>(a, prm, cs, (int)grid1);
  if (st != PKV_OK) return st;

  CombineParams cp{};
  cp.part_out = sc.part_out;
  cp.part_m = sc.part_m;
  cp.part_l = sc.part_l;
  cp.context_lens = a.context_lens;
  cp.split_header = sc.header;
  cp.out = static_cast<__half*>(a.out);
  cp.num_rows = num_seqs * num_heads;
  cp.num_heads = num_heads;
  cp.num_splits = S_eff;
  cp.block_size = block_size;
  cp.cap_tokens = max_blocks_per_seq * block_size;
  const cudaError_t e = launch_combine(splitk_combine_kernel<64>, splitk_combine_kernel<128>,
                                       head_dim, (long long)num_seqs * num_heads, cs, cp);
  if (e != cudaSuccess) return cuda_fail(e, "split-K combine launch");
  return PKV_OK;
}

// The body of pkv_varlen_attention and its vLLM-layout twin.
pkv_status varlen_impl(const void* q, const void* k_cache, const void* v_cache,
                       const int32_t* cu_seqlens_q, const int32_t* pos_offsets,
                       const int32_t* block_tables, int num_seqs, int total_q, int max_q_len,
                       int max_blocks_per_seq, int num_blocks, float scale, int num_heads,
                       int num_kv_heads, int head_dim, int block_size, void* out,
                       int num_splits, void* scratch, size_t scratch_bytes, cudaStream_t cs,
                       bool vllm) {
  // pos_offsets stands in for context_lens in the shared checks
  const DecodeArgs a{q, k_cache, v_cache, block_tables, pos_offsets, num_seqs,
                     max_blocks_per_seq, num_blocks, scale, num_heads, num_kv_heads,
                     head_dim, block_size, out};
  pkv_status st = validate_decode(a);
  if (st != PKV_OK) return st;
  if (!cu_seqlens_q || !aligned(cu_seqlens_q, 4))
    return fail(PKV_ERR_INVALID_ARG, "cu_seqlens_q must be a 4-byte aligned device pointer");
  if (total_q < 0 || max_q_len < 0) return fail(PKV_ERR_INVALID_ARG, "total_q / max_q_len < 0");
  if (num_splits < 0 || num_splits > PKV_MAX_SPLITS)
    return fail(PKV_ERR_INVALID_ARG, "num_splits %d outside 0..%d", num_splits, PKV_MAX_SPLITS);
  if (num_seqs == 0 || total_q == 0 || max_q_len == 0) return PKV_OK;
  const int G = num_heads / num_kv_heads;
  // two n-tiles (16 columns) once a sequence has more than 8 (query, head)
  // pairs: each chunk then reads its context once for twice the queries
  const int NT = (long long)max_q_len * G > 8 ? 2 : 1;
  const int qc = G >= 8 * NT ? 1 : 8 * NT / G;
  const int chunks = (max_q_len + qc - 1) / qc;
  const long long grid = (long long)num_seqs * num_kv_heads * chunks;
  if (grid >= (1ll << 31)) return fail(PKV_ERR_INVALID_ARG, "grid too large");
  VarlenParams vp{};
  vp.q = static_cast<const __half*>(q);
  vp.cu_seqlens_q = cu_seqlens_q;
  vp.pos_offsets = pos_offsets;
  vp.block_tables = block_tables;
  vp.out = static_cast<__half*>(out);
  vp.total_q = total_q;
  vp.num_heads = num_heads;
  vp.num_kv_heads = num_kv_heads;
  vp.group = G;
  vp.qc = qc;
  vp.num_chunks = chunks;
  vp.num_seqs = num_seqs;
  vp.max_blocks_per_seq = max_blocks_per_seq;
  vp.num_blocks = num_blocks;
  vp.scale_log2 = scale * 1.4426950408889634f;
  vp.num_splits = 1;
  vp.min_chunk_blocks = 1;

  int S_eff = 1;
  st = resolve_varlen_splits(num_seqs, num_heads, num_kv_heads, max_q_len, max_blocks_per_seq,
                             block_size, head_dim, num_splits, &S_eff);
  if (st != PKV_OK) return st;
  // chunked prefill on blocked pools: pairs of tiles of 128 / G queries,
  // 2 x 128 (query, head) rows per CTA, on the tcgen05 prefill kernel
  const bool prefill = !vllm && prefill_shaped(num_heads, num_kv_heads, max_q_len, head_dim);
  long long base_grid = grid;
  if (prefill) {
    vp.qc = TcPrefillShape::kTiles * (TcPrefillShape::kRows / G);
    vp.num_chunks = (max_q_len + vp.qc - 1) / vp.qc;
    base_grid = (long long)num_seqs * num_kv_heads * vp.num_chunks;
  }
  auto launch_prefill = [&](bool split, long long g) {
    if (split)
      return block_size == 16 ? launch_prefill_tc<16, true>(a, vp, cs, (int)g)
                              : launch_prefill_tc<32, true>(a, vp, cs, (int)g);
    return block_size == 16 ? launch_prefill_tc<16, false>(a, vp, cs, (int)g)
                            : launch_prefill_tc<32, false>(a, vp, cs, (int)g);
  };
  if (S_eff <= 1) {
    if (base_grid >= (1ll << 31)) return fail(PKV_ERR_INVALID_ARG, "grid too large");
    return prefill ? launch_prefill(false, base_grid)
                   : dispatch_varlen<false>(a, vp, cs, (int)grid, NT, vllm);
  }

  const size_t need = pkv_splitk_scratch_bytes(total_q, num_heads, head_dim, S_eff);
  if (!scratch || scratch_bytes < need)
    return fail(PKV_ERR_SCRATCH_TOO_SMALL, "varlen split-K with %d splits needs %zu scratch bytes, got %zu",
                S_eff, need, scratch ? scratch_bytes : (size_t)0);
  if (!aligned(scratch, 16)) return fail(PKV_ERR_INVALID_ARG, "scratch must be 16-byte aligned");
  const long long grid1 = base_grid * S_eff;
  const long long grid2 = (long long)total_q * num_heads;
  if (grid1 >= (1ll << 31) || grid2 >= (1ll << 31))
    return fail(PKV_ERR_INVALID_ARG, "grid too large");
  const size_t rows = (size_t)total_q * num_heads * S_eff;
  const SplitScratch sc = carve_scratch(scratch, rows, head_dim);
  vp.num_splits = S_eff;
  const int min_tokens = prefill ? kMinPrefillSplitTokens : kMinSplitTokens;
  vp.min_chunk_blocks = num_splits == 0 ? (min_tokens + block_size - 1) / block_size : 1;
  vp.part_out = sc.part_out;
  vp.part_m = sc.part_m;
  vp.part_l = sc.part_l;
  st = prefill ? launch_prefill(true, grid1) : dispatch_varlen<true>(a, vp, cs, (int)grid1, NT, vllm);
  if (st != PKV_OK) return st;

  VarlenCombineParams cp{};
  cp.part_out = vp.part_out;
  cp.part_m = vp.part_m;
  cp.part_l = vp.part_l;
  cp.cu_seqlens_q = cu_seqlens_q;
  cp.out = static_cast<__half*>(out);
  cp.num_seqs = num_seqs;
  cp.total_q = total_q;
  cp.num_heads = num_heads;
  cp.num_splits = S_eff;
  cp.covered_q = vp.num_chunks * vp.qc;
  const cudaError_t e = launch_combine(varlen_combine_kernel<64>, varlen_combine_kernel<128>,
                                       head_dim, grid2, cs, cp);
  if (e != cudaSuccess) return cuda_fail(e, "varlen split-K combine launch");
  return PKV_OK;
}

}  // namespace
}  // namespace pkv

extern "C" {

pkv_status pkv_decode_splitk(const void* q, const void* k_cache, const void* v_cache,
                             const int32_t* block_tables, const int32_t* context_lens,
                             int32_t num_seqs, int32_t max_blocks_per_seq, int32_t num_blocks,
                             float scale, int32_t num_heads, int32_t num_kv_heads,
                             int32_t head_dim, int32_t block_size, void* out, int32_t num_splits,
                             void* scratch, size_t scratch_bytes, void* stream) {
  const DecodeArgs a{q, k_cache, v_cache, block_tables, context_lens, num_seqs,
                     max_blocks_per_seq, num_blocks, scale, num_heads, num_kv_heads,
                     head_dim, block_size, out};
  pkv_status st = validate_decode(a);
  if (st != PKV_OK) return st;
  return decode_impl(a, num_splits, scratch, scratch_bytes, static_cast<cudaStream_t>(stream),
                     nullptr);
}

pkv_status pkv_decode_vllm_layout(const void* q, const void* k_cache, const void* v_cache,
                                  const int32_t* block_tables, const int32_t* context_lens,
                                  int32_t num_seqs, int32_t max_blocks_per_seq,
                                  int32_t num_blocks, float scale, int32_t num_heads,
                                  int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                                  void* out, int32_t num_splits, void* scratch,
                                  size_t scratch_bytes, void* stream) {
  DecodeArgs a{q, k_cache, v_cache, block_tables, context_lens, num_seqs,
               max_blocks_per_seq, num_blocks, scale, num_heads, num_kv_heads,
               head_dim, block_size, out};
  a.vllm = true;
  pkv_status st = validate_decode(a);
  if (st != PKV_OK) return st;
  return decode_impl(a, num_splits, scratch, scratch_bytes, static_cast<cudaStream_t>(stream),
                     nullptr);
}

pkv_status pkv_append_decode(const void* k_new, const void* v_new, const int32_t* slot_mapping,
                             void* k_cache, void* v_cache, const void* q,
                             const int32_t* block_tables, const int32_t* context_lens,
                             int32_t num_seqs, int32_t max_blocks_per_seq, int32_t num_blocks,
                             float scale, int32_t num_heads, int32_t num_kv_heads,
                             int32_t head_dim, int32_t block_size, void* out, int32_t num_splits,
                             void* scratch, size_t scratch_bytes, void* stream) {
  const DecodeArgs a{q, k_cache, v_cache, block_tables, context_lens, num_seqs,
                     max_blocks_per_seq, num_blocks, scale, num_heads, num_kv_heads,
                     head_dim, block_size, out};
  pkv_status st = validate_decode(a);
  if (st != PKV_OK) return st;
  if (!k_new || !v_new || !slot_mapping)
    return fail(PKV_ERR_INVALID_ARG, "k_new, v_new and slot_mapping must not be NULL");
  if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(slot_mapping, 4))
    return fail(PKV_ERR_INVALID_ARG,
                "k_new and v_new must be 16-byte aligned, slot_mapping 4-byte aligned");
  FuseArgs f;
  f.k_new = k_new;
  f.v_new = v_new;
  f.slots = slot_mapping;
  f.k_cache = k_cache;
  f.v_cache = v_cache;
  return decode_impl(a, num_splits, scratch, scratch_bytes, static_cast<cudaStream_t>(stream), &f);
}

pkv_status pkv_varlen_attention(const void* q, const void* k_cache, const void* v_cache,
                                const int32_t* cu_seqlens_q, const int32_t* pos_offsets,
                                const int32_t* block_tables, int32_t num_seqs, int32_t total_q,
                                int32_t max_q_len, int32_t max_blocks_per_seq,
                                int32_t num_blocks, float scale, int32_t num_heads,
                                int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                                void* out, void* stream) {
  return varlen_impl(q, k_cache, v_cache, cu_seqlens_q, pos_offsets, block_tables, num_seqs,
                     total_q, max_q_len, max_blocks_per_seq, num_blocks, scale, num_heads,
                     num_kv_heads, head_dim, block_size, out, 1, nullptr, 0,
                     static_cast<cudaStream_t>(stream), false);
}

pkv_status pkv_varlen_attention_vllm_layout(
    const void* q, const void* k_cache, const void* v_cache, const int32_t* cu_seqlens_q,
    const int32_t* pos_offsets, const int32_t* block_tables, int32_t num_seqs, int32_t total_q,
    int32_t max_q_len, int32_t max_blocks_per_seq, int32_t num_blocks, float scale,
    int32_t num_heads, int32_t num_kv_heads, int32_t head_dim, int32_t block_size, void* out,
    void* stream) {
  return varlen_impl(q, k_cache, v_cache, cu_seqlens_q, pos_offsets, block_tables, num_seqs,
                     total_q, max_q_len, max_blocks_per_seq, num_blocks, scale, num_heads,
                     num_kv_heads, head_dim, block_size, out, 1, nullptr, 0,
                     static_cast<cudaStream_t>(stream), true);
}

pkv_status pkv_varlen_attention_splitk(
    const void* q, const void* k_cache, const void* v_cache, const int32_t* cu_seqlens_q,
    const int32_t* pos_offsets, const int32_t* block_tables, int32_t num_seqs, int32_t total_q,
    int32_t max_q_len, int32_t max_blocks_per_seq, int32_t num_blocks, float scale,
    int32_t num_heads, int32_t num_kv_heads, int32_t head_dim, int32_t block_size, void* out,
    int32_t num_splits, void* scratch, size_t scratch_bytes, void* stream) {
  return varlen_impl(q, k_cache, v_cache, cu_seqlens_q, pos_offsets, block_tables, num_seqs,
                     total_q, max_q_len, max_blocks_per_seq, num_blocks, scale, num_heads,
                     num_kv_heads, head_dim, block_size, out, num_splits, scratch, scratch_bytes,
                     static_cast<cudaStream_t>(stream), false);
}

pkv_status pkv_varlen_attention_splitk_vllm_layout(
    const void* q, const void* k_cache, const void* v_cache, const int32_t* cu_seqlens_q,
    const int32_t* pos_offsets, const int32_t* block_tables, int32_t num_seqs, int32_t total_q,
    int32_t max_q_len, int32_t max_blocks_per_seq, int32_t num_blocks, float scale,
    int32_t num_heads, int32_t num_kv_heads, int32_t head_dim, int32_t block_size, void* out,
    int32_t num_splits, void* scratch, size_t scratch_bytes, void* stream) {
  return varlen_impl(q, k_cache, v_cache, cu_seqlens_q, pos_offsets, block_tables, num_seqs,
                     total_q, max_q_len, max_blocks_per_seq, num_blocks, scale, num_heads,
                     num_kv_heads, head_dim, block_size, out, num_splits, scratch, scratch_bytes,
                     static_cast<cudaStream_t>(stream), true);
}

pkv_status pkv_decode_splitk_plan(int32_t num_seqs, int32_t num_heads, int32_t num_kv_heads,
                                  int32_t head_dim, int32_t max_blocks_per_seq,
                                  int32_t block_size, int32_t num_splits, int32_t* splits,
                                  size_t* scratch_bytes) {
  if (!splits || !scratch_bytes) return fail(PKV_ERR_INVALID_ARG, "splits and scratch_bytes must not be NULL");
  if (num_seqs < 0 || num_heads <= 0 || num_kv_heads <= 0 || num_heads % num_kv_heads != 0 ||
      head_dim <= 0 || max_blocks_per_seq <= 0 || block_size <= 0)
    return fail(PKV_ERR_INVALID_ARG, "invalid sizes");
  if ((long long)max_blocks_per_seq * block_size >= (1ll << 31))
    return fail(PKV_ERR_INVALID_ARG, "max_blocks_per_seq * block_size overflows");
  int S = 1;
  const pkv_status st = resolve_decode_splits(num_seqs, num_kv_heads, max_blocks_per_seq,
                                              block_size, num_splits, &S);
  if (st != PKV_OK) return st;
  *splits = S;
  *scratch_bytes = (S == 1 || num_seqs == 0) ? 0 : pkv_splitk_scratch_bytes(num_seqs, num_heads, head_dim, S);
  return PKV_OK;
}

pkv_status pkv_varlen_splitk_plan(int32_t num_seqs, int32_t total_q, int32_t max_q_len,
                                  int32_t num_heads, int32_t num_kv_heads, int32_t head_dim,
                                  int32_t max_blocks_per_seq, int32_t block_size,
                                  int32_t num_splits, int32_t* splits, size_t* scratch_bytes) {
  if (!splits || !scratch_bytes) return fail(PKV_ERR_INVALID_ARG, "splits and scratch_bytes must not be NULL");
  if (num_seqs < 0 || total_q < 0 || max_q_len < 0 || num_heads <= 0 || num_kv_heads <= 0 ||
      num_heads % num_kv_heads != 0 || head_dim <= 0 || max_blocks_per_seq <= 0 || block_size <= 0)
    return fail(PKV_ERR_INVALID_ARG, "invalid sizes");
  if ((long long)max_blocks_per_seq * block_size >= (1ll << 31))
    return fail(PKV_ERR_INVALID_ARG, "max_blocks_per_seq * block_size overflows");
  if (num_seqs == 0 || total_q == 0 || max_q_len == 0) {
    if (num_splits < 0 || num_splits > PKV_MAX_SPLITS)
      return fail(PKV_ERR_INVALID_ARG, "num_splits %d outside 0..%d", num_splits, PKV_MAX_SPLITS);
    *splits = 1;
    *scratch_bytes = 0;
    return PKV_OK;
  }
  int S = 1;
  const pkv_status st = resolve_varlen_splits(num_seqs, num_heads, num_kv_heads, max_q_len,
                                              max_blocks_per_seq, block_size, head_dim,
                                              num_splits, &S);
  if (st != PKV_OK) return st;
  *splits = S;
  *scratch_bytes = S == 1 ? 0 : pkv_splitk_scratch_bytes(total_q, num_heads, head_dim, S);
  return PKV_OK;
}

}  // extern "C"

namespace pkv {
namespace {

// qkv_norm_rope_kernel<D, BS, NS> for the runtime head_dim, block_size and
// slot count (NS0 .. 4).
template <int NS0>
cudaError_t launch_qkv(int head_dim, int block_size, int NS, dim3 grid, cudaStream_t cs,
                       const QkvRopeParams& qp) {
  if constexpr (NS0 <= 4) {
    if (NS != NS0) return launch_qkv<NS0 + 1>(head_dim, block_size, NS, grid, cs, qp);
    if (head_dim == 128)
      return block_size == 16 ? launch_pdl(qkv_norm_rope_kernel<128, 16, NS0>, grid, 128, 0, cs, qp)
                              : launch_pdl(qkv_norm_rope_kernel<128, 32, NS0>, grid, 128, 0, cs, qp);
    return block_size == 16 ? launch_pdl(qkv_norm_rope_kernel<64, 16, NS0>, grid, 128, 0, cs, qp)
                            : launch_pdl(qkv_norm_rope_kernel<64, 32, NS0>, grid, 128, 0, cs, qp);
  } else {
    return cudaErrorInvalidValue;
  }
}

}  // namespace
}  // namespace pkv

extern "C" {

pkv_status pkv_qkv_norm_rope_append(const void* qkv, const void* q_norm_w, const void* k_norm_w,
                                    const float* cos_table, const float* sin_table, void* q_out,
                                    void* k_cache, void* v_cache, const int32_t* cu_seqlens_q,
                                    const int32_t* pos_offsets, const int32_t* block_tables,
                                    int32_t num_seqs, int32_t total_q, int32_t max_blocks_per_seq,
                                    int32_t num_blocks, int32_t num_heads, int32_t num_kv_heads,
                                    int32_t head_dim, int32_t block_size, int32_t max_pos, float eps,
                                    void* stream) {
  if (!qkv || !cos_table || !sin_table || !q_out || !k_cache || !v_cache || !cu_seqlens_q ||
      !pos_offsets || !block_tables)
    return fail(PKV_ERR_INVALID_ARG, "a required pointer is NULL");
  if (num_seqs < 0 || total_q < 0) return fail(PKV_ERR_INVALID_ARG, "num_seqs / total_q < 0");
  if (num_heads <= 0 || num_kv_heads <= 0 || num_heads % num_kv_heads != 0)
    return fail(PKV_ERR_INVALID_ARG, "num_heads (%d) must be a positive multiple of num_kv_heads (%d)",
                num_heads, num_kv_heads);
  if (max_blocks_per_seq <= 0 || num_blocks <= 0 || max_pos <= 0 || head_dim <= 0 ||
      block_size <= 0)
    return fail(PKV_ERR_INVALID_ARG, "sizes must be positive");
  if (!std::isfinite(eps) || eps < 0.f) return fail(PKV_ERR_INVALID_ARG, "eps must be finite and >= 0");
  if (head_dim != 64 && head_dim != 128)
    return fail(PKV_ERR_UNSUPPORTED, "head_dim %d (built: 64, 128)", head_dim);
  if (block_size != 16 && block_size != 32)
    return fail(PKV_ERR_UNSUPPORTED, "block_size %d (built: 16, 32)", block_size);
  if ((long long)num_blocks * block_size >= (1ll << 31) ||
      (long long)max_blocks_per_seq * block_size >= (1ll << 31))
    return fail(PKV_ERR_INVALID_ARG, "pool or table too large for 32-bit positions");
  if (!aligned(qkv, 16) || !aligned(q_out, 16) || !aligned(k_cache, 16) ||
      !aligned(v_cache, 16) || (q_norm_w && !aligned(q_norm_w, 16)) ||
      (k_norm_w && !aligned(k_norm_w, 16)) || !aligned(cos_table, 16) ||
      !aligned(sin_table, 16) || !aligned(cu_seqlens_q, 4) || !aligned(pos_offsets, 4) ||
      !aligned(block_tables, 4))
    return fail(PKV_ERR_INVALID_ARG,
                "misaligned pointer (rows, weights, tables and pools: 16 bytes; indices: 4)");
  if (num_seqs == 0 || total_q == 0) return PKV_OK;
  QkvRopeParams qp{};
  qp.qkv = static_cast<const __half*>(qkv);
  qp.q_norm_w = static_cast<const __half*>(q_norm_w);
  qp.k_norm_w = static_cast<const __half*>(k_norm_w);
  qp.cos_t = cos_table;
  qp.sin_t = sin_table;
  qp.q_out = static_cast<__half*>(q_out);
  qp.k_cache = static_cast<__half*>(k_cache);
  qp.v_cache = static_cast<__half*>(v_cache);
  qp.cu_seqlens_q = cu_seqlens_q;
  qp.pos_offsets = pos_offsets;
  qp.block_tables = block_tables;
  qp.num_seqs = num_seqs;
  qp.total_q = total_q;
  qp.num_heads = num_heads;
  qp.num_kv_heads = num_kv_heads;
  qp.max_blocks_per_seq = max_blocks_per_seq;
  qp.num_blocks = num_blocks;
  qp.block_size = block_size;
  qp.max_pos = max_pos;
  qp.eps = eps;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  // slots per warp: the fewest idle head slots per row, then the most heads per CTA
  const int heads = num_heads + 2 * num_kv_heads;
  int NS = 1, best = 1 << 30;
  for (int ns = 1; ns <= 4; ++ns) {
    const int per = qkv_heads_per_cta(head_dim, ns);
    const int waste = (heads + per - 1) / per * per - heads;
    if (waste <= best) {
      best = waste;
      NS = ns;
    }
  }
  const int per_cta = qkv_heads_per_cta(head_dim, NS);
  const int groups = (heads + per_cta - 1) / per_cta;
  if (groups > 65535) return fail(PKV_ERR_INVALID_ARG, "too many heads");
  const dim3 grid((unsigned)total_q, (unsigned)groups, 1);  // x: token, y: group of heads
  cudaError_t e = launch_qkv<1>(head_dim, block_size, NS, grid, cs, qp);
  if (e != cudaSuccess) return cuda_fail(e, "qkv norm/rope/append launch");
  return PKV_OK;
}

pkv_status pkv_qkv_norm_rope_append_decode(
    const void* qkv, const void* q_norm_w, const void* k_norm_w, const float* cos_table,
    const float* sin_table, int32_t max_pos, float eps, void* k_cache, void* v_cache,
    const int32_t* block_tables, const int32_t* context_lens, int32_t num_seqs,
    int32_t max_blocks_per_seq, int32_t num_blocks, float scale, int32_t num_heads,
    int32_t num_kv_heads, int32_t head_dim, int32_t block_size, void* out, int32_t num_splits,
    void* scratch, size_t scratch_bytes, void* stream) {
  // qkv stands in for q in the shared checks (4-byte alignment)
  const DecodeArgs a{qkv, k_cache, v_cache, block_tables, context_lens, num_seqs,
                     max_blocks_per_seq, num_blocks, scale, num_heads, num_kv_heads,
                     head_dim, block_size, out};
  pkv_status st = validate_decode(a);
  if (st != PKV_OK) return st;
  if (!cos_table || !sin_table) return fail(PKV_ERR_INVALID_ARG, "a required pointer is NULL");
  if (max_pos <= 0) return fail(PKV_ERR_INVALID_ARG, "max_pos must be positive");
  if (!std::isfinite(eps) || eps < 0.f) return fail(PKV_ERR_INVALID_ARG, "eps must be finite and >= 0");
  if ((q_norm_w && !aligned(q_norm_w, 2)) || (k_norm_w && !aligned(k_norm_w, 2)) ||
      !aligned(cos_table, 4) || !aligned(sin_table, 4))
    return fail(PKV_ERR_INVALID_ARG, "misaligned pointer");
  if ((long long)num_seqs * (num_heads + 2 * num_kv_heads) * head_dim >= (1ll << 40))
    return fail(PKV_ERR_INVALID_ARG, "qkv too large");
  FuseArgs f;
  f.k_cache = k_cache;
  f.v_cache = v_cache;
  f.qkv = qkv;
  f.q_norm_w = q_norm_w;
  f.k_norm_w = k_norm_w;
  f.cos_t = cos_table;
  f.sin_t = sin_table;
  f.max_pos = max_pos;
  f.eps = eps;
  return decode_impl(a, num_splits, scratch, scratch_bytes, static_cast<cudaStream_t>(stream), &f);
}

pkv_status pkv_selftest_wait_timeout(void* stream) {
  const cudaError_t e = launch_pdl(wait_timeout_probe_kernel, 1, 32, 0,
                                   static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "wait-timeout probe launch");
  return PKV_OK;
}

pkv_status pkv_read_device_status(int32_t* flags, void* stream) {
  if (!flags) return fail(PKV_ERR_INVALID_ARG, "flags is NULL");
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  unsigned int host = 0;
  cudaError_t e = cudaMemcpyFromSymbolAsync(&host, g_device_status, sizeof(host), 0,
                                            cudaMemcpyDeviceToHost, cs);
  if (e != cudaSuccess) return cuda_fail(e, "reading the device status word");
  void* addr = nullptr;
  e = cudaGetSymbolAddress(&addr, g_device_status);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(status)");
  e = cudaMemsetAsync(addr, 0, sizeof(unsigned int), cs);
  if (e != cudaSuccess) return cuda_fail(e, "clearing the device status word");
  e = cudaStreamSynchronize(cs);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  *flags = (int32_t)host;
  return PKV_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// pkv_decode_splitk_noalloc: split-K with a built-in static scratch buffer,
// for callers that cannot allocate device memory (see include/pagedkv.h).
// ---------------------------------------------------------------------------

namespace pkv {
namespace {

// The built-in split-K scratch.  In host code this name is only a stand-in
// for the device array: its device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_noalloc_scratch[PKV_NOALLOC_SCRATCH_BYTES];

std::mutex g_noalloc_mutex;
void* g_noalloc_ptr[64] = {};  // per device ordinal, filled on first use

// Device address of g_noalloc_scratch on the current device.
pkv_status noalloc_scratch(void** ptr) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  if (dev >= 0 && dev < 64 && g_noalloc_ptr[dev]) {
    *ptr = g_noalloc_ptr[dev];
    return PKV_OK;
  }
  void* p = nullptr;
  e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
  if (e != cudaSuccess || !p) return cuda_fail(e, "cudaGetSymbolAddress(built-in scratch)");
  if (dev >= 0 && dev < 64) g_noalloc_ptr[dev] = p;
  *ptr = p;
  return PKV_OK;
}

}  // namespace
}  // namespace pkv

extern "C" pkv_status pkv_decode_splitk_noalloc(
    const void* q, const void* k_cache, const void* v_cache, const int32_t* block_tables,
    const int32_t* context_lens, int32_t num_seqs, int32_t max_blocks_per_seq, int32_t num_blocks,
    float scale, int32_t num_heads, int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
    void* out, int32_t num_splits, void* stream) {
  const DecodeArgs a{q, k_cache, v_cache, block_tables, context_lens, num_seqs,
                     max_blocks_per_seq, num_blocks, scale, num_heads, num_kv_heads,
                     head_dim, block_size, out};
  pkv_status st = validate_decode(a);
  if (st != PKV_OK) return st;
  if (num_splits < 0 || num_splits > PKV_MAX_SPLITS)
    return fail(PKV_ERR_INVALID_ARG, "num_splits %d outside 0..%d", num_splits, PKV_MAX_SPLITS);
  if (num_seqs == 0) return PKV_OK;

  // The split count pkv_decode_splitk will use, and the scratch it needs.
  int S_eff = 1;
  size_t need = 0;
  st = pkv_decode_splitk_plan(num_seqs, num_heads, num_kv_heads, head_dim, max_blocks_per_seq,
                              block_size, num_splits, &S_eff, &need);
  if (st != PKV_OK) return st;
  if (need > (size_t)PKV_NOALLOC_SCRATCH_BYTES)
    return fail(PKV_ERR_SCRATCH_TOO_SMALL,
                "%d splits need %zu bytes of scratch but the built-in buffer holds %zu; use "
                "pkv_decode_splitk with caller scratch or fewer splits",
                S_eff, need, (size_t)PKV_NOALLOC_SCRATCH_BYTES);

  void* scratch = nullptr;
  st = noalloc_scratch(&scratch);
  if (st != PKV_OK) return st;
  return pkv_decode_splitk(q, k_cache, v_cache, block_tables, context_lens, num_seqs,
                           max_blocks_per_seq, num_blocks, scale, num_heads, num_kv_heads,
                           head_dim, block_size, out, num_splits, scratch,
                           (size_t)PKV_NOALLOC_SCRATCH_BYTES, stream);
}
