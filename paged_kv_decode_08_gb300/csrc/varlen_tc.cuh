// paged_varlen_tc_kernel: several causal queries per sequence over the paged
// cache (the varlen attention of kernels.cuh) with both products on the
// 5th-generation tensor cores, for head_dim 128 and chunks of more than 8
// (query, head) columns (speculative verification, multi-token decode).
//
// One CTA per (sequence, KV head, chunk of queries[, split]) as in
// paged_varlen_kernel; its 16 columns n = (query n / G, head n % G) (padded
// with zero queries) are the N of two MMAs per span of 128 context tokens:
//
//   S  [128 tok x 16]  = K_span [128 x 128] . Q^T              (M = 128, tensor memory)
//   O^T[128 d x 16]   += V_span^T [128 x 128] . P^T [128 x 16]  (M = 128, tensor memory)
//
// Warp roles.  Warps 5 .. copy each span's K and V (eight 16-row sub-tiles
// per tensor, one TMA box per 64-element half, each warp issuing its share
// of the 16 boxes, one per lane, landing as [2 halves][128 rows][64] with
// the 128-byte swizzle: the K-major and MN-major shared-memory layouts of
// the two MMAs) into a ring of three 32 KB slots taken in the order K0, K1,
// V0, K2, V1, ... (a span's V goes out after the next span's K, so that it
// is in flight while the span's scores and softmax run rather than held in
// a slot); a K slot is released when S has read it, a V slot when PV has.
// Warp 4 (one lane) issues each
// product as soon as its inputs are ready (S is double-buffered in tensor
// memory, so the next span's scores are computed during this span's
// softmax).  Warps 0-3 run the online softmax: lane l of warp w owns token
// 32w + l of the span (tensor-memory lane 32w + l) for all 16 columns,
// writes P (f16) to shared memory as the K-major B operand of the second
// MMA, and, in a span that holds positions that do not count, zeroes their
// V rows (0 x NaN would poison the product).  Each column keeps a reference
// maximum that moves only when a score exceeds it by 2^8 (one CTA vote per
// span decides; the new maxima go through shared memory and O is rescaled
// in tensor memory only then).  A span whose positions all count for every
// column (all but the last one or two of a chunk) takes a short path: one
// FMA per score, a max over the 16 columns for the vote, and the exponential.
//
// Every wait is bounded; a wait that runs out sets PKV_DEV_WAIT_TIMEOUT and
// the CTA stops, lets its copies and MMAs drain (bounded as well), writes
// nothing and frees its tensor memory.
#pragma once

#include "kernels.cuh"

// Warps that issue the copies (each takes 16 / n of a load's boxes): a warp
// issues TMA boxes at a bounded rate, so the copies of one CTA go faster
// when several warps share them.
#ifndef PKV_TC_COPY_WARPS
#define PKV_TC_COPY_WARPS 2
#endif

// Sleep (ns) between polls of the copy and MMA threads; 0 spins.
#ifndef PKV_TC_POLL_NS
#define PKV_TC_POLL_NS 0
#endif

namespace pkv {

template <int D>
struct TcVarlenShape {
  static_assert(D == 128, "the tcgen05 varlen kernel is built for head_dim 128");
  static constexpr int kSpan = 128;                  // context tokens per span (M of S)
  static constexpr int kSubs = kSpan / 16;           // 16-row sub-tiles per span
  static constexpr int kHalves = D / 64;             // 128-byte rows per token
  static constexpr int kHalfBytes = kSpan * 128;     // one 64-element half of a span: 16 KB
  static constexpr int kSlotBytes = kHalves * kHalfBytes;  // K (or V) of a span: 32 KB
  static constexpr int kSlots = 3;
  static constexpr int kRingBytes = kSlots * kSlotBytes;   // 96 KB
  static constexpr int kQBytes = kHalves * 16 * 128;       // Q [d halves][16 cols][64]
  static constexpr int kPBytes = (kSpan / 64) * 16 * 128;  // P^T [token halves][16 cols][64]
  static constexpr int kQOff = kRingBytes;
  static constexpr int kPOff = kQOff + kQBytes;            // two P buffers
  static constexpr int kBarOff = kPOff + 2 * kPBytes;
  // full[3], empty[3], s_ready[2], s_free[2], p_ready[2], pv_done[2]
  static constexpr int kNumBars = 14;
  static constexpr int kSmemBytes = 1024 + kBarOff + kNumBars * 8;
  static constexpr int kTmemCols = 64;  // S[2] (16 columns each), O (16)
  static constexpr int kMmaWarp = 4;     // softmax warps 0-3, MMA warp 4, copy warps 5 ..
  static constexpr int kCopyWarps = PKV_TC_COPY_WARPS;
  static constexpr int kBoxesPerWarp = 2 * kSubs / kCopyWarps;
  static_assert(kHalves == 2 && kBoxesPerWarp % 2 == 0 && kBoxesPerWarp * kCopyWarps == 2 * kSubs,
                "each copy warp takes whole sub-tiles");
  static constexpr int kWarps = kMmaWarp + 1 + kCopyWarps;
  static constexpr int kThreads = kWarps * 32;
  static constexpr uint32_t kIdescS = mma_idesc_f16(128, 16, false, false);
  static constexpr uint32_t kIdescPV = mma_idesc_f16(128, 16, true, false);
};

// Element (row, e) of a [rows][64] f16 block stored with the 128-byte
// swizzle (16-byte chunk index XOR row % 8), as TMA writes it.
__device__ __forceinline__ uint32_t sw128_off(int row, int e) {
  return (uint32_t)(row * 128 + ((((e >> 3) ^ (row & 7))) << 4) + (e & 7) * 2);
}

// max(a, b, c) in one instruction (the three-input form of max.f32).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float y;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(y) : "f"(a), "f"(b), "f"(c));
  return y;
}

// 2^x by the hardware approximation (x <= 8 here; -inf gives 0).
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <int D, int BS, bool SPLIT>
__global__ void __launch_bounds__(TcVarlenShape<D>::kThreads, 2)
paged_varlen_tc_kernel(const __grid_constant__ CUtensorMap kmap,
                       const __grid_constant__ CUtensorMap vmap, const VarlenParams p) {
  using Sh = TcVarlenShape<D>;
  constexpr int SUB = BS / 16;  // 16-row sub-tiles per pool block
  extern __shared__ uint8_t smem_raw[];
  __shared__ int s_abort;
  __shared__ uint32_t s_tmem;
  __shared__ int s_max[Sh::kWarps];
  __shared__ float s_red[2][4][16];             // column maxima per warp (double-buffered)
  __shared__ float s_sum[4][16];                // final column sums per warp
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t ring = smem_addr(smem);
  const uint32_t qbuf = ring + Sh::kQOff;
  const uint32_t pbuf = ring + Sh::kPOff;
  const uint32_t bars = ring + Sh::kBarOff;
  auto full = [&](int i) { return bars + 8 * i; };
  auto empty = [&](int i) { return bars + 8 * (3 + i); };
  auto s_ready = [&](int i) { return bars + 8 * (6 + i); };
  auto s_free = [&](int i) { return bars + 8 * (8 + i); };
  auto p_ready = [&](int i) { return bars + 8 * (10 + i); };
  auto pv_done = [&](int i) { return bars + 8 * (12 + i); };
  // Ring loads in issue order: K0, then K(i+1), V(i) for each span i, V of
  // the last span last; load n goes to slot n % 3, its (n / 3)-th use.
  auto slot_of = [](int n) { return n % Sh::kSlots; };
  auto use_of = [](int n) { return (uint32_t)(n / Sh::kSlots); };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  int item = blockIdx.x;
  const int split = SPLIT ? item % p.num_splits : 0;
  if (SPLIT) item /= p.num_splits;
  const int qc_idx = item % p.num_chunks;
  item /= p.num_chunks;
  const int g = item % p.num_kv_heads;
  const int s = item / p.num_kv_heads;
  const int G = p.group;

  pdl_launch_dependents();
  if (threadIdx.x == 0) s_abort = 0;
  if (warp == Sh::kMmaWarp && lane == 0) {
#pragma unroll
    for (int i = 0; i < 3; ++i) {
      mbar_init(full(i), Sh::kCopyWarps);  // one arrival (with its bytes) per copy warp
      mbar_init(empty(i), 1);
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      mbar_init(s_ready(i), 1);
      mbar_init(s_free(i), 4);
      mbar_init(p_ready(i), 4);
      mbar_init(pv_done(i), 1);
    }
    fence_mbar_init();
  }
  pdl_wait();

  // ---- the chunk of queries and the positions it reads (as paged_varlen_kernel)
  const unsigned int status = *reinterpret_cast<volatile unsigned int*>(&g_device_status);
  const int cap = p.max_blocks_per_seq * BS;
  const int q_begin = __ldg(p.cu_seqlens_q + s);
  const int q_end = __ldg(p.cu_seqlens_q + s + 1);
  int pos0 = __ldg(p.pos_offsets + s);
  if (SPLIT) {
    int mx = 0;
    for (int i = threadIdx.x; i < p.num_seqs; i += Sh::kThreads) {
      int last = __ldg(p.pos_offsets + i) + __ldg(p.cu_seqlens_q + i + 1) -
                 __ldg(p.cu_seqlens_q + i);
      last = last < 0 ? 0 : (last > cap ? cap : last);
      mx = max(mx, (last + BS - 1) / BS);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if (lane == 0) s_max[warp] = mx;
  }
  if (__syncthreads_or(status & kDevWaitTimeout)) return;
  int nblk_max = 0;
  if (SPLIT) {
#pragma unroll
    for (int w = 0; w < Sh::kWarps; ++w) nblk_max = max(nblk_max, s_max[w]);
  }
  const int chunk = SPLIT ? max(p.min_chunk_blocks, (nblk_max + p.num_splits - 1) / p.num_splits)
                          : p.max_blocks_per_seq;
  if (q_begin < 0 || q_end < q_begin || q_end > p.total_q) {
    if (threadIdx.x == 0) atomicOr(&g_device_status, kDevBadContextLen);
    return;
  }
  const int q_len = q_end - q_begin;
  if (qc_idx == p.num_chunks - 1 && q_len > p.num_chunks * p.qc && threadIdx.x == 0)
    atomicOr(&g_device_status, kDevBadContextLen);
  const int t0 = qc_idx * p.qc;
  if (t0 >= q_len) return;
  const int nq = min(p.qc, q_len - t0);
  if (pos0 < 0 || pos0 + q_len > cap) {
    if (threadIdx.x == 0) atomicOr(&g_device_status, kDevBadContextLen);
    pos0 = pos0 < 0 ? 0 : max(0, cap - q_len);
  }
  const int chunk_end = min(cap, pos0 + t0 + nq);
  const int ncols = nq * G;  // <= 16
  int tok_begin = 0;
  int tok_end = chunk_end;
  if (SPLIT) {
    if ((long long)split * chunk * BS >= chunk_end) {
      for (int n = threadIdx.x; n < ncols; n += Sh::kThreads) {
        const size_t row = (size_t)(q_begin + t0 + n / G) * p.num_heads + (size_t)g * G + n % G;
        p.part_m[row * p.num_splits + split] = -CUDART_INF_F;
        p.part_l[row * p.num_splits + split] = 0.f;
      }
      return;
    }
    tok_begin = split * chunk * BS;
    tok_end = (int)min((long long)chunk_end, (long long)tok_begin + (long long)chunk * BS);
  }
  const int sub_begin = tok_begin / 16;
  const int n_tiles = (tok_end - tok_begin + 15) / 16;
  const int n_spans = (n_tiles + Sh::kSubs - 1) / Sh::kSubs;  // >= 1
  const int32_t* table = p.block_tables + (size_t)s * p.max_blocks_per_seq;

  auto kload = [&](int j) { return j == 0 ? 0 : 2 * j - 1; };                  // K(j)'s load
  auto vload = [&](int i) { return i == n_spans - 1 ? 2 * n_spans - 1 : 2 * i + 2; };  // V(i)'s

  // ---- set-up: tensor memory, the queries as the B operand of S
  if (warp == 0) tmem_alloc(smem_addr(&s_tmem), Sh::kTmemCols);
  if (warp < 4) {
    // 16 columns x D halves of 16 bytes; columns past ncols are zero
    for (int x = threadIdx.x; x < 16 * (D / 8); x += 128) {
      const int n = x / (D / 8), c = x % (D / 8);  // column, 16-byte chunk
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (n < ncols) {
        const size_t row = (size_t)(q_begin + t0 + n / G) * p.num_heads + (size_t)g * G + n % G;
        const uint32_t* src = reinterpret_cast<const uint32_t*>(p.q + row * D + c * 8);
        v = make_uint4(__ldg(src), __ldg(src + 1), __ldg(src + 2), __ldg(src + 3));
      }
      const uint32_t dst = qbuf + (c / 8) * (16 * 128) + sw128_off(n, (c % 8) * 8);
      asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(dst), "r"(v.x), "r"(v.y),
                   "r"(v.z), "r"(v.w)
                   : "memory");
    }
    fence_proxy_async_smem();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = s_tmem;
  const uint32_t tS = tbase;        // S buffers: columns 0..15 and 16..31
  const uint32_t tO = tbase + 32;   // O: columns 32..47

  auto abort_now = [&]() {
    atomicOr(&g_device_status, kDevWaitTimeout);
    *reinterpret_cast<volatile int*>(&s_abort) = 1;
  };
  auto aborted = [&]() { return *reinterpret_cast<volatile int*>(&s_abort) != 0; };
  auto wait = [&](uint32_t bar, uint32_t parity) {
    if (!mbar_wait_bounded(bar, parity, kWaitLimitNs)) {
      abort_now();
      return false;
    }
    return true;
  };

  if (warp > Sh::kMmaWarp) {
    // ================= copies (warps 5 ..) =================
    // A load is 16 boxes (8 sub-tiles x 2 halves).  Copy warp c issues boxes
    // c B .. c B + B - 1 (B = 16 / copy warps), one per lane (box 2u + h:
    // sub-tile u, half h).  Every copy warp walks the whole load sequence:
    // its lane 0 waits for the slot itself and arrives on the slot's full
    // barrier with the bytes of its own boxes before any of them is issued.
    const int box = (warp - Sh::kMmaWarp - 1) * Sh::kBoxesPerWarp + lane;
    const int u = box >> 1, hh = box & 1;
    const bool boxer = lane < Sh::kBoxesPerWarp;
    // this lane's table entry for span i (-1: no data)
    auto lookup = [&](int i) {
      const int t = i * Sh::kSubs + u;
      return (boxer && t < n_tiles) ? __ldg(table + (sub_begin + t) / SUB) : -1;
    };
    int issued = 0;
    // the entry of the span being loaded, the next span's (a span ahead), and
    // the validated entries of the last two spans' K loads (their V loads
    // follow one K later)
    int nxt = lookup(0), e0 = -1, e1 = -1;
    for (int n = 0; n < 2 * n_spans; ++n) {
      const bool last = n == 2 * n_spans - 1;
      const bool is_v = last || (n > 0 && !(n & 1));
      const int i = last ? n_spans - 1 : (is_v ? n / 2 - 1 : (n + 1) / 2);
      int e;
      if (!is_v) {
        e = nxt;
        if (i + 1 < n_spans) nxt = lookup(i + 1);  // in flight during the wait below
      } else {
        e = (i & 1) ? e1 : e0;
      }
      // the slot's previous load (n - 3) must have been released
      const int slot = slot_of(n);
      const uint32_t use = use_of(n);
      bool go = true;
      if (lane == 0) {
        if (use >= 1 && !(PKV_TC_POLL_NS ? mbar_wait_backoff(empty(slot), (use - 1) & 1,
                                                           kWaitLimitNs, PKV_TC_POLL_NS)
                                        : mbar_wait_bounded(empty(slot), (use - 1) & 1,
                                                            kWaitLimitNs))) {
          abort_now();
          go = false;
        }
        go = go && !aborted();
      }
      if (!__shfl_sync(0xffffffffu, go, 0)) break;
      if (!is_v) {
        const int t = i * Sh::kSubs + u;
        if (boxer && (e >= p.num_blocks || (e < 0 && t < n_tiles))) {
          if (hh == 0) atomicOr(&g_device_status, kDevBadBlockId);
          e = -1;
        }
        if (i & 1)
          e1 = e;
        else
          e0 = e;
      }
      const uint32_t ok = __ballot_sync(0xffffffffu, boxer && e >= 0);
      const uint32_t dst = ring + slot * Sh::kSlotBytes;
      if (lane == 0) mbar_arrive_expect_tx(full(slot), (uint32_t)(__popc(ok) * 2048));
      __syncwarp();
      if (boxer && e >= 0) {
        const int t = sub_begin + i * Sh::kSubs + u;
        tma_load_4d(dst + hh * Sh::kHalfBytes + u * 2048, is_v ? &vmap : &kmap, full(slot), 0,
                    (t % SUB) * 16, hh, e * p.num_kv_heads + g);
      }
      issued = n + 1;
    }
    // every started copy lands before the CTA can exit (bounded)
    if (lane == 0)
      for (int n = max(0, issued - Sh::kSlots); n < issued; ++n)
        (void)mbar_wait_bounded(full(slot_of(n)), use_of(n) & 1, kWaitLimitNs);
  } else if (warp == Sh::kMmaWarp) {
    // ================= MMAs (warp 4, lane 0) =================
    if (lane == 0) {
      uint32_t last_bar = 0, last_phase = 0;  // the last commit (drained before exit)
      // Issue whichever product is ready.  PV products go in span order (the
      // softmax warps rescale O between them) and need P and V; S(j) needs
      // K(j) and S buffer j % 2 read by the softmax warps (span j - 2).
      // A barrier's phase is tested by its parity alone, so a test must not
      // run while the slot's previous load can still be in flight (it would
      // see the completion before that one): K(j)'s slot held V(j - 3) (K0
      // for j = 2), which has landed once PV(j - 3) has been issued; V(i)'s
      // slot held K(i) (V(i - 2) for the last span), landed before S(i) (or
      // PV(i - 2)) was issued.
      int next_s = 0, next_pv = 0;
      uint64_t t_last = global_timer_ns();
      int idle = 0;
      while (next_pv < n_spans) {
        bool progressed = false;
        const int i = next_pv;
        const int vs = slot_of(vload(i));
        if (mbar_test(p_ready(i & 1), (i >> 1) & 1) && mbar_test(full(vs), use_of(vload(i)) & 1)) {
          tc_fence_after();
          // V^T is MN-major: its two d halves kHalfBytes apart, 8-token
          // groups 1 KB apart.  A descriptor's address field is the byte
          // address / 16, so a step within the operand adds its offset / 16.
          const uint64_t a0 = smem_desc_sw128(ring + vs * Sh::kSlotBytes, Sh::kHalfBytes, 1024);
          const uint64_t b0 = smem_desc_sw128(pbuf + (i & 1) * Sh::kPBytes, 16, 1024);
#pragma unroll
          for (int ks = 0; ks < Sh::kSpan / 16; ++ks)
            tc_mma_f16(tO, a0 + (uint64_t)((ks * 2048) >> 4),
                       b0 + (uint64_t)(((ks / 4) * 2048 + (ks % 4) * 32) >> 4), Sh::kIdescPV,
                       (i > 0 || ks > 0) ? 1u : 0u);
          tc_commit(empty(vs));
          tc_commit(pv_done(i & 1));
          last_bar = pv_done(i & 1);
          last_phase = (i >> 1) & 1;
          ++next_pv;
          progressed = true;
        }
        const int j = next_s;
        const int ks_slot = slot_of(kload(j));
        if (j < n_spans && j <= next_pv + 2 && mbar_test(full(ks_slot), use_of(kload(j)) & 1) &&
            (j < 2 || mbar_test(s_free(j & 1), ((j - 2) >> 1) & 1))) {
          tc_fence_after();
          const uint64_t a0 = smem_desc_sw128(ring + ks_slot * Sh::kSlotBytes, 16, 1024);
          const uint64_t b0 = smem_desc_sw128(qbuf, 16, 1024);
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks) {
            const int h = ks / 4, w4 = ks % 4;
            tc_mma_f16(tS + (j & 1) * 16, a0 + (uint64_t)((h * Sh::kHalfBytes + w4 * 32) >> 4),
                       b0 + (uint64_t)((h * (16 * 128) + w4 * 32) >> 4), Sh::kIdescS, ks > 0);
          }
          tc_commit(empty(ks_slot));
          tc_commit(s_ready(j & 1));
          last_bar = s_ready(j & 1);
          last_phase = (j >> 1) & 1;
          ++next_s;
          progressed = true;
        }
        if (progressed) {
          idle = 0;
        } else {
          if (aborted()) break;
          if (PKV_TC_POLL_NS) __nanosleep(PKV_TC_POLL_NS);
          // the clock is read once every 64 idle polls (it is slow to read)
          if ((++idle & 63) == 0) {
            const uint64_t t = global_timer_ns();
            if (idle == 64) {
              t_last = t;
            } else if (t - t_last > kWaitLimitNs) {
              abort_now();
              break;
            }
          }
        }
      }
      // every issued product completes before tensor memory is freed
      if (last_bar) (void)mbar_wait_bounded(last_bar, last_phase, kWaitLimitNs);
    }
  } else {
    // ================= softmax warps 0..3 =================
    // They never leave the span loop early: on an abort they skip the work
    // but still pass every CTA barrier among them, so none of them waits on
    // a barrier another one will not reach.
    const int row = 32 * warp + lane;  // this thread's token in a span (tensor-memory lane)
    // Lazy rescaling: a column's reference maximum moves only when a score
    // exceeds it by more than 2^kLazy, so P stays <= 2^kLazy (exact in f16,
    // and the running sums and O scale together, cancelling in O / l).
    constexpr float kLazy = 8.f;
    float m_run[16], l_part[16];
    int lim[16];  // causal limit of each column (positions below it count)
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      m_run[j] = -CUDART_INF_F;
      l_part[j] = 0.f;
      lim[j] = j < ncols ? pos0 + t0 + j / G + 1 : 0;
    }
    // positions below this count for every column (the first query's limit)
    const int all_see = min(tok_end, pos0 + t0 + 1);
    const float sl2 = p.scale_log2;
    // whether this thread's sub-tile of span i holds data (the copy thread
    // skips, and flags, a sub-tile whose table entry is out of range); the
    // entry is read one span ahead
    auto sub_entry = [&](int i) {
      const int t = i * Sh::kSubs + row / 16;
      return t < n_tiles ? __ldg(table + (sub_begin + t) / SUB) : -1;
    };
    int entry_next = sub_entry(0);
    bool dead = false;
    for (int i = 0; i < n_spans; ++i) {
      const int entry = entry_next;
      if (i + 1 < n_spans) entry_next = sub_entry(i + 1);
      const int b = i & 1;
      dead = dead || aborted();
      uint32_t r[16];
      if (!dead && !wait(s_ready(b), (i >> 1) & 1)) dead = true;
      dead = __any_sync(0xffffffffu, dead);  // warp-uniform before the .sync.aligned loads
      if (!dead) {
        tc_fence_after();
        tmem_ld16(tS + b * 16 + ((uint32_t)(32 * warp) << 16), r);
        tc_fence_before();
      }
      __syncwarp();
      if (!dead && lane == 0) mbar_arrive(s_free(b));
      const int span0 = tok_begin + i * Sh::kSpan;
      const int tok = span0 + row;
      const bool valid = !dead && entry >= 0 && entry < p.num_blocks && tok < tok_end;
      // every position of this warp's 32 counts for every column: no masks
      const bool simple =
          __all_sync(0xffffffffu, valid) && span0 + 32 * warp + 32 <= all_see;
      float d[16];  // log2-domain score minus the column's reference maximum
      bool grow = false;
      if (simple) {
        float mx[4] = {-CUDART_INF_F, -CUDART_INF_F, -CUDART_INF_F, -CUDART_INF_F};
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          d[j] = fmaf(__uint_as_float(r[j]), sl2, -m_run[j]);
          mx[j & 3] = fmaxf(mx[j & 3], d[j]);
        }
        grow = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) > kLazy;
      } else {
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          d[j] = (valid && tok < lim[j]) ? fmaf(__uint_as_float(r[j]), sl2, -m_run[j])
                                         : -CUDART_INF_F;
          grow |= d[j] > kLazy;
        }
      }
      // does any column's reference maximum move?  (CTA-wide, one barrier)
      const int any_grow = __syncthreads_or_among(grow, 128);
      float alpha[16];
      if (any_grow) {
        // the new reference maxima: column maxima of the span's scores
        float x[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const bool ok = simple || (valid && tok < lim[j]);
          x[j] = ok ? __uint_as_float(r[j]) * sl2 : -CUDART_INF_F;
          float mx = x[j];
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
          if (lane == 0) s_red[b][warp][j] = mx;
        }
        named_barrier(1, 128);
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const float sm = fmaxf(fmaxf(s_red[b][0][j], s_red[b][1][j]),
                                 fmaxf(s_red[b][2][j], s_red[b][3][j]));
          alpha[j] = 1.f;
          if (sm > m_run[j] + kLazy || (sm != -CUDART_INF_F && m_run[j] == -CUDART_INF_F)) {
            alpha[j] = m_run[j] == -CUDART_INF_F ? 0.f : ex2_approx(m_run[j] - sm);
            m_run[j] = sm;
          }
          const float mu = m_run[j] == -CUDART_INF_F ? 0.f : m_run[j];
          d[j] = x[j] - mu;
          l_part[j] *= alpha[j];
        }
      }
      // P (f16) and the running sums
      uint32_t ph[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const float p0 = ex2_approx(d[2 * k]), p1 = ex2_approx(d[2 * k + 1]);
        l_part[2 * k] += p0;
        l_part[2 * k + 1] += p1;
        const __half2 h2 = __floats2half2_rn(p0, p1);
        ph[k] = *reinterpret_cast<const uint32_t*>(&h2);
      }
      // P buffer b was read by PV(i-2); O changes only after PV(i-1)
      if (!dead && i >= 2 && !wait(pv_done(b), ((i - 2) >> 1) & 1)) dead = true;
      if (any_grow && i >= 1) {
        if (!dead && !wait(pv_done((i - 1) & 1), ((i - 1) >> 1) & 1)) dead = true;
        dead = __any_sync(0xffffffffu, dead);
        if (!dead) {
          tc_fence_after();
          uint32_t o[16];
          const uint32_t ta = tO + ((uint32_t)(32 * warp) << 16);
          tmem_ld16(ta, o);
#pragma unroll
          for (int j = 0; j < 16; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * alpha[j]);
          tmem_st16(ta, o);
        }
      }
      if (!dead) {
        // P^T as [token half][16 columns][64 tokens], K-major with the swizzle
        const uint32_t pb = pbuf + b * Sh::kPBytes + (row / 64) * 2048;
        const int e = row % 64;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          asm volatile("st.shared.u16 [%0], %1;" ::"r"(pb + sw128_off(2 * k, e)),
                       "h"((unsigned short)(ph[k] & 0xFFFFu))
                       : "memory");
          asm volatile("st.shared.u16 [%0], %1;" ::"r"(pb + sw128_off(2 * k + 1, e)),
                       "h"((unsigned short)(ph[k] >> 16))
                       : "memory");
        }
        if (!simple && !valid) {
          // a V row that does not count: zero it once it has landed (the
          // pool, or what a slot held before, may be NaN there)
          // (V(i)'s slot held K(i), landed: S(i) has run; or, for the last
          // span, V(i - 2), landed: PV(i - 2) completed, waited for above)
          if (wait(full(slot_of(vload(i))), use_of(vload(i)) & 1)) {
            const uint32_t vb = ring + slot_of(vload(i)) * Sh::kSlotBytes + row * 128;
#pragma unroll
            for (int h = 0; h < Sh::kHalves; ++h)
#pragma unroll
              for (int c = 0; c < 8; ++c)
                asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(
                                 vb + h * Sh::kHalfBytes + c * 16),
                             "r"(0)
                             : "memory");
          }
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (!dead && lane == 0) mbar_arrive(p_ready(b));
    }
    // ---- the result: O^T rows d = 32 warp + lane, column sums, output
    const int last = n_spans - 1;
    if (!dead && !wait(pv_done(last & 1), (last >> 1) & 1)) dead = true;
    dead = __any_sync(0xffffffffu, dead);
    uint32_t o[16];
    if (!dead) {
      tc_fence_after();
      tmem_ld16(tO + ((uint32_t)(32 * warp) << 16), o);
    }
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      float sum = l_part[j];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
      if (lane == 0) s_sum[warp][j] = sum;
    }
    named_barrier(1, 128);
    if (!aborted()) {
      const int dd = 32 * warp + lane;
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        if (j >= ncols) continue;
        const float den = s_sum[0][j] + s_sum[1][j] + s_sum[2][j] + s_sum[3][j];
        const float num = __uint_as_float(o[j]);
        const size_t qrow = (size_t)(q_begin + t0 + j / G) * p.num_heads + (size_t)g * G + j % G;
        if (SPLIT) {
          const size_t slot = qrow * p.num_splits + split;
          p.part_out[slot * D + dd] = num;
          if (dd == 0) {
            p.part_m[slot] = m_run[j];
            p.part_l[slot] = den;
          }
        } else {
          p.out[qrow * D + dd] = __float2half_rn(den > 0.f ? num / den : 0.f);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tbase, Sh::kTmemCols);
}

}  // namespace pkv
