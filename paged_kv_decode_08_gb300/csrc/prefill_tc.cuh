// paged_prefill_tc_kernel: many causal queries per sequence over the paged
// cache (chunked prefill: the varlen attention of kernels.cuh once a
// sequence brings at least 128 (query, head) rows), with both products on
// the 5th-generation tensor cores, head_dim 128.
//
// One CTA per (sequence, KV head, pair of query tiles).  A tile holds
// Q_T = 128 / G queries: its 128 rows r = (query r / G, head r % G) (rows
// past the tile's queries hold zero queries) are the M of both products of
// every span of 128 context tokens:
//
//   S_X[128 rows x 128 tok] = Q_X [128 x 128 d] . K_span^T     (K-major A and B)
//   O_X[128 rows x 128 d]  += P_X [128 x 128 tok] . V_span     (K-major A, MN-major B)
//
// for tiles X = A, B.  The two tiles share each K/V span, so a span's bytes
// feed twice the products of one tile, and the tiles take turns on the
// tensor cores: while one tile's softmax runs, the other's products do.
// Tensor memory holds S and O of each tile (4 x 128 columns); shared memory
// the ring, Q and P of each tile (225 KB).
//
// Warp roles (416 threads).  Warps 9-12 copy K and V into a ring of three
// 32 KB slots in the order K0, K1, V0, K2, V1, ... (16-row sub-tiles, one TMA
// box per 64-element half, each warp issuing its share of a load's 16 boxes,
// one per lane: a warp issues boxes at a bounded rate).  Warp 8 (one lane)
// issues each product once its inputs are ready.  Warps 0-3 run the online
// softmax of tile A and warps 4-7 that of tile B, one thread per row
// (tensor-memory lane r), over the span in two chunks of 64 tokens: the
// thread loads a chunk of its row of S, keeps the row's reference maximum,
// which moves only when a score exceeds it by 2^8 (then the row of O, and
// the first chunk's P when the second chunk moves it, are rescaled), writes
// the chunk of its row of P (f16) to shared memory as the K-major A operand
// of the second product, and adds the exponentials to the row's sum.  Positions past a query's causal limit get
// P = 0; V rows of positions that count for no row (past the pair's last
// query, or in a sub-tile whose table entry is out of range) are zeroed
// before PV, since 0 x NaN would poison it.
//
// Every wait is bounded; a wait that runs out sets PKV_DEV_WAIT_TIMEOUT and
// the CTA stops, lets its copies and MMAs drain (bounded as well), writes
// nothing and frees its tensor memory.
#pragma once

#include "varlen_tc.cuh"

// Warps that issue the copies (each takes 16 / n of a load's boxes).
#ifndef PKV_PREFILL_COPY_WARPS
#define PKV_PREFILL_COPY_WARPS 4
#endif

namespace pkv {

struct TcPrefillShape {
  static constexpr int D = 128;
  static constexpr int kTiles = 2;                    // query tiles per CTA
  static constexpr int kRows = 128;                   // (query, head) rows per tile: M
  static constexpr int kSpan = 128;                   // context tokens per span: N of S
  static constexpr int kSubs = kSpan / 16;            // 16-row sub-tiles per span
  static constexpr int kHalfBytes = kSpan * 128;      // a 64-element half of K or V: 16 KB
  static constexpr int kSlotBytes = 2 * kHalfBytes;   // K (or V) of a span: 32 KB
  static constexpr int kSlots = 3;
  static constexpr int kRingBytes = kSlots * kSlotBytes;  // 96 KB
  static constexpr int kQBytes = 2 * kRows * 128;         // Q_X [d halves][128 rows][64]: 32 KB
  static constexpr int kPBytes = 2 * kRows * 128;  // P_X [token halves][128 rows][64]: 32 KB
  static constexpr int kQOff = kRingBytes;
  static constexpr int kPOff = kQOff + kTiles * kQBytes;  // P [tile]
  static constexpr int kBarOff = kPOff + kTiles * kPBytes;
  // full[3], empty[3], then per tile s_ready, s_free, p_ready, pv_done
  static constexpr int kNumBars = 6 + kTiles * 4;
  static constexpr int kSmemBytes = 1024 + kBarOff + kNumBars * 8;  // ~225 KB: one CTA per SM
  static constexpr int kTmemCols = 512;  // S [tile] (128 columns each), O [tile] (128)
  static constexpr int kSoftWarps = 4 * kTiles;  // one thread per row of each tile
  static constexpr int kMmaWarp = kSoftWarps;
  static constexpr int kCopyWarps = PKV_PREFILL_COPY_WARPS;  // warps kMmaWarp + 1 ..
  static constexpr int kBoxesPerWarp = 2 * kSubs / kCopyWarps;
  static_assert(kBoxesPerWarp >= 1 && kBoxesPerWarp * kCopyWarps == 2 * kSubs,
                "the copy warps share a load's boxes evenly");
  static constexpr int kThreads = (kMmaWarp + 1 + kCopyWarps) * 32;
  static constexpr uint32_t kIdescS = mma_idesc_f16(kRows, kSpan, false, false);
  static constexpr uint32_t kIdescPV = mma_idesc_f16(kRows, D, false, true);
};

template <int BS, bool SPLIT>
__global__ void __launch_bounds__(TcPrefillShape::kThreads, 1)
paged_prefill_tc_kernel(const __grid_constant__ CUtensorMap kmap,
                        const __grid_constant__ CUtensorMap vmap, const VarlenParams p) {
  using Sh = TcPrefillShape;
  constexpr int SUB = BS / 16;  // 16-row sub-tiles per pool block
  extern __shared__ uint8_t smem_raw[];
  __shared__ int s_abort;
  __shared__ uint32_t s_tmem;
  __shared__ int s_max[Sh::kThreads / 32];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t ring = smem_addr(smem);
  const uint32_t qbuf = ring + Sh::kQOff;
  const uint32_t pbuf = ring + Sh::kPOff;
  const uint32_t bars = ring + Sh::kBarOff;
  auto full = [&](int i) { return bars + 8 * i; };
  auto empty = [&](int i) { return bars + 8 * (3 + i); };
  // per tile X: one phase per span
  auto s_ready = [&](int X) { return bars + 8 * (6 + 4 * X); };
  auto s_free = [&](int X) { return bars + 8 * (7 + 4 * X); };
  auto p_ready = [&](int X) { return bars + 8 * (8 + 4 * X); };
  auto pv_done = [&](int X) { return bars + 8 * (9 + 4 * X); };
  // Ring loads in issue order: K0, then K(i+1), V(i) for each span i, V of
  // the last span last; load n goes to slot n % 3, its (n / 3)-th use.
  auto slot_of = [](int n) { return n % Sh::kSlots; };
  auto use_of = [](int n) { return (uint32_t)(n / Sh::kSlots); };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // the pair index is the slowest and runs backwards: the pairs with the
  // most positions (the latest queries) start first, the short ones last;
  // the split (split-K) is the fastest
  const int nsplit = SPLIT ? p.num_splits : 1;
  const int per_pair = gridDim.x / (p.num_chunks * nsplit);  // sequences x KV heads
  const int split = SPLIT ? (int)blockIdx.x % nsplit : 0;
  const int idx = (int)blockIdx.x / nsplit;
  const int qt = p.num_chunks - 1 - idx / per_pair;
  const int item = idx % per_pair;
  const int g = item % p.num_kv_heads;
  const int s = item / p.num_kv_heads;
  const int G = p.group;
  const int QT = p.qc / Sh::kTiles;  // queries per tile (128 / G)

  pdl_launch_dependents();
  if (threadIdx.x == 0) s_abort = 0;
  if (warp == Sh::kMmaWarp && lane == 0) {
#pragma unroll
    for (int i = 0; i < 3; ++i) {
      mbar_init(full(i), Sh::kCopyWarps);  // one arrival (with its bytes) per copy warp
      mbar_init(empty(i), 1);
    }
#pragma unroll
    for (int X = 0; X < Sh::kTiles; ++X) {
      mbar_init(s_ready(X), 1);
      mbar_init(s_free(X), 4);
      mbar_init(p_ready(X), 4);
      mbar_init(pv_done(X), 1);
    }
    fence_mbar_init();
  }
  pdl_wait();

  // ---- the queries of the pair and the positions they read (as paged_varlen_kernel)
  const unsigned int status = *reinterpret_cast<volatile unsigned int*>(&g_device_status);
  const int cap = p.max_blocks_per_seq * BS;
  const int q_begin = __ldg(p.cu_seqlens_q + s);
  const int q_end = __ldg(p.cu_seqlens_q + s + 1);
  int pos0 = __ldg(p.pos_offsets + s);
  if (SPLIT) {
    // the longest context of the call, in blocks: the split chunks are cut
    // from it (as the varlen split kernels cut theirs)
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
    for (int w = 0; w < Sh::kThreads / 32; ++w) nblk_max = max(nblk_max, s_max[w]);
  }
  const int chunk = SPLIT ? max(p.min_chunk_blocks, (nblk_max + nsplit - 1) / nsplit) : 0;
  if (q_begin < 0 || q_end < q_begin || q_end > p.total_q) {
    if (threadIdx.x == 0) atomicOr(&g_device_status, kDevBadContextLen);
    return;
  }
  const int q_len = q_end - q_begin;
  if (qt == p.num_chunks - 1 && q_len > p.num_chunks * p.qc && threadIdx.x == 0)
    atomicOr(&g_device_status, kDevBadContextLen);
  const int t0 = qt * p.qc;
  if (t0 >= q_len) return;
  const int nq = min(p.qc, q_len - t0);
  if (pos0 < 0 || pos0 + q_len > cap) {
    if (threadIdx.x == 0) atomicOr(&g_device_status, kDevBadContextLen);
    pos0 = pos0 < 0 ? 0 : max(0, cap - q_len);
  }
  // >= 1: the pair's last query's limit
  const int chunk_end = min(cap, pos0 + t0 + nq);
  // this CTA's positions: [tok_begin, tok_end) (all of them in one pass)
  int tok_begin = 0, tok_end = chunk_end;
  if (SPLIT) {
    if ((long long)split * chunk * BS >= chunk_end) {
      // the split holds none of the pair's positions: maximum -inf and sum 0
      // for its rows (the combine gives them weight 0)
      for (int n = threadIdx.x; n < nq * G; n += Sh::kThreads) {
        const size_t row = (size_t)(q_begin + t0 + n / G) * p.num_heads + (size_t)g * G + n % G;
        p.part_m[row * nsplit + split] = -CUDART_INF_F;
        p.part_l[row * nsplit + split] = 0.f;
      }
      return;
    }
    tok_begin = split * chunk * BS;
    tok_end = (int)min((long long)chunk_end, (long long)tok_begin + (long long)chunk * BS);
  }
  const int sub_begin = tok_begin / 16;  // 16-row sub-tile of the first position
  const int n_tiles = (tok_end - tok_begin + 15) / 16;
  const int n_spans = (n_tiles + Sh::kSubs - 1) / Sh::kSubs;  // >= 1
  // tile B holds queries only when the pair has more than Q_T of them
  const int ntile = nq > QT ? 2 : 1;
  const int32_t* table = p.block_tables + (size_t)s * p.max_blocks_per_seq;
  auto kload = [&](int j) { return j == 0 ? 0 : 2 * j - 1; };                        // K(j)'s load
  auto vload = [&](int i) { return i == n_spans - 1 ? 2 * n_spans - 1 : 2 * i + 2; };  // V(i)'s

  // ---- set-up: tensor memory, the queries as the A operand of S
  if (warp == 0) tmem_alloc(smem_addr(&s_tmem), Sh::kTmemCols);
  if (warp < Sh::kSoftWarps) {
    // thread = (tile X, row r): query t0 + X Q_T + r / G, head g G + r % G
    // (zeros past the tile's rows), 16 chunks of 16 bytes into
    // [d halves][128 rows][64] with the swizzle
    const int X = threadIdx.x / Sh::kRows, r = threadIdx.x % Sh::kRows;
    const int nrows = max(0, min(QT, nq - X * QT)) * G;
    const bool live = r < nrows;
    const size_t row = (size_t)(q_begin + t0 + X * QT + (live ? r / G : 0)) * p.num_heads +
                       (size_t)g * G + (live ? r % G : 0);
    const uint4* src = reinterpret_cast<const uint4*>(p.q + row * Sh::D);
    const uint32_t qx = qbuf + X * Sh::kQBytes;
#pragma unroll
    for (int c = 0; c < 16; ++c) {
      const uint4 v = live ? __ldg(src + c) : make_uint4(0u, 0u, 0u, 0u);
      const uint32_t dst = qx + (c / 8) * (Sh::kRows * 128) + sw128_off(r, (c % 8) * 8);
      asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(dst), "r"(v.x), "r"(v.y),
                   "r"(v.z), "r"(v.w)
                   : "memory");
    }
    fence_proxy_async_smem();
  }
  // whether any table entry the pair reads is out of range (the copies skip
  // such sub-tiles; the softmax then masks them span by span)
  bool bad_entry = false;
  for (int t = sub_begin / SUB + threadIdx.x; t * SUB < sub_begin + n_tiles; t += Sh::kThreads) {
    const int e = __ldg(table + t);
    bad_entry = bad_entry || e < 0 || e >= p.num_blocks;
  }
  tc_fence_before();
  const bool any_bad = __syncthreads_or(bad_entry);
  tc_fence_after();
  const uint32_t tbase = s_tmem;
  auto tS = [&](int X) { return tbase + (uint32_t)(X * 128); };
  auto tO = [&](int X) { return tbase + 256u + (uint32_t)(X * 128); };

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
    // ================= copies (warps 9 ..) =================
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
        if (use >= 1 && !mbar_wait_bounded(empty(slot), (use - 1) & 1, kWaitLimitNs)) {
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
    // ================= MMAs (warp 8, lane 0) =================
    if (lane == 0) {
      uint32_t last_bar = 0, last_phase = 0;  // the last commit (drained before exit)
      // Issue whichever product is ready.  S products go in order S_A(j),
      // S_B(j), S_A(j+1), ...; PV products in order PV_A(i), PV_B(i), ...
      // (the softmax warps rescale O between them).  S_X(j) needs K(j) and
      // S_X(j - 1) read by the softmax warps of tile X; PV_X(i) needs P_X(i)
      // and V(i).
      // A barrier's phase is tested by its parity alone, so a test must not
      // run while the phase two back can still be pending: K(j)'s slot held
      // V(j - 3) (K0 for j = 2), landed once PV(j - 3) was issued (the gate
      // j <= next_pv + 2) or, for K0, before S(0); V(i)'s slot held K(i)
      // (V(i - 2) for the last span), landed before S(i) (or PV(i - 2)) was
      // issued, and V(i) is tested only once P_A(i) is ready (after S(i));
      // s_free, p_ready: the span before was waited on before the product
      // that followed it.
      int next_s = 0, sx = 0, next_pv = 0, px = 0;
      uint64_t t_last = global_timer_ns();
      int idle = 0;
      while (next_pv < n_spans) {
        bool progressed = false;
        {
          const int i = next_pv, X = px;
          const int vs = slot_of(vload(i));
          if (mbar_test(p_ready(X), i & 1) &&
              (X > 0 || mbar_test(full(vs), use_of(vload(i)) & 1))) {
            tc_fence_after();
            // P: K-major over the span's tokens; V: MN-major (d contiguous),
            // its two d halves kHalfBytes apart, 8-token groups 1 KB apart.
            // A descriptor's address field is the byte address / 16, so a
            // step within the operand adds its offset / 16.
            const uint64_t a0 = smem_desc_sw128(pbuf + X * Sh::kPBytes, 16, 1024);
            const uint64_t b0 = smem_desc_sw128(ring + vs * Sh::kSlotBytes, Sh::kHalfBytes, 1024);
#pragma unroll
            for (int ks = 0; ks < Sh::kSpan / 16; ++ks)
              tc_mma_f16(tO(X), a0 + (uint64_t)(((ks / 4) * (Sh::kRows * 128) + (ks % 4) * 32) >> 4),
                         b0 + (uint64_t)((ks * 2048) >> 4), Sh::kIdescPV,
                         (i > 0 || ks > 0) ? 1u : 0u);
            tc_commit(pv_done(X));
            last_bar = pv_done(X);
            last_phase = i & 1;
            if (X + 1 == ntile) {
              tc_commit(empty(vs));
              ++next_pv;
              px = 0;
            } else {
              ++px;
            }
            progressed = true;
          }
        }
        {
          const int j = next_s, X = sx;
          const int ks_slot = slot_of(kload(j));
          if (j < n_spans && j <= next_pv + 2 &&
              (X > 0 || mbar_test(full(ks_slot), use_of(kload(j)) & 1)) &&
              (j < 1 || mbar_test(s_free(X), (j - 1) & 1))) {
            tc_fence_after();
            const uint64_t a0 = smem_desc_sw128(qbuf + X * Sh::kQBytes, 16, 1024);
            const uint64_t b0 = smem_desc_sw128(ring + ks_slot * Sh::kSlotBytes, 16, 1024);
#pragma unroll
            for (int ks = 0; ks < Sh::D / 16; ++ks) {
              const int h = ks / 4, w4 = ks % 4;
              tc_mma_f16(tS(X), a0 + (uint64_t)((h * (Sh::kRows * 128) + w4 * 32) >> 4),
                         b0 + (uint64_t)((h * Sh::kHalfBytes + w4 * 32) >> 4), Sh::kIdescS, ks > 0);
            }
            tc_commit(s_ready(X));
            last_bar = s_ready(X);
            last_phase = j & 1;
            if (X + 1 == ntile) {
              tc_commit(empty(ks_slot));
              ++next_s;
              sx = 0;
            } else {
              ++sx;
            }
            progressed = true;
          }
        }
        if (progressed) {
          idle = 0;
        } else {
          if (aborted()) break;
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
  } else if (warp < Sh::kSoftWarps && (warp >> 2) < ntile) {
    // ============ softmax warps: tile X = warp / 4, one thread per row ============
    // Every wait is bounded; on an abort a warp skips the work but still
    // walks its spans (no barrier among the softmax warps depends on it).
    const int X = warp >> 2;
    const int r = 32 * (warp & 3) + lane;  // this thread's row (tensor-memory lane)
    const int nrows = max(0, min(QT, nq - X * QT)) * G;
    const bool live = r < nrows;
    const int qx0 = t0 + X * QT;  // the tile's first query
    // positions below it count: the row's causal limit, clipped to this
    // CTA's range (a split's last span may run past it into the next split,
    // whose positions were not loaded)
    const int lim = live ? min(pos0 + qx0 + r / G + 1, tok_end) : 0;
    // positions below this count for every row of the tile (its first query's limit)
    const int all_see = min(tok_end, pos0 + qx0 + 1);
    const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
    // Lazy rescaling: the row's reference maximum moves only when a score
    // exceeds it by more than 2^kLazy, so P stays <= 2^kLazy (exact in f16,
    // and the running sum and O scale together, cancelling in O / l).
    constexpr float kLazy = 8.f;
    constexpr uint32_t kAllOk = (1u << Sh::kSubs) - 1;
    const float sl2 = p.scale_log2;
    float m_run = -CUDART_INF_F, l_run = 0.f;
    // which sub-tiles of span i hold data (bit u; the copy warps skip, and
    // flag, a sub-tile whose table entry is out of range), read a span ahead
    // when the pair reads any such entry (else every sub-tile holds data;
    // those past the last position are masked by the causal limit)
    auto span_ok = [&](int i) {
      uint32_t bits = 0;
#pragma unroll
      for (int u = 0; u < Sh::kSubs; ++u) {
        const int t = i * Sh::kSubs + u;
        const int e = t < n_tiles ? __ldg(table + (sub_begin + t) / SUB) : -1;
        if (e >= 0 && e < p.num_blocks) bits |= 1u << u;
      }
      return bits;
    };
    uint32_t ok_next = any_bad ? span_ok(0) : kAllOk;
    bool dead = false;
    // O is rescaled (rows of this warp that moved their reference) once
    // PV_X(i-1) completed (waited before the first chunk's P is written)
    auto rescale_o = [&](float alpha) {
      tc_fence_after();
#pragma unroll 1
      for (int c = 0; c < Sh::D / 16; ++c) {
        uint32_t o[16];
        const uint32_t ta = tO(X) + c * 16 + lane_base;
        tmem_ld16(ta, o);
#pragma unroll
        for (int k = 0; k < 16; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * alpha);
        tmem_st16(ta, o);
      }
    };
    for (int i = 0; i < n_spans; ++i) {
      const uint32_t okb = ok_next;
      if (any_bad && i + 1 < n_spans) ok_next = span_ok(i + 1);
      dead = dead || aborted();
      if (!dead && !wait(s_ready(X), i & 1)) dead = true;
      dead = __any_sync(0xffffffffu, dead);  // warp-uniform before the .sync.aligned loads
      const int span0 = tok_begin + i * Sh::kSpan;  // the span's first position
      // every position of the span counts for every row of the tile: no masks
      const bool simple = okb == kAllOk && span0 + Sh::kSpan <= all_see;
      // The scores are taken in two chunks of 64 tokens.  Each chunk's
      // maximum (log2 domain) may move the row's reference; P of a chunk is
      // written against the reference at that time, so when the second
      // chunk moves it the first chunk's P is rescaled in shared memory.
      // With no masks and a positive scale the scores stay raw (scaling by a
      // positive factor keeps their order, so the scaled maximum is the raw
      // one scaled) and each exponent is fma(s, scale log2 e, -mu); else
      // they are scaled (and masked) in place.  Four independent
      // three-input max chains; four independent partial sums.
      const bool raw = simple && sl2 > 0.f;
      const float mul = raw ? sl2 : 1.f;
      const uint32_t pb = pbuf + X * Sh::kPBytes;
#pragma unroll 1
      for (int ch = 0; ch < 2; ++ch) {
        uint32_t ra[64];  // this row's scores, tokens 64 ch .. 64 ch + 63 of the span
        dead = __any_sync(0xffffffffu, dead);  // warp-uniform before the .sync.aligned loads
        if (!dead) {
          tc_fence_after();
          tmem_ld64(tS(X) + ch * 64 + lane_base, ra);
          tc_fence_before();
        } else {
#pragma unroll
          for (int j = 0; j < 64; ++j) ra[j] = 0u;
        }
        if (ch == 1) {
          // S_X(i) is read: the next span's scores may go in
          __syncwarp();
          if (!dead && lane == 0) mbar_arrive(s_free(X));
        }
        const int tok0 = span0 + ch * 64;
        float m4[4] = {-CUDART_INF_F, -CUDART_INF_F, -CUDART_INF_F, -CUDART_INF_F};
        if (raw) {
#pragma unroll
          for (int j = 0; j < 64; j += 2)
            m4[(j >> 1) & 3] = fmax3(m4[(j >> 1) & 3], __uint_as_float(ra[j]),
                                     __uint_as_float(ra[j + 1]));
        } else if (simple) {
#pragma unroll
          for (int j = 0; j < 64; j += 2) {
            const float x0 = __uint_as_float(ra[j]) * sl2, x1 = __uint_as_float(ra[j + 1]) * sl2;
            ra[j] = __float_as_uint(x0);
            ra[j + 1] = __float_as_uint(x1);
            m4[(j >> 1) & 3] = fmax3(m4[(j >> 1) & 3], x0, x1);
          }
        } else {
#pragma unroll
          for (int j = 0; j < 64; j += 2) {
            float x[2];
#pragma unroll
            for (int k = 0; k < 2; ++k) {
              const bool ok = ((okb >> ((ch * 64 + j + k) >> 4)) & 1u) && tok0 + j + k < lim;
              x[k] = ok ? __uint_as_float(ra[j + k]) * sl2 : -CUDART_INF_F;
              ra[j + k] = __float_as_uint(x[k]);
            }
            m4[(j >> 1) & 3] = fmax3(m4[(j >> 1) & 3], x[0], x[1]);
          }
        }
        float mx = fmaxf(fmax3(m4[0], m4[1], m4[2]), m4[3]);
        if (raw) mx *= sl2;
        const bool grow =
            mx > m_run + kLazy || (m_run == -CUDART_INF_F && mx != -CUDART_INF_F);
        float alpha = 1.f;
        if (grow) {
          alpha = m_run == -CUDART_INF_F ? 0.f : ex2_approx(m_run - mx);
          m_run = mx;
          l_run *= alpha;
        }
        const float mu = m_run == -CUDART_INF_F ? 0.f : m_run;
        // P_X and O_X were last read by PV_X(i-1)
        if (ch == 0 && !dead && i >= 1 && !wait(pv_done(X), (i - 1) & 1)) dead = true;
        if (__any_sync(0xffffffffu, grow)) {
          dead = __any_sync(0xffffffffu, dead);
          if (!dead && i >= 1) rescale_o(alpha);  // O holds products from span 1 on
          if (!dead && ch == 1 && grow) {
            // the first chunk's P was written against the old reference
#pragma unroll
            for (int c = 0; c < 8; ++c) {
              const uint32_t a = pb + sw128_off(r, c * 8);
              uint32_t w[4];
              asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                           : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3])
                           : "r"(a)
                           : "memory");
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[e]));
                const __half2 h2 = __floats2half2_rn(f.x * alpha, f.y * alpha);
                w[e] = *reinterpret_cast<const uint32_t*>(&h2);
              }
              asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(w[0]),
                           "r"(w[1]), "r"(w[2]), "r"(w[3])
                           : "memory");
            }
          }
        }
        if (!dead) {
          // this chunk of the row of P (f16), [token half ch][128 rows][64],
          // K-major with the swizzle; the running sum adds the same exponentials
          const uint32_t pc = pb + ch * (Sh::kRows * 128);
          float l4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int j = c * 8 + 2 * e;
              const float p0 = ex2_approx(fmaf(__uint_as_float(ra[j]), mul, -mu));
              const float p1 = ex2_approx(fmaf(__uint_as_float(ra[j + 1]), mul, -mu));
              l4[e] += p0 + p1;
              const __half2 h2 = __floats2half2_rn(p0, p1);
              w[e] = *reinterpret_cast<const uint32_t*>(&h2);
            }
            asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(pc + sw128_off(r, c * 8)),
                         "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3])
                         : "memory");
          }
          l_run += (l4[0] + l4[1]) + (l4[2] + l4[3]);
        }
      }
      // V row r of the span (tile A's threads): zero it when its position
      // counts for no row of the pair (past the pair's last query, or in a
      // sub-tile with no data) once it has landed.  PV_B(i) is issued after
      // PV_A(i), so after this.  V(i)'s slot held K(i) (V(i - 2) for the last
      // span), landed before S(i) (or PV(i - 2), completed: PV_A(i-1) was
      // waited above).  Tile A's simple spans hold no such position.
      const int tok = span0 + r;
      if (!dead && X == 0 && !simple && (!((okb >> (r >> 4)) & 1u) || tok >= tok_end)) {
        if (wait(full(slot_of(vload(i))), use_of(vload(i)) & 1)) {
          const uint32_t vb = ring + slot_of(vload(i)) * Sh::kSlotBytes + r * 128;
#pragma unroll
          for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int c = 0; c < 8; ++c)
              asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(
                               vb + h * Sh::kHalfBytes + c * 16),
                           "r"(0)
                           : "memory");
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (!dead && lane == 0) mbar_arrive(p_ready(X));
    }
    // ---- the result: the row of O over the row's sum
    const int last = n_spans - 1;
    if (!dead && !wait(pv_done(X), last & 1)) dead = true;
    dead = __any_sync(0xffffffffu, dead);
    const bool write = !dead && !aborted();
    if (__any_sync(0xffffffffu, write)) {
      tc_fence_after();
      const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
      const size_t orow = (size_t)(q_begin + qx0 + (live ? r / G : 0)) * p.num_heads +
                          (size_t)g * G + (live ? r % G : 0);
      // split-K: the unnormalised row of O, the reference maximum and the
      // sum, for the combine; else the row of O over its sum (f16)
      const size_t slot = orow * nsplit + split;
#pragma unroll 1
      for (int hf = 0; hf < 2; ++hf) {
        uint32_t o[64];
        __syncwarp();  // converged for the .sync.aligned load
        tmem_ld64(tO(X) + hf * 64 + lane_base, o);
        if (!(write && live)) {
        } else if (SPLIT) {
          float4* po = reinterpret_cast<float4*>(p.part_out + slot * Sh::D) + hf * 16;
#pragma unroll
          for (int c = 0; c < 16; ++c)
            po[c] = make_float4(__uint_as_float(o[4 * c]), __uint_as_float(o[4 * c + 1]),
                                __uint_as_float(o[4 * c + 2]), __uint_as_float(o[4 * c + 3]));
        } else {
          uint4* dst = reinterpret_cast<uint4*>(p.out + orow * Sh::D) + hf * 8;
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const __half2 h2 = __floats2half2_rn(__uint_as_float(o[c * 8 + 2 * e]) * inv,
                                                   __uint_as_float(o[c * 8 + 2 * e + 1]) * inv);
              w[e] = *reinterpret_cast<const uint32_t*>(&h2);
            }
            dst[c] = make_uint4(w[0], w[1], w[2], w[3]);
          }
        }
      }
      if (SPLIT && write && live) {
        p.part_m[slot] = m_run;
        p.part_l[slot] = l_run;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tbase, Sh::kTmemCols);
}

}  // namespace pkv
