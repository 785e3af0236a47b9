// paged_prefill_tc_kernel: many causal queries per sequence over the paged
// cache (chunked prefill: the varlen attention of kernels.cuh once a
// sequence brings at least 128 (query, head) rows), with both products on
// the 5th-generation tensor cores, head_dim 128.
//
// One CTA per (sequence, KV head, tile of Q_T = 128 / G queries); its 128
// rows r = (query r / G, head r % G) (rows past the tile's queries hold zero
// queries) are the M of both MMAs per span of 128 context tokens:
//
//   S[128 rows x 128 tok] = Q [128 x 128 d] . K_span^T       (K-major A and B)
//   O[128 rows x 128 d]  += P [128 x 128 tok] . V_span        (K-major A, MN-major B)
//
// both accumulated in tensor memory (S double-buffered, 2 x 128 columns; O
// 128 columns).  Warps 9 .. copy K and V as the tcgen05 varlen kernel does
// (16-row sub-tiles, one TMA box per 64-element half, a ring of three 32 KB
// slots in the order K0, K1, V0, K2, V1, ...), each warp issuing its share
// of a load's 16 boxes, one per lane.  Warp 8 (one lane) issues each
// product once its inputs are ready.  Warps 0-7 run the
// online softmax with two threads per row (tensor-memory lane r = row r;
// warps w and w + 4 share a lane quarter and take one half of the span's
// tokens each): a thread loads its half of the row of S, the two halves
// exchange their maxima through shared memory, and each keeps the row's
// reference maximum, which moves only when a score exceeds it by 2^8 (then
// its half of the row of O is rescaled in tensor memory), writes its half of
// the row of P (f16) to shared memory as the K-major A operand of the second
// product, and adds the exponentials to its share of the row's sum.  Positions
// past a query's causal limit get P = 0; V rows of positions that count for
// no row (past the tile's last query, or in a sub-tile whose table entry is
// out of range) are zeroed before PV, since 0 x NaN would poison it.
//
// Every wait is bounded; a wait that runs out sets PKV_DEV_WAIT_TIMEOUT and
// the CTA stops, lets its copies and MMAs drain (bounded as well), writes
// nothing and frees its tensor memory.
#pragma once

#include "varlen_tc.cuh"

// Warps that issue the copies (each takes 16 / n of a load's boxes): a warp
// issues TMA boxes at a bounded rate, so the copies of one CTA go faster
// when several warps share them.
#ifndef PKV_PREFILL_COPY_WARPS
#define PKV_PREFILL_COPY_WARPS 4
#endif

// Sleep (ns) between idle polls of the MMA thread (0: spin); it shares a
// warp scheduler with two softmax warps.
#ifndef PKV_PREFILL_MMA_POLL_NS
#define PKV_PREFILL_MMA_POLL_NS 0
#endif

namespace pkv {

struct TcPrefillShape {
  static constexpr int D = 128;
  static constexpr int kRows = 128;                   // (query, head) rows per tile: M
  static constexpr int kSpan = 128;                   // context tokens per span: N of S
  static constexpr int kSubs = kSpan / 16;            // 16-row sub-tiles per span
  static constexpr int kHalfBytes = kSpan * 128;      // a 64-element half of K or V: 16 KB
  static constexpr int kSlotBytes = 2 * kHalfBytes;   // K (or V) of a span: 32 KB
  static constexpr int kSlots = 3;
  static constexpr int kRingBytes = kSlots * kSlotBytes;  // 96 KB
  static constexpr int kQBytes = 2 * kRows * 128;         // Q [d halves][128 rows][64]: 32 KB
  static constexpr int kPBytes = 2 * kRows * 128;         // P [token halves][128 rows][64]
  static constexpr int kQOff = kRingBytes;
  static constexpr int kPOff = kQOff + kQBytes;           // two P buffers
  static constexpr int kBarOff = kPOff + 2 * kPBytes;
  // full[3], empty[3], s_ready[2], s_free[2], p_ready[2], pv_done[2]
  static constexpr int kNumBars = 14;
  static constexpr int kSmemBytes = 1024 + kBarOff + kNumBars * 8;  // ~193 KB: one CTA per SM
  static constexpr int kTmemCols = 512;  // S[2] (128 columns each), O (128)
  static constexpr int kSoftWarps = 8;   // two per tensor-memory lane quarter
  static constexpr int kMmaWarp = 8;
  static constexpr int kCopyWarps = PKV_PREFILL_COPY_WARPS;  // warps 9 ..
  static constexpr int kBoxesPerWarp = 2 * kSubs / kCopyWarps;
  static_assert(kBoxesPerWarp % 2 == 0 && kBoxesPerWarp * kCopyWarps == 2 * kSubs,
                "each copy warp takes whole sub-tiles");
  static constexpr int kThreads = (kMmaWarp + 1 + kCopyWarps) * 32;
  static constexpr uint32_t kIdescS = mma_idesc_f16(128, 128, false, false);
  static constexpr uint32_t kIdescPV = mma_idesc_f16(128, 128, false, true);
};

template <int BS>
__global__ void __launch_bounds__(TcPrefillShape::kThreads, 1)
paged_prefill_tc_kernel(const __grid_constant__ CUtensorMap kmap,
                        const __grid_constant__ CUtensorMap vmap, const VarlenParams p) {
  using Sh = TcPrefillShape;
  constexpr int SUB = BS / 16;  // 16-row sub-tiles per pool block
  extern __shared__ uint8_t smem_raw[];
  __shared__ int s_abort;
  __shared__ uint32_t s_tmem;
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

  // the tile index is the slowest and runs backwards: the tiles with the
  // most positions (the latest queries) start first, the short ones last
  const int per_tile = gridDim.x / p.num_chunks;  // sequences x KV heads
  const int qt = p.num_chunks - 1 - (int)blockIdx.x / per_tile;
  const int item = (int)blockIdx.x % per_tile;
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
      mbar_init(s_free(i), Sh::kSoftWarps);
      mbar_init(p_ready(i), Sh::kSoftWarps);
      mbar_init(pv_done(i), 1);
    }
    fence_mbar_init();
  }
  pdl_wait();

  // ---- the tile of queries and the positions it reads (as paged_varlen_kernel)
  const unsigned int status = *reinterpret_cast<volatile unsigned int*>(&g_device_status);
  const int cap = p.max_blocks_per_seq * BS;
  const int q_begin = __ldg(p.cu_seqlens_q + s);
  const int q_end = __ldg(p.cu_seqlens_q + s + 1);
  int pos0 = __ldg(p.pos_offsets + s);
  if (__syncthreads_or(status & kDevWaitTimeout)) return;
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
  const int tok_end = min(cap, pos0 + t0 + nq);  // >= 1: the last query's limit
  const int nrows = nq * G;                       // <= 128
  const int n_tiles = (tok_end + 15) / 16;
  const int n_spans = (n_tiles + Sh::kSubs - 1) / Sh::kSubs;  // >= 1
  const int32_t* table = p.block_tables + (size_t)s * p.max_blocks_per_seq;
  auto kload = [&](int j) { return j == 0 ? 0 : 2 * j - 1; };                        // K(j)'s load
  auto vload = [&](int i) { return i == n_spans - 1 ? 2 * n_spans - 1 : 2 * i + 2; };  // V(i)'s

  // ---- set-up: tensor memory, the queries as the A operand of S
  if (warp == 0) tmem_alloc(smem_addr(&s_tmem), Sh::kTmemCols);
  if (warp < 4) {
    // row r = threadIdx.x (warps 0-3): query t0 + r / G, head g G + r % G (zeros past nrows),
    // 16 chunks of 16 bytes into [d halves][128 rows][64] with the swizzle
    const int r = threadIdx.x;
    const bool live = r < nrows;
    const size_t row = (size_t)(q_begin + t0 + (live ? r / G : 0)) * p.num_heads + (size_t)g * G +
                       (live ? r % G : 0);
    const uint4* src = reinterpret_cast<const uint4*>(p.q + row * Sh::D);
#pragma unroll
    for (int c = 0; c < 16; ++c) {
      const uint4 v = live ? __ldg(src + c) : make_uint4(0u, 0u, 0u, 0u);
      const uint32_t dst = qbuf + (c / 8) * (Sh::kRows * 128) + sw128_off(r, (c % 8) * 8);
      asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(dst), "r"(v.x), "r"(v.y),
                   "r"(v.z), "r"(v.w)
                   : "memory");
    }
    fence_proxy_async_smem();
  }
  // whether any table entry the tile reads is out of range (the copies skip
  // such sub-tiles; the softmax then masks them span by span)
  bool bad_entry = false;
  for (int t = threadIdx.x; t * SUB < n_tiles; t += Sh::kThreads) {
    const int e = __ldg(table + t);
    bad_entry = bad_entry || e < 0 || e >= p.num_blocks;
  }
  tc_fence_before();
  const bool any_bad = __syncthreads_or(bad_entry);
  tc_fence_after();
  const uint32_t tbase = s_tmem;
  const uint32_t tS = tbase;         // S buffers: columns 0..127 and 128..255
  const uint32_t tO = tbase + 256;   // O: columns 256..383

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
      return (boxer && t < n_tiles) ? __ldg(table + t / SUB) : -1;
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
        const int t = i * Sh::kSubs + u;
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
      // Issue whichever product is ready.  PV products go in span order (the
      // softmax warps rescale O between them) and need P and V; S(j) needs
      // K(j) and S buffer j % 2 read by the softmax warps (span j - 2).
      // A barrier's phase is tested by its parity alone, so a test must not
      // run while the slot's previous load can still be in flight: K(j)'s
      // slot held V(j - 3) (K0 for j = 2), landed once PV(j - 3) was issued;
      // V(i)'s slot held K(i) (V(i - 2) for the last span), landed before S(i)
      // (or PV(i - 2)) was issued.
      int next_s = 0, next_pv = 0;
      uint64_t t_last = global_timer_ns();
      int idle = 0;
      while (next_pv < n_spans) {
        bool progressed = false;
        const int i = next_pv;
        const int vs = slot_of(vload(i));
        if (mbar_test(p_ready(i & 1), (i >> 1) & 1) && mbar_test(full(vs), use_of(vload(i)) & 1)) {
          tc_fence_after();
          const uint32_t vb = ring + vs * Sh::kSlotBytes;
          const uint32_t pb = pbuf + (i & 1) * Sh::kPBytes;
#pragma unroll
          for (int ks = 0; ks < Sh::kSpan / 16; ++ks) {
            // P: K-major over the span's tokens; V: MN-major (d contiguous),
            // its two d halves kHalfBytes apart, 8-token groups 1 KB apart
            const uint64_t a = smem_desc_sw128(pb + (ks / 4) * (Sh::kRows * 128) + (ks % 4) * 32,
                                               16, 1024);
            const uint64_t b = smem_desc_sw128(vb + ks * 2048, Sh::kHalfBytes, 1024);
            tc_mma_f16(tO, a, b, Sh::kIdescPV, (i > 0 || ks > 0) ? 1u : 0u);
          }
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
          const uint32_t kb = ring + ks_slot * Sh::kSlotBytes;
#pragma unroll
          for (int ks = 0; ks < Sh::D / 16; ++ks) {
            const int h = ks / 4, w4 = ks % 4;
            const uint64_t a = smem_desc_sw128(qbuf + h * (Sh::kRows * 128) + w4 * 32, 16, 1024);
            const uint64_t b = smem_desc_sw128(kb + h * Sh::kHalfBytes + w4 * 32, 16, 1024);
            tc_mma_f16(tS + (j & 1) * 128, a, b, Sh::kIdescS, ks > 0);
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
          if (PKV_PREFILL_MMA_POLL_NS > 0) __nanosleep(PKV_PREFILL_MMA_POLL_NS);
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
    // ============ softmax warps 0..7: two threads per row ============
    // Warps w and w + 4 share tensor-memory lanes 32 (w % 4) .. + 31 (rows);
    // `hf` = w / 4 picks the half of the span's tokens a thread handles (and
    // the half of O's columns it rescales and writes).  A row's two halves
    // exchange their maxima through shared memory once per span, and their
    // sums at the end.  The warps never leave the span loop early: on an
    // abort they skip the work but still pass every barrier among them.
    __shared__ float s_mx[2][2][Sh::kRows];  // [span parity][half][row]
    __shared__ float s_l[2][Sh::kRows];      // final sums [half][row]
    const int hf = warp >> 2;
    const int r = 32 * (warp & 3) + lane;    // this thread's row (tensor-memory lane)
    const bool live = r < nrows;
    const int lim = live ? pos0 + t0 + r / G + 1 : 0;  // positions below it count
    // positions below this count for every row (the first query's limit)
    const int all_see = min(tok_end, pos0 + t0 + 1);
    const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
    constexpr int kSoftThreads = Sh::kSoftWarps * 32;
    // Lazy rescaling: the row's reference maximum moves only when a score
    // exceeds it by more than 2^kLazy, so P stays <= 2^kLazy (exact in f16,
    // and the running sum and O scale together, cancelling in O / l).  Both
    // threads of a row take the same decisions from the same maxima.
    constexpr float kLazy = 8.f;
    const float sl2 = p.scale_log2;
    float m_run = -CUDART_INF_F, l_run = 0.f;
    // which sub-tiles of span i hold data (bit u; the copy warps skip, and
    // flag, a sub-tile whose table entry is out of range), read a span ahead
    // when the tile reads any such entry (else every sub-tile holds data;
    // those past the last position are masked by the causal limit)
    auto span_ok = [&](int i) {
      uint32_t bits = 0;
#pragma unroll
      for (int u = 0; u < Sh::kSubs; ++u) {
        const int t = i * Sh::kSubs + u;
        const int e = t < n_tiles ? __ldg(table + t / SUB) : -1;
        if (e >= 0 && e < p.num_blocks) bits |= 1u << u;
      }
      return bits;
    };
    uint32_t ok_next = any_bad ? span_ok(0) : 0xFFu;
    bool dead = false;
    for (int i = 0; i < n_spans; ++i) {
      const int b = i & 1;
      const uint32_t okb = ok_next;
      if (any_bad && i + 1 < n_spans) ok_next = span_ok(i + 1);
      dead = dead || aborted();
      if (!dead && !wait(s_ready(b), (i >> 1) & 1)) dead = true;
      dead = __any_sync(0xffffffffu, dead);  // warp-uniform before the .sync.aligned loads
      uint32_t ra[64];                       // this row's scores, tokens 64 hf .. 64 hf + 63
      if (!dead) {
        tc_fence_after();
        tmem_ld64(tS + b * 128 + hf * 64 + lane_base, ra);
        tc_fence_before();
      } else {
#pragma unroll
        for (int j = 0; j < 64; ++j) ra[j] = 0u;
      }
      __syncwarp();
      if (!dead && lane == 0) mbar_arrive(s_free(b));
      const int span0 = i * Sh::kSpan;
      const int tok0 = span0 + hf * 64;  // this thread's first position
      // every position of the span counts for every row: no masks
      const bool simple = okb == 0xFFu && span0 + Sh::kSpan <= all_see;
      // this half's maximum in the log2 domain; the exponents below are
      // fma(ra, mul, -mu).  With no masks and a positive scale the scores
      // stay raw (scaling by a positive factor keeps their order, so the
      // scaled maximum is the raw one scaled); else they are scaled (and
      // masked) in place.
      const bool raw = simple && sl2 > 0.f;
      const float mul = raw ? sl2 : 1.f;
      float mx = -CUDART_INF_F;
      if (raw) {
#pragma unroll
        for (int j = 0; j < 64; ++j) mx = fmaxf(mx, __uint_as_float(ra[j]));
        mx *= sl2;
      } else if (simple) {
#pragma unroll
        for (int j = 0; j < 64; ++j) {
          const float x = __uint_as_float(ra[j]) * sl2;
          ra[j] = __float_as_uint(x);
          mx = fmaxf(mx, x);
        }
      } else {
#pragma unroll
        for (int j = 0; j < 64; ++j) {
          const bool ok = ((okb >> ((hf * 64 + j) >> 4)) & 1u) && tok0 + j < lim;
          const float x = ok ? __uint_as_float(ra[j]) * sl2 : -CUDART_INF_F;
          ra[j] = __float_as_uint(x);
          mx = fmaxf(mx, x);
        }
      }
      // the row's maximum: this half's and the other's
      s_mx[b][hf][r] = mx;
      named_barrier(1, kSoftThreads);
      mx = fmaxf(mx, s_mx[b][hf ^ 1][r]);
      const bool grow =
          mx > m_run + kLazy || (m_run == -CUDART_INF_F && mx != -CUDART_INF_F);
      float alpha = 1.f;
      if (grow) {
        alpha = m_run == -CUDART_INF_F ? 0.f : ex2_approx(m_run - mx);
        m_run = mx;
        l_run *= alpha;
      }
      const float mu = m_run == -CUDART_INF_F ? 0.f : m_run;
      // P buffer b was read by PV(i-2); O changes only after PV(i-1)
      if (!dead && i >= 2 && !wait(pv_done(b), ((i - 2) >> 1) & 1)) dead = true;
      if (__any_sync(0xffffffffu, grow && i >= 1)) {
        // some row of this warp moved its maximum: rescale this warp's half
        // of those rows of O (alpha = 1 for the others) once PV(i-1) completed
        if (!dead && !wait(pv_done((i - 1) & 1), ((i - 1) >> 1) & 1)) dead = true;
        dead = __any_sync(0xffffffffu, dead);
        if (!dead) {
          tc_fence_after();
#pragma unroll 1
          for (int c = 0; c < 4; ++c) {
            uint32_t o[16];
            const uint32_t ta = tO + hf * 64 + c * 16 + lane_base;
            tmem_ld16(ta, o);
#pragma unroll
            for (int k = 0; k < 16; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * alpha);
            tmem_st16(ta, o);
          }
        }
      }
      if (!dead) {
        // this half of the row of P (f16), [token half][128 rows][64 tokens],
        // K-major with the swizzle; the running sum adds the same exponentials
        const uint32_t pb = pbuf + b * Sh::kPBytes + hf * (Sh::kRows * 128);
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          uint32_t w[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int j = c * 8 + 2 * e;
            const float p0 = ex2_approx(fmaf(__uint_as_float(ra[j]), mul, -mu));
            const float p1 = ex2_approx(fmaf(__uint_as_float(ra[j + 1]), mul, -mu));
            l_run += p0 + p1;
            const __half2 h2 = __floats2half2_rn(p0, p1);
            w[e] = *reinterpret_cast<const uint32_t*>(&h2);
          }
          asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(pb + sw128_off(r, c * 8)),
                       "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3])
                       : "memory");
        }
        // V row r of the span (threads of half 0): zero it when its position
        // counts for no row (past the tile's last query, or in a sub-tile with
        // no data) once it has landed; V(i)'s slot held K(i) (V(i - 2) for the
        // last span), landed before S(i) (or PV(i - 2), completed above)
        const int tok = span0 + r;
        if (hf == 0 && !simple && (!((okb >> (r >> 4)) & 1u) || tok >= tok_end)) {
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
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (!dead && lane == 0) mbar_arrive(p_ready(b));
    }
    // ---- the result: this half of the row of O over the row's sum
    const int last = n_spans - 1;
    if (!dead && !wait(pv_done(last & 1), (last >> 1) & 1)) dead = true;
    dead = __any_sync(0xffffffffu, dead);
    s_l[hf][r] = l_run;
    named_barrier(1, kSoftThreads);  // every softmax warp has seen the end (or the abort)
    const bool write = !dead && !aborted();
    if (__any_sync(0xffffffffu, write)) {
      tc_fence_after();
      const float den = s_l[0][r] + s_l[1][r];
      const float inv = den > 0.f ? 1.f / den : 0.f;
      const size_t orow = (size_t)(q_begin + t0 + (live ? r / G : 0)) * p.num_heads +
                          (size_t)g * G + (live ? r % G : 0);
      uint4* dst = reinterpret_cast<uint4*>(p.out + orow * Sh::D + hf * 64);
      uint32_t o[64];
      tmem_ld64(tO + hf * 64 + lane_base, o);
      if (write && live) {
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
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tbase, Sh::kTmemCols);
}

}  // namespace pkv
