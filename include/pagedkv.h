/*
 * libpagedkv — batched paged-KV decode attention for one GB300 (sm_103a).
 *
 * One new query token per sequence attends over f16 K/V stored in fixed-size
 * physical blocks, reached through a per-sequence block table and context
 * length, with grouped-query heads.  The operations follow the paged-decode
 * backends of the Rust LLM-serving crates:
 *   - ferrum-kernels src/backend/cuda/paged.rs — paged_decode_attention,
 *     paged_batched_decode_attention, paged_batched_flash_dispatch (split-K
 *     phase 1 + reduce, split-count heuristic), paged_batched_decode_single_pass;
 *   - kapsl-backends src/gguf_native.rs — forward_batch_decode_greedy and
 *     one_token_compute (kv write at (physical block, position in block),
 *     paged attention with block tables and context_lens, scale argument);
 *   - cortiq-engine src/gpu_cuda.rs — GQA grouping hpk = nh / nkv.
 *
 * Conventions for every call
 *   - Pointers named "device" are CUDA device pointers (or managed memory).
 *     Every one of them except the K/V pools (which the kernels read with
 *     TMA tensor copies and must be device memory) may instead point at
 *     page-locked host memory (cudaMallocHost, cudaHostAlloc, or memory
 *     registered with cudaHostRegister): the kernels then read and write it
 *     in place over the host link, so a decode step needs no separate copy
 *     of its small inputs (q, new rows, slots, tables, lengths) or of its
 *     output.
 *     The caller owns every buffer.  The library allocates nothing per call.
 *     Its own device memory is static, declared in the library and held by
 *     every GPU that loads it until the process exits: one 32-bit status
 *     word (see pkv_read_device_status) and the PKV_NOALLOC_SCRATCH_BYTES
 *     buffer of pkv_decode_splitk_noalloc.
 *   - f16 is IEEE binary16 (2 bytes).  All arrays are dense, row-major,
 *     with no padding between rows.
 *   - KV cache layout: k_cache and v_cache are each
 *       f16 [num_blocks][num_kv_heads][block_size][head_dim],
 *     so the (block, kv_head) tile of block_size x head_dim is contiguous.
 *     Both must be 16-byte aligned.
 *   - Supported: head_dim in {64, 128}; block_size in {16, 32};
 *     num_heads / num_kv_heads (the group) in 1..8.
 *   - stream is a cudaStream_t (NULL = the legacy default stream).  Every
 *     call is asynchronous on it, reads no device memory on the host and
 *     never synchronizes, so a sequence of calls can be captured into a CUDA
 *     graph (pkv_read_device_status is the one exception).
 *   - Errors: a call returns a pkv_status.  Arguments are validated on the
 *     host before any CUDA call; a rejected call launches nothing.
 *     PKV_ERR_CUDA means a launch failed; pkv_last_error() has the message.
 *   - Bad data inside device arrays (a block id outside [0, num_blocks), a
 *     context length above max_blocks_per_seq * block_size, a slot past the
 *     pool) is never dereferenced: the kernel skips it and sets a bit of the
 *     device status word.
 */
#ifndef PAGEDKV_H
#define PAGEDKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int32_t pkv_status;

#define PKV_OK 0
#define PKV_ERR_INVALID_ARG (-1)       /* bad size, null pointer, misalignment */
#define PKV_ERR_UNSUPPORTED (-2)       /* valid but not built: head_dim, block_size, group */
#define PKV_ERR_SCRATCH_TOO_SMALL (-3) /* split-K scratch missing or too small */
#define PKV_ERR_CUDA (-4)              /* a CUDA call failed; see pkv_last_error */

/* Bits of the device status word (OR-ed by kernels, read by
 * pkv_read_device_status). */
#define PKV_DEV_BAD_SLOT 0x1u        /* append: slot >= num_blocks*block_size; token skipped */
#define PKV_DEV_BAD_BLOCK_ID 0x2u    /* decode: table entry outside [0,num_blocks); block skipped */
#define PKV_DEV_BAD_CONTEXT_LEN 0x4u /* decode: context_len < 0 (taken as 0) or above
                                        max_blocks_per_seq*block_size (clamped) */
#define PKV_DEV_WAIT_TIMEOUT 0x8u    /* decode: a tile copy did not land within 100 ms;
                                        the affected outputs were not written, and
                                        decode calls write nothing until the word
                                        is cleared by pkv_read_device_status */

/* Largest num_splits pkv_decode_splitk accepts. */
#define PKV_MAX_SPLITS 128

/*
 * pkv_append — slot-mapped KV write (kapsl-backends src/gguf_native.rs,
 * forward_batch_decode_greedy / one_token_compute: launch_batch_kv_write and
 * launch_kv_write store a token's K and V at (physical block, position in
 * block); here the pair is one integer slot = block * block_size + offset).
 *
 *   k, v          device f16 [num_tokens][num_kv_heads][head_dim], 16-byte aligned
 *   slot_mapping  device int32 [num_tokens]; slot < 0 skips the token
 *   k_cache, v_cache  device f16 pools (layout above), written in place
 *
 * For token t with s = slot_mapping[t] >= 0 and every kv head h:
 *   k_cache[s / block_size][h][s % block_size][:] = k[t][h][:]  (same for v),
 * bit for bit.  Two tokens with the same non-negative slot race (undefined).
 * num_tokens == 0 returns PKV_OK without a launch.
 */
pkv_status pkv_append(const void* k, const void* v, const int32_t* slot_mapping,
                      int32_t num_tokens, void* k_cache, void* v_cache,
                      int32_t num_blocks, int32_t block_size, int32_t num_kv_heads,
                      int32_t head_dim, void* stream);

/*
 * pkv_decode — single-pass batched paged decode attention (ferrum-kernels
 * src/backend/cuda/paged.rs, paged_batched_decode_single_pass and
 * paged_decode_attention with q_len == 1; kapsl-backends
 * launch_paged_attention parameters).
 *
 *   q             device f16 [num_seqs][num_heads][head_dim], 4-byte aligned
 *   k_cache, v_cache  device f16 pools (layout above), read only
 *   block_tables  device int32 [num_seqs][max_blocks_per_seq]: physical block
 *                 of logical block j of sequence s; entries at or past
 *                 ceil(context_lens[s] / block_size) are never read
 *   context_lens  device int32 [num_seqs]: tokens to attend to, including the
 *                 one appended this step (positions 0 .. L-1)
 *   scale         softmax scale applied to q.k (usually 1/sqrt(head_dim))
 *   out           device f16 [num_seqs][num_heads][head_dim], 4-byte aligned
 *
 * For sequence s, query head h, kv head g = h / (num_heads / num_kv_heads):
 *   out[s][h] = sum_i softmax_i(scale * q[s][h] . K_s[i]) V_s[i],
 *   K_s[i] = k_cache[block_tables[s][i / block_size]][g][i % block_size].
 * Accumulation is f32; out is rounded to nearest-even f16.  L == 0 gives
 * zeros.  num_seqs == 0 returns PKV_OK without a launch.
 */
pkv_status pkv_decode(const void* q, const void* k_cache, const void* v_cache,
                      const int32_t* block_tables, const int32_t* context_lens,
                      int32_t num_seqs, int32_t max_blocks_per_seq, int32_t num_blocks,
                      float scale, int32_t num_heads, int32_t num_kv_heads,
                      int32_t head_dim, int32_t block_size, void* out, void* stream);

/*
 * pkv_decode_splitk — the same result as pkv_decode, with each sequence's
 * context split into chunks processed by separate CTAs and merged by a
 * log-sum-exp combine (ferrum-kernels src/backend/cuda/paged.rs,
 * paged_batched_flash_dispatch: phase 1 writes f32 partial out / max / sum,
 * phase 2 reduces them per (sequence, head)).
 *
 *   num_splits    0 = pick with pkv_pick_num_splits for the current GPU; 1 =
 *                 run the single-pass kernel (no scratch needed);
 *                 2..PKV_MAX_SPLITS = that many splits (at most
 *                 max_blocks_per_seq; pkv_decode_splitk_plan gives the count
 *                 launched).  The chunks are cut on the GPU from the longest
 *                 context in context_lens, Lmax: split k takes blocks
 *                 [k c, (k+1) c) of every sequence, c = ceil(ceil(Lmax /
 *                 block_size) / S) blocks (with num_splits = 0, at least
 *                 256 tokens' worth), so tables sized beyond the contexts
 *                 they hold still spread the work; splits past a sequence's
 *                 end do no work.
 *   scratch       device memory of at least the bytes pkv_decode_splitk_plan
 *                 returns for these sizes and num_splits
 *                 (pkv_splitk_scratch_bytes of the split count launched),
 *                 16-byte aligned, caller-owned; its contents need no
 *                 initialisation and are overwritten.  Calls that overlap on
 *                 the GPU must not share scratch.
 *   other arguments as pkv_decode.
 *
 * Returns PKV_ERR_SCRATCH_TOO_SMALL when S > 1 and the scratch is null or
 * smaller than required.
 */
pkv_status pkv_decode_splitk(const void* q, const void* k_cache, const void* v_cache,
                             const int32_t* block_tables, const int32_t* context_lens,
                             int32_t num_seqs, int32_t max_blocks_per_seq,
                             int32_t num_blocks, float scale, int32_t num_heads,
                             int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                             void* out, int32_t num_splits, void* scratch,
                             size_t scratch_bytes, void* stream);

/*
 * pkv_append_decode — one decode step in one launch: the slot-mapped append
 * of each sequence's newest token followed by the decode of
 * pkv_decode_splitk (the per-layer kv write then paged attention of
 * kapsl-backends src/gguf_native.rs, forward_batch_decode_greedy).
 *
 *   k_new, v_new  device f16 [num_seqs][num_kv_heads][head_dim], 16-byte
 *                 aligned: row s is sequence s's newest token, at position
 *                 context_lens[s] - 1
 *   slot_mapping  device int32 [num_seqs]: the slot of that position
 *                 (block_tables[s][p / block_size] * block_size +
 *                 p % block_size, p = context_lens[s] - 1), or < 0 to
 *                 append nothing for sequence s
 *   other arguments as pkv_decode_splitk
 *
 * The result equals pkv_append(k_new, v_new, slot_mapping, num_seqs, ...)
 * then pkv_decode_splitk(...): the cache ends with the new rows written and
 * out holds the attention over every context including them.  The decode CTA
 * that reads position context_lens[s] - 1 writes the row and uses it
 * directly.  A non-negative slot that is not that position's slot is not
 * written (PKV_DEV_BAD_SLOT is set) and the decode reads the cache as it is.
 */
pkv_status pkv_append_decode(const void* k_new, const void* v_new, const int32_t* slot_mapping,
                             void* k_cache, void* v_cache, const void* q,
                             const int32_t* block_tables, const int32_t* context_lens,
                             int32_t num_seqs, int32_t max_blocks_per_seq, int32_t num_blocks,
                             float scale, int32_t num_heads, int32_t num_kv_heads,
                             int32_t head_dim, int32_t block_size, void* out,
                             int32_t num_splits, void* scratch, size_t scratch_bytes,
                             void* stream);

/*
 * pkv_varlen_attention — several query tokens per sequence over its paged
 * context, causal (ferrum-kernels src/backend/cuda/paged.rs,
 * paged_varlen_attention, and paged_decode_attention with q_len > 1:
 * pos_offset = final_kv_len - q_len): prefill chunks, speculative-decode
 * verification, multi-token decode.
 *
 *   q             device f16 [total_q][num_heads][head_dim], token-major,
 *                 4-byte aligned
 *   cu_seqlens_q  device int32 [num_seqs + 1]: the queries of sequence s are
 *                 rows cu_seqlens_q[s] .. cu_seqlens_q[s+1]-1 (rising from 0
 *                 to total_q)
 *   pos_offsets   device int32 [num_seqs]: position of sequence s's first
 *                 query; query t sits at pos_offsets[s] + t and attends to
 *                 positions 0 .. pos_offsets[s] + t, whose K/V must already
 *                 be in the cache (so pos_offsets[s] + q_len <=
 *                 max_blocks_per_seq * block_size)
 *   max_q_len     a host-side bound on every sequence's query count (sizes
 *                 the grid; queries past it are not computed and
 *                 PKV_DEV_BAD_CONTEXT_LEN is set)
 *   out           device f16 [total_q][num_heads][head_dim]
 *   other arguments as pkv_decode.
 *
 * Two kernels serve it.  For short query runs (a few tokens per sequence)
 * one CTA covers max(1, 8 / group) queries of one sequence and KV head and
 * reads the context once per chunk of queries.  When max_q_len x group >=
 * 128 at head_dim 128 on blocked pools (chunked prefill), the call runs the
 * prefill kernel instead: one CTA per pair of tiles of 128 / group queries
 * of a sequence and KV head, both products on the 5th-generation tensor
 * cores (tcgen05.mma, 128 (query, head) rows per tile x 128-token spans,
 * scores and output in tensor memory), one CTA per SM.  The two compute the same attention within the
 * stated tolerance; arguments, flags and errors are the same.
 */
pkv_status pkv_varlen_attention(const void* q, const void* k_cache, const void* v_cache,
                                const int32_t* cu_seqlens_q, const int32_t* pos_offsets,
                                const int32_t* block_tables, int32_t num_seqs, int32_t total_q,
                                int32_t max_q_len, int32_t max_blocks_per_seq,
                                int32_t num_blocks, float scale, int32_t num_heads,
                                int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                                void* out, void* stream);

/*
 * The vLLM cache layout: the pools that ferrum-kernels
 * src/backend/cuda/paged.rs reaches through its vLLM-layout paged write
 * (split_qkv_norm_rope_into_paged_cache_vllm) and vLLM paged attention
 * (paged_decode_attention_v2).  The pages name this layout without
 * spelling it out; it is read as vLLM's published paged-attention layout,
 * with x = 16 bytes / sizeof(f16) = 8:
 *
 *   k_cache  f16 [num_blocks][num_kv_heads][head_dim / 8][block_size][8]:
 *            element d of the token at offset o of block b, kv head h, is
 *            k_cache[b][h][d / 8][o][d % 8]
 *   v_cache  f16 [num_blocks][num_kv_heads][head_dim][block_size]:
 *            v_cache[b][h][d][o]
 *
 * Each (block, kv head) tile is still one contiguous block_size * head_dim
 * f16 run per pool, so these calls read the same bytes as the blocked ones.
 * Slots, tables, lengths, q, out, scratch and every status, flag and
 * size rule are those of pkv_append / pkv_decode_splitk.
 */

/*
 * pkv_append_vllm_layout — pkv_append into vLLM-layout pools: for token t
 * with slot_mapping[t] = b * block_size + o >= 0, k[t][h][d] goes to
 * k_cache[b][h][d / 8][o][d % 8] and v[t][h][d] to v_cache[b][h][d][o],
 * bit for bit.  Arguments, skips, flags and errors as pkv_append.
 */
pkv_status pkv_append_vllm_layout(const void* k, const void* v, const int32_t* slot_mapping,
                                  int32_t num_tokens, void* k_cache, void* v_cache,
                                  int32_t num_blocks, int32_t block_size, int32_t num_kv_heads,
                                  int32_t head_dim, void* stream);

/*
 * pkv_decode_vllm_layout — pkv_decode_splitk over vLLM-layout pools (the
 * decode of paged_decode_attention_v2 in ferrum-kernels
 * src/backend/cuda/paged.rs): the same attention, the same outputs within
 * rounding.  num_splits 0, 1 or 2..PKV_MAX_SPLITS as for pkv_decode_splitk
 * (same scratch).
 */
pkv_status pkv_decode_vllm_layout(const void* q, const void* k_cache, const void* v_cache,
                                  const int32_t* block_tables, const int32_t* context_lens,
                                  int32_t num_seqs, int32_t max_blocks_per_seq,
                                  int32_t num_blocks, float scale, int32_t num_heads,
                                  int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                                  void* out, int32_t num_splits, void* scratch,
                                  size_t scratch_bytes, void* stream);

/*
 * pkv_varlen_attention_vllm_layout — pkv_varlen_attention over vLLM-layout
 * pools (ferrum-kernels src/backend/cuda/paged.rs,
 * paged_varlen_attention_vllm_layout: several causal queries per sequence on
 * the vLLM cache).  Arguments, results, flags and errors as
 * pkv_varlen_attention; only the pool layout differs.
 */
pkv_status pkv_varlen_attention_vllm_layout(
    const void* q, const void* k_cache, const void* v_cache, const int32_t* cu_seqlens_q,
    const int32_t* pos_offsets, const int32_t* block_tables, int32_t num_seqs, int32_t total_q,
    int32_t max_q_len, int32_t max_blocks_per_seq, int32_t num_blocks, float scale,
    int32_t num_heads, int32_t num_kv_heads, int32_t head_dim, int32_t block_size, void* out,
    void* stream);

/*
 * pkv_varlen_attention_splitk — pkv_varlen_attention with each chunk of
 * queries' context split over CTAs and merged by a log-sum-exp combine
 * (ferrum-kernels src/backend/cuda/paged.rs, paged_varlen_split_k_dispatch:
 * phase 1 per (query token, head, split) writes f32 partial out / max / sum,
 * a reduce per (query token, head) merges them).  The same result as
 * pkv_varlen_attention within rounding; it pays off when few sequences have
 * long contexts.
 *
 *   num_splits    0 = pick: when the unsplit grid (num_seqs x num_kv_heads x
 *                 query chunks) is under one wave of resident CTAs, the
 *                 split count that brings it nearest one wave, capped so a
 *                 split keeps >= 256 tokens of max_blocks_per_seq *
 *                 block_size, at most 64; else 1.  Chunked-prefill sizes
 *                 (max_q_len x group >= 128 at head_dim 128, either layout)
 *                 count instead the prefill kernel's pairs of 128 / group
 *                 query tiles against one CTA per SM, each split keeping
 *                 >= 512 tokens.  1 = no split (no scratch needed);
 *                 2..PKV_MAX_SPLITS = that many splits (at most
 *                 max_blocks_per_seq).  As in pkv_decode_splitk the chunks
 *                 are cut on the GPU: c = ceil(n / S) blocks, n the most
 *                 blocks any chunk of queries reads (with num_splits = 0, at
 *                 least 256 tokens' worth, 512 for chunked prefill).  On
 *                 blocked pools a chunked-prefill call runs the prefill
 *                 kernel for every split (see pkv_varlen_attention).
 *   scratch       device memory of at least the bytes pkv_varlen_splitk_plan
 *                 returns (pkv_splitk_scratch_bytes(total_q, num_heads,
 *                 head_dim, S) for the split count launched), 16-byte
 *                 aligned, caller-owned, no initialisation needed; calls that
 *                 overlap on the GPU must not share it.
 *   other arguments, results and flags as pkv_varlen_attention.
 *
 * Returns PKV_ERR_SCRATCH_TOO_SMALL when S > 1 and the scratch is null or
 * smaller than required; PKV_ERR_INVALID_ARG for num_splits outside
 * 0..PKV_MAX_SPLITS.
 */
pkv_status pkv_varlen_attention_splitk(
    const void* q, const void* k_cache, const void* v_cache, const int32_t* cu_seqlens_q,
    const int32_t* pos_offsets, const int32_t* block_tables, int32_t num_seqs, int32_t total_q,
    int32_t max_q_len, int32_t max_blocks_per_seq, int32_t num_blocks, float scale,
    int32_t num_heads, int32_t num_kv_heads, int32_t head_dim, int32_t block_size, void* out,
    int32_t num_splits, void* scratch, size_t scratch_bytes, void* stream);

/*
 * pkv_varlen_pick_num_splits — the split count pkv_varlen_attention_splitk
 * uses for num_splits = 0 (host arithmetic only; num_sms is the GPU's SM
 * count) at sizes other than chunked prefill at head_dim 128, whose rule
 * (pkv_varlen_attention_splitk) pkv_varlen_splitk_plan applies.  Returns 1
 * for invalid arguments.
 */
int32_t pkv_varlen_pick_num_splits(int32_t num_seqs, int32_t num_heads, int32_t num_kv_heads,
                                   int32_t max_q_len, int32_t max_blocks_per_seq,
                                   int32_t block_size, int32_t num_sms);

/*
 * pkv_set_varlen_tensor_path — which kernel pkv_varlen_attention and
 * pkv_varlen_attention_splitk run (blocked pools, head_dim 128) when a CTA
 * covers more than 8 (query, head) columns (group x queries per sequence
 * above 8, e.g. 4 draft tokens at group 4): 0 (the initial setting) the
 * mma.sync kernel; 1 the kernel that computes both products on the
 * 5th-generation tensor cores (tcgen05.mma, scores and output accumulated
 * in tensor memory, 128-token spans).  Both compute the same attention
 * (within the stated tolerance; they round differently) from the same
 * arguments, split-K partials included.  Other calls, the vLLM layout,
 * head_dim 64 and smaller column counts are unaffected.  Process-wide;
 * calls already enqueued keep the kernel they were launched with.
 * Returns the previous setting, or -1 (nothing changed) for a value other
 * than 0 or 1.
 */
int32_t pkv_set_varlen_tensor_path(int32_t on);

/*
 * pkv_varlen_attention_splitk_vllm_layout — pkv_varlen_attention_splitk over
 * vLLM-layout pools.
 */
pkv_status pkv_varlen_attention_splitk_vllm_layout(
    const void* q, const void* k_cache, const void* v_cache, const int32_t* cu_seqlens_q,
    const int32_t* pos_offsets, const int32_t* block_tables, int32_t num_seqs, int32_t total_q,
    int32_t max_q_len, int32_t max_blocks_per_seq, int32_t num_blocks, float scale,
    int32_t num_heads, int32_t num_kv_heads, int32_t head_dim, int32_t block_size, void* out,
    int32_t num_splits, void* scratch, size_t scratch_bytes, void* stream);

/*
 * pkv_qkv_norm_rope_append — the step before attention in one launch: split
 * each token's fused projection row into query, key and value heads, RMS-norm
 * the query and key heads, turn them by the rotary angles of the token's
 * position, write the queries token-major and append the keys and values to
 * the paged pools (ferrum-kernels src/backend/cuda/paged.rs,
 * split_qkv_norm_rope_into_paged_cache and its _varlen form; the pages give
 * the launch, the arithmetic below is its plainest reading).
 *
 *   qkv           device f16 [total_q][(num_heads + 2 num_kv_heads) * head_dim]:
 *                 each row holds the query heads, then the key heads, then
 *                 the value heads
 *   q_norm_w, k_norm_w  device f16 [head_dim], or NULL for no norm of that
 *                 kind: y = x / sqrt(mean(x^2) + eps) * w over a head
 *   cos_table, sin_table  device f32 [max_pos][head_dim / 2]: the rotary
 *                 angle's cosine and sine per position and pair
 *   q_out         device f16 [total_q][num_heads][head_dim]
 *   k_cache, v_cache  device f16 pools (layout above), written in place
 *   cu_seqlens_q  device int32 [num_seqs + 1], rising from 0 to total_q
 *   pos_offsets   device int32 [num_seqs]: row t of sequence s is at
 *                 position p = pos_offsets[s] + t, its rotary position and
 *                 its cache row
 *   block_tables  device int32 [num_seqs][max_blocks_per_seq]
 *
 * Rotation: pair (x[i], x[i + head_dim/2]) of a (normed) query or key head
 * becomes (x[i] c - x[i + head_dim/2] s, x[i + head_dim/2] c + x[i] s) with
 * c = cos_table[p][i], s = sin_table[p][i]; f32 arithmetic, f16 results
 * rounded to nearest even.  Value heads are copied bit for bit.  Keys and
 * values land at slot block_tables[s][p / block_size] * block_size +
 * p % block_size, as pkv_append writes.  A row whose sequence range or
 * position is invalid (p < 0, p >= max_pos or beyond the table) is skipped
 * and sets PKV_DEV_BAD_CONTEXT_LEN; a table entry outside [0, num_blocks)
 * skips that row's key and value writes and sets PKV_DEV_BAD_BLOCK_ID.
 * head_dim in {64, 128}, block_size in {16, 32}; eps >= 0.  qkv, q_out, the
 * pools, the weights and the rotary tables must be 16-byte aligned (the
 * kernel moves 16-byte words), cu_seqlens_q, pos_offsets and block_tables
 * 4-byte aligned.
 */
pkv_status pkv_qkv_norm_rope_append(const void* qkv, const void* q_norm_w, const void* k_norm_w,
                                    const float* cos_table, const float* sin_table, void* q_out,
                                    void* k_cache, void* v_cache, const int32_t* cu_seqlens_q,
                                    const int32_t* pos_offsets, const int32_t* block_tables,
                                    int32_t num_seqs, int32_t total_q, int32_t max_blocks_per_seq,
                                    int32_t num_blocks, int32_t num_heads, int32_t num_kv_heads,
                                    int32_t head_dim, int32_t block_size, int32_t max_pos, float eps,
                                    void* stream);

/*
 * pkv_qkv_norm_rope_append_decode — a whole decode attention step in one
 * launch (two with splits): pkv_qkv_norm_rope_append of each sequence's
 * newest token (one row per sequence, at position context_lens[s] - 1)
 * followed by the decode of pkv_decode_splitk with the rotated queries.  The
 * decode CTA of (sequence, KV head[, split]) computes its group's queries
 * itself; the CTA whose chunk holds the newest position computes that KV
 * head's key and value row, writes it to the pools and attends to it
 * directly (ferrum-kernels src/backend/cuda/paged.rs,
 * split_qkv_norm_rope_into_paged_cache then paged_decode_attention, the
 * per-layer order of one decode step).
 *
 *   qkv           device f16 [num_seqs][(num_heads + 2 num_kv_heads) * head_dim],
 *                 4-byte aligned: sequence s's newest token's projection row
 *   q_norm_w, k_norm_w, cos_table, sin_table, eps  as
 *                 pkv_qkv_norm_rope_append
 *   max_pos       rows in the rotary tables; a sequence with
 *                 context_lens[s] > max_pos sets PKV_DEV_BAD_CONTEXT_LEN,
 *                 appends nothing and attends with zero queries (its output
 *                 is written but meaningless)
 *   k_cache, v_cache  the pools (blocked layout), read and written in place
 *   other arguments as pkv_decode_splitk
 *
 * The cache ends as pkv_qkv_norm_rope_append would leave it (the key and
 * value rows of position context_lens[s] - 1 written) and out holds the
 * attention of the rotated queries over every context including the new
 * rows.  The queries are not written out.  A table entry outside
 * [0, num_blocks) at the newest position sets PKV_DEV_BAD_SLOT and the row
 * is neither written nor used (the decode flags the tile as well).
 */
pkv_status pkv_qkv_norm_rope_append_decode(
    const void* qkv, const void* q_norm_w, const void* k_norm_w, const float* cos_table,
    const float* sin_table, int32_t max_pos, float eps, void* k_cache, void* v_cache,
    const int32_t* block_tables, const int32_t* context_lens, int32_t num_seqs,
    int32_t max_blocks_per_seq, int32_t num_blocks, float scale, int32_t num_heads,
    int32_t num_kv_heads, int32_t head_dim, int32_t block_size, void* out, int32_t num_splits,
    void* scratch, size_t scratch_bytes, void* stream);

/*
 * pkv_selftest_wait_timeout — a diagnostic of the failure path (the pages
 * have no counterpart): launches one warp that waits on a barrier nothing
 * arrives on.  The bounded wait gives up after 100 ms and sets
 * PKV_DEV_WAIT_TIMEOUT, as a decode kernel does when a tile copy is lost; the
 * kernel then returns and the context stays usable.  Until
 * pkv_read_device_status clears the word, decode and varlen calls write
 * nothing.  Asynchronous on stream; no memory is touched but the status word.
 */
pkv_status pkv_selftest_wait_timeout(void* stream);

/*
 * pkv_splitk_scratch_bytes — bytes of scratch pkv_decode_splitk needs for S
 * splits: a 256-byte header (the chunk size phase 1 chose, read by the
 * combine), f32 partial outputs [num_seqs][num_heads][S][head_dim], then f32
 * running max and running sum [num_seqs][num_heads][S] each (every part
 * 256-byte aligned).  0 when S is 0 or 1 or for invalid sizes.
 * (ferrum-kernels paged.rs keeps these three buffers process-global and grows
 * them on demand; here the caller owns them.)
 */
size_t pkv_splitk_scratch_bytes(int32_t num_seqs, int32_t num_heads, int32_t head_dim,
                                int32_t num_splits);

/*
 * pkv_pick_num_splits — the split count pkv_decode_splitk uses when given 0
 * (ferrum-kernels paged.rs, paged_batched_flash_dispatch: the grid wants
 * enough CTAs to fill the SMs; once the base grid saturates them, splitting
 * pays only for long contexts).  Here the base grid is num_seqs *
 * num_kv_heads (one CTA per sequence and KV head covers the whole group),
 * measured against num_sms x 2 resident CTAs.  max_context_len is the
 * longest context the call may see (pkv_decode_splitk passes
 * max_blocks_per_seq * block_size; the host never reads context_lens).
 * Below one wave: the split count that brings the grid nearest one wave;
 * at or above it: ceil(max_context_len / 2048); either capped at
 * max_context_len / 256, the block count and 64.  Returns 1 (single pass)
 * or a split count in 2..64; 1 for invalid sizes.
 */
int32_t pkv_pick_num_splits(int32_t num_seqs, int32_t num_kv_heads,
                            int32_t max_context_len, int32_t block_size,
                            int32_t num_sms);

/*
 * pkv_decode_splitk_plan — what pkv_decode_splitk (and pkv_append_decode,
 * pkv_decode_vllm_layout, pkv_qkv_norm_rope_append_decode) will launch for
 * these sizes and num_splits, so a caller can size its scratch without
 * repeating the library's rules (ferrum-kernels src/backend/cuda/paged.rs
 * sizes its process-global split scratch from the split count it picks;
 * here the caller sizes it).
 *
 *   *splits         1 (single pass) or the split count launched
 *                   (2..PKV_MAX_SPLITS; num_splits capped at
 *                   max_blocks_per_seq)
 *   *scratch_bytes  the scratch that call needs (0 for single pass)
 *
 * num_splits = 0 applies pkv_pick_num_splits for the current GPU (the one
 * query this makes to CUDA, for the SM count); no other CUDA call.  Returns
 * PKV_ERR_INVALID_ARG for null outputs, invalid sizes or num_splits outside
 * 0..PKV_MAX_SPLITS.
 */
pkv_status pkv_decode_splitk_plan(int32_t num_seqs, int32_t num_heads, int32_t num_kv_heads,
                                  int32_t head_dim, int32_t max_blocks_per_seq,
                                  int32_t block_size, int32_t num_splits, int32_t* splits,
                                  size_t* scratch_bytes);

/*
 * pkv_varlen_splitk_plan — the same for pkv_varlen_attention_splitk (and its
 * vLLM-layout twin): *splits is 1 or the split count launched, and
 * *scratch_bytes the scratch needed (0 when unsplit or when the call has no
 * queries).  num_splits 0..PKV_MAX_SPLITS (0 = the pick of
 * pkv_varlen_attention_splitk on the current GPU: pkv_varlen_pick_num_splits,
 * or the chunked-prefill rule for those sizes).
 */
pkv_status pkv_varlen_splitk_plan(int32_t num_seqs, int32_t total_q, int32_t max_q_len,
                                  int32_t num_heads, int32_t num_kv_heads, int32_t head_dim,
                                  int32_t max_blocks_per_seq, int32_t block_size,
                                  int32_t num_splits, int32_t* splits, size_t* scratch_bytes);

/*
 * pkv_decode_splitk_noalloc — pkv_decode_splitk without caller scratch and
 * without any allocation, for callers that cannot allocate device memory: a
 * plugin or extension whose host hands it only the input and output buffers
 * and owns every allocation itself, or a decode loop under a latency budget
 * where cudaMalloc (which can block and synchronize the device) is not
 * allowed.  The pages have no counterpart; it is an addition of this library.
 *
 * The split-K partials live in one static device buffer of
 * PKV_NOALLOC_SCRATCH_BYTES that the library declares; every GPU that loads
 * the library holds it until the process exits.  The first call on a device
 * looks up that buffer's device address (cudaGetSymbolAddress, with the
 * device current) and caches it; make that first call before any stream
 * capture.  Nothing in the buffer needs to start at zero: phase 1 writes
 * every partial the combine reads.  All calls share the one buffer, which
 * keeps the last call's contents, so calls that may overlap on the GPU (on
 * different streams, or from different host threads) race and must not be
 * issued; calls on one stream are ordered and safe.
 *
 * Arguments and result are those of pkv_decode_splitk (num_splits 0 = the
 * heuristic, 1 = single pass).  Returns PKV_ERR_SCRATCH_TOO_SMALL, before any
 * launch, when the partials for the chosen split count need more than
 * PKV_NOALLOC_SCRATCH_BYTES (pkv_decode_splitk_plan gives the need); call
 * pkv_decode_splitk with caller-owned scratch, or fewer splits, instead.
 */
#define PKV_NOALLOC_SCRATCH_BYTES (8u * 1024u * 1024u)
pkv_status pkv_decode_splitk_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                     const int32_t* block_tables, const int32_t* context_lens,
                                     int32_t num_seqs, int32_t max_blocks_per_seq,
                                     int32_t num_blocks, float scale, int32_t num_heads,
                                     int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                                     void* out, int32_t num_splits, void* stream);

/* Static text for a status code (never NULL). */
const char* pkv_status_string(pkv_status status);

/* The message of the last failed call on this host thread ("" if none).
 * Valid until the next failing call on the thread. */
const char* pkv_last_error(void);

/*
 * pkv_read_device_status — copy the current GPU's status word (PKV_DEV_* bits
 * OR-ed by kernels since the last read) into *flags and clear it.  Enqueued
 * on stream and then synchronizes that stream: for tests and diagnostics,
 * not for the decode loop.
 */
pkv_status pkv_read_device_status(int32_t* flags, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDKV_H */
