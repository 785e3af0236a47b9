/* End-to-end decode steps from plain C: the Llama-3-8B-shaped workload
 * (B = 32 sequences, H = 32, Hkv = 8, D = 128, block size 16, context
 * lengths uniform in [512, 2048], tables drawn without replacement from a
 * 16384-block pool) driven through the C ABI with host buffers, as a serving
 * loop written in C would drive it.  Each step copies its inputs (q, the new
 * K/V rows, slots, tables, lengths), packed in one pinned host buffer, to
 * the device, calls pkv_append_decode, and copies the output back to pinned
 * memory.
 *
 * Printed (one JSON line): the host time spent inside pkv_append_decode per
 * call (the library's own cost: validation, tensor maps, the launch), the
 * device time per step (CUDA events around the copy-step-copy chain of back-
 * to-back steps), and the wall time per step with a stream synchronisation
 * after each step.  Then the same steps without the two copies: the kernels
 * read the inputs from, and write the output to, the pinned host buffers
 * directly over the host link (zero-copy; the pools stay in device memory),
 * and the outputs of both forms are compared bit for bit.  Exits non-zero
 * on any error.
 *
 * usage: e2e_step [steps] [warmup]
 */
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>
#include <time.h>

#include "pagedkv.h"

#define CK(x)                                                                    \
  do {                                                                           \
    cudaError_t e_ = (x);                                                        \
    if (e_ != cudaSuccess) {                                                     \
      fprintf(stderr, "%s:%d %s: %s\n", __FILE__, __LINE__, #x,                  \
              cudaGetErrorString(e_));                                           \
      return 1;                                                                  \
    }                                                                            \
  } while (0)

enum { B = 32, H = 32, HKV = 8, D = 128, BS = 16, NB = 16384, MBPS = 128 };

static uint64_t rng_state = 0x2026120212345ull;
static uint32_t rng_next(void) { /* xorshift64* */
  rng_state ^= rng_state >> 12;
  rng_state ^= rng_state << 25;
  rng_state ^= rng_state >> 27;
  return (uint32_t)((rng_state * 0x2545F4914F6CDD1Dull) >> 32);
}

/* An f16 bit pattern of a value in (-1, 1): sign, a small exponent range and
 * a random mantissa (normal numbers only; the timing does not depend on the
 * values). */
static uint16_t rand_half(void) {
  const uint32_t r = rng_next();
  const uint16_t sign = (uint16_t)((r >> 31) << 15);
  const uint16_t expo = (uint16_t)(10 + (r >> 26) % 4); /* 2^-5 .. 2^-2 */
  return (uint16_t)(sign | (expo << 10) | (r & 0x3ff));
}

static double now_us(void) {
  struct timespec ts;
  clock_gettime(CLOCK_MONOTONIC, &ts);
  return ts.tv_sec * 1e6 + ts.tv_nsec / 1e3;
}

static int cmp_double(const void* a, const void* b) {
  const double x = *(const double*)a, y = *(const double*)b;
  return (x > y) - (x < y);
}

int main(int argc, char** argv) {
  const int steps = argc > 1 ? atoi(argv[1]) : 200;
  const int warmup = argc > 2 ? atoi(argv[2]) : 20;
  if (steps <= 0 || warmup < 0) return 2;

  /* host inputs: lengths, tables (a permutation of the pool), slots of the
   * newest positions, q and the new K/V rows */
  int32_t lens[B];
  int32_t* perm = (int32_t*)malloc(sizeof(int32_t) * NB);
  for (int i = 0; i < NB; ++i) perm[i] = i;
  for (int i = NB - 1; i > 0; --i) {
    const int j = (int)(rng_next() % (uint32_t)(i + 1));
    const int32_t t = perm[i];
    perm[i] = perm[j];
    perm[j] = t;
  }
  const size_t q_bytes = (size_t)B * H * D * 2, kv_bytes = (size_t)B * HKV * D * 2;
  const size_t tab_bytes = (size_t)B * MBPS * 4;
  const size_t off_q = 0, off_k = off_q + q_bytes, off_v = off_k + kv_bytes;
  const size_t off_slot = off_v + kv_bytes, off_tab = off_slot + 256;
  const size_t off_len = off_tab + tab_bytes, packed = off_len + 256;
  uint8_t* h_in = NULL;
  uint16_t* h_out = NULL;
  CK(cudaMallocHost((void**)&h_in, packed));
  CK(cudaMallocHost((void**)&h_out, q_bytes));
  memset(h_in, 0, packed);
  int32_t* tab = (int32_t*)(h_in + off_tab);
  int32_t* slots = (int32_t*)(h_in + off_slot);
  long long total_tokens = 0;
  int cur = 0;
  for (int s = 0; s < B; ++s) {
    lens[s] = 512 + (int)(rng_next() % 1537u);
    total_tokens += lens[s];
    const int nblk = (lens[s] + BS - 1) / BS;
    for (int j = 0; j < MBPS; ++j) tab[s * MBPS + j] = j < nblk ? perm[cur + j] : perm[NB - 1];
    cur += nblk;
    const int pos = lens[s] - 1;
    slots[s] = tab[s * MBPS + pos / BS] * BS + pos % BS;
  }
  memcpy(h_in + off_len, lens, sizeof(lens));
  uint16_t* hq = (uint16_t*)(h_in + off_q);
  for (size_t i = 0; i < q_bytes / 2; ++i) hq[i] = rand_half();
  uint16_t* hk = (uint16_t*)(h_in + off_k);
  for (size_t i = 0; i < 2 * kv_bytes / 2; ++i) hk[i] = rand_half(); /* k then v */

  /* device buffers: the pools (1 GB, filled with a finite constant), the
   * packed step inputs, the output and the split scratch of the plan */
  const size_t pool_bytes = (size_t)NB * HKV * BS * D * 2;
  void *k_cache = NULL, *v_cache = NULL, *d_in = NULL, *d_out = NULL, *scratch = NULL;
  CK(cudaMalloc(&k_cache, pool_bytes));
  CK(cudaMalloc(&v_cache, pool_bytes));
  CK(cudaMemset(k_cache, 0x2c, pool_bytes)); /* f16 0x2c2c = 0.0637 */
  CK(cudaMemset(v_cache, 0x2c, pool_bytes));
  CK(cudaMalloc(&d_in, packed));
  CK(cudaMalloc(&d_out, q_bytes));
  int32_t splits = 0;
  size_t scratch_bytes = 0;
  if (pkv_decode_splitk_plan(B, H, HKV, D, MBPS, BS, 0, &splits, &scratch_bytes) != PKV_OK) {
    fprintf(stderr, "plan: %s\n", pkv_last_error());
    return 1;
  }
  if (scratch_bytes) CK(cudaMalloc(&scratch, scratch_bytes));
  cudaStream_t st;
  CK(cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking));
  uint8_t* din = (uint8_t*)d_in;

  double* host_us = (double*)malloc(sizeof(double) * (size_t)steps);
  double* wall_us = (double*)malloc(sizeof(double) * (size_t)steps);
  cudaEvent_t ev0, ev1;
  CK(cudaEventCreate(&ev0));
  CK(cudaEventCreate(&ev1));
  /* phase 0: warm-up; 1: back-to-back steps between two events, the
   * library's host time per call measured around the call alone; 2: one
   * step at a time with a synchronisation (wall time per step) */
  for (int phase = 0; phase < 3; ++phase) {
    const int n = phase == 0 ? warmup : steps;
    if (phase == 1) CK(cudaEventRecord(ev0, st));
    for (int i = 0; i < n; ++i) {
      const double w0 = now_us();
      CK(cudaMemcpyAsync(d_in, h_in, packed, cudaMemcpyHostToDevice, st));
      const double t0 = now_us();
      const pkv_status rc = pkv_append_decode(
          din + off_k, din + off_v, (const int32_t*)(din + off_slot), k_cache, v_cache,
          din + off_q, (const int32_t*)(din + off_tab), (const int32_t*)(din + off_len), B, MBPS,
          NB, 0.08838834764831845f, H, HKV, D, BS, d_out, 0, scratch, scratch_bytes, st);
      const double t1 = now_us();
      if (rc != PKV_OK) {
        fprintf(stderr, "pkv_append_decode: %s: %s\n", pkv_status_string(rc), pkv_last_error());
        return 1;
      }
      CK(cudaMemcpyAsync(h_out, d_out, q_bytes, cudaMemcpyDeviceToHost, st));
      if (phase == 1) host_us[i] = t1 - t0;
      if (phase == 2) {
        CK(cudaStreamSynchronize(st));
        wall_us[i] = now_us() - w0;
      }
    }
    if (phase == 1) CK(cudaEventRecord(ev1, st));
    CK(cudaStreamSynchronize(st));
  }
  float ev_ms = 0.f;
  CK(cudaEventElapsedTime(&ev_ms, ev0, ev1));

  /* zero-copy: the same steps on the host buffers themselves (page-locked
   * host memory is addressable from the device with the same pointer) */
  uint16_t* h_out_zc = NULL;
  CK(cudaMallocHost((void**)&h_out_zc, q_bytes));
  for (int phase = 0; phase < 2; ++phase) {
    const int n = phase == 0 ? warmup : steps;
    if (phase == 1) CK(cudaEventRecord(ev0, st));
    for (int i = 0; i < n; ++i) {
      const pkv_status rc = pkv_append_decode(
          h_in + off_k, h_in + off_v, (const int32_t*)(h_in + off_slot), k_cache, v_cache,
          h_in + off_q, (const int32_t*)(h_in + off_tab), (const int32_t*)(h_in + off_len), B,
          MBPS, NB, 0.08838834764831845f, H, HKV, D, BS, h_out_zc, 0, scratch, scratch_bytes, st);
      if (rc != PKV_OK) {
        fprintf(stderr, "pkv_append_decode (zero-copy): %s: %s\n", pkv_status_string(rc),
                pkv_last_error());
        return 1;
      }
    }
    if (phase == 1) CK(cudaEventRecord(ev1, st));
    CK(cudaStreamSynchronize(st));
  }
  float zc_ms = 0.f;
  CK(cudaEventElapsedTime(&zc_ms, ev0, ev1));
  if (memcmp(h_out, h_out_zc, q_bytes) != 0) {
    fprintf(stderr, "zero-copy output differs from the copied one\n");
    return 1;
  }
  int32_t flags = -1;
  if (pkv_read_device_status(&flags, st) != PKV_OK || flags != 0) {
    fprintf(stderr, "device status flags %d\n", (int)flags);
    return 1;
  }
  /* the output must be finite f16 (exponent field not all ones) */
  for (size_t i = 0; i < q_bytes / 2; ++i)
    if ((h_out[i] & 0x7c00) == 0x7c00) {
      fprintf(stderr, "non-finite output at %zu\n", i);
      return 1;
    }
  qsort(host_us, (size_t)steps, sizeof(double), cmp_double);
  qsort(wall_us, (size_t)steps, sizeof(double), cmp_double);
  const double kv = (double)total_tokens * 2 * HKV * D * 2;
  const double step_us = 1e3 * ev_ms / steps;
  const double zc_us = 1e3 * zc_ms / steps;
  printf("{\"workload\": \"B=32 H=32 Hkv=8 D=128 bs=16 L~U[512,2048], 16384-block pool\", "
         "\"splits\": %d, \"steps\": %d, \"host_us_per_call_median\": %.2f, "
         "\"host_us_per_call_min\": %.2f, \"e2e_us_per_step\": %.2f, \"e2e_gbs\": %.1f, "
         "\"wall_us_per_step_median\": %.2f, \"h2d_bytes_per_step\": %zu, "
         "\"d2h_bytes_per_step\": %zu, \"zero_copy_us_per_step\": %.2f, "
         "\"zero_copy_gbs\": %.1f}\n",
         (int)splits, steps, host_us[steps / 2], host_us[0], step_us, kv / (step_us * 1e3),
         wall_us[steps / 2], packed, q_bytes, zc_us, kv / (zc_us * 1e3));
  return 0;
}
