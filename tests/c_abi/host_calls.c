/* A plain C99 caller of libpagedkv: includes the header, links the shared
 * library and exercises the host-only entry points (no GPU needed).  Prints
 * one line per check and exits non-zero on the first failure. */
#include <stdio.h>
#include <string.h>

#include "pagedkv.h"

#define CHECK(cond)                                   \
  do {                                                \
    if (!(cond)) {                                    \
      printf("FAIL %s (line %d)\n", #cond, __LINE__); \
      return 1;                                       \
    }                                                 \
    printf("ok %s\n", #cond);                         \
  } while (0)

int main(void) {
  /* split heuristics: host arithmetic only */
  CHECK(pkv_pick_num_splits(32, 8, 2048, 16, 152) == 1);
  CHECK(pkv_pick_num_splits(4, 8, 131072, 16, 152) > 1);
  CHECK(pkv_pick_num_splits(0, 8, 2048, 16, 152) == 1);
  CHECK(pkv_varlen_pick_num_splits(4, 32, 8, 4, 8192, 16, 152) == 10);
  /* the varlen kernel switch: initially the mma.sync kernel; bad values
     change nothing */
  CHECK(pkv_set_varlen_tensor_path(1) == 0);
  CHECK(pkv_set_varlen_tensor_path(2) == -1);
  CHECK(pkv_set_varlen_tensor_path(0) == 1);
  CHECK(pkv_set_varlen_tensor_path(-1) == -1);
  /* scratch sizes */
  CHECK(pkv_splitk_scratch_bytes(4, 32, 128, 1) == 0);
  CHECK(pkv_splitk_scratch_bytes(4, 32, 128, 16) >= (size_t)4 * 32 * 16 * 130 * 4);
  /* split plans: what the decode calls launch and the scratch they need */
  {
    int32_t S = 0;
    size_t need = 0;
    CHECK(pkv_decode_splitk_plan(4, 32, 8, 128, 8192, 16, 16, &S, &need) == PKV_OK);
    CHECK(S == 16 && need == pkv_splitk_scratch_bytes(4, 32, 128, 16));
    CHECK(pkv_decode_splitk_plan(3, 8, 2, 64, 7, 16, 64, &S, &need) == PKV_OK);
    CHECK(S == 7 && need == pkv_splitk_scratch_bytes(3, 8, 64, 7));
    CHECK(pkv_decode_splitk_plan(4, 32, 8, 128, 8192, 16, 1, &S, &need) == PKV_OK);
    CHECK(S == 1 && need == 0);
    CHECK(pkv_decode_splitk_plan(4, 32, 8, 128, 8192, 16, 200, &S, &need) ==
          PKV_ERR_INVALID_ARG);
    CHECK(pkv_decode_splitk_plan(4, 32, 8, 128, 8192, 16, 4, NULL, &need) ==
          PKV_ERR_INVALID_ARG);
    CHECK(pkv_varlen_splitk_plan(4, 16, 4, 32, 8, 128, 8192, 16, 10, &S, &need) == PKV_OK);
    CHECK(S == 10 && need == pkv_splitk_scratch_bytes(16, 32, 128, 10));
  }
  /* status strings */
  CHECK(strcmp(pkv_status_string(PKV_OK), "ok") == 0);
  CHECK(strlen(pkv_status_string(PKV_ERR_SCRATCH_TOO_SMALL)) > 0);
  /* argument validation returns before any CUDA call */
  CHECK(pkv_decode(NULL, NULL, NULL, NULL, NULL, 1, 1, 1, 0.125f, 4, 2, 64, 16, NULL, NULL) ==
        PKV_ERR_INVALID_ARG);
  CHECK(strlen(pkv_last_error()) > 0);
  CHECK(pkv_append((void*)0x10000, (void*)0x10000, (const int32_t*)0x10000, 0, (void*)0x10000,
                   (void*)0x10000, 8, 16, 2, 64, NULL) == PKV_OK);
  /* every other compute entry, called through its C prototype with a NULL
   * input: rejected on the host, nothing launched */
  CHECK(pkv_decode_splitk(NULL, NULL, NULL, NULL, NULL, 1, 1, 1, 0.125f, 4, 2, 64, 16, NULL, 0,
                          NULL, 0, NULL) == PKV_ERR_INVALID_ARG);
  CHECK(pkv_append_decode(NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, 1, 1, 1, 0.125f, 4, 2,
                          64, 16, NULL, 0, NULL, 0, NULL) == PKV_ERR_INVALID_ARG);
  CHECK(pkv_varlen_attention(NULL, NULL, NULL, NULL, NULL, NULL, 1, 1, 1, 1, 1, 0.125f, 4, 2, 64,
                             16, NULL, NULL) == PKV_ERR_INVALID_ARG);
  CHECK(pkv_varlen_attention_vllm_layout(NULL, NULL, NULL, NULL, NULL, NULL, 1, 1, 1, 1, 1, 0.125f,
                                         4, 2, 64, 16, NULL, NULL) == PKV_ERR_INVALID_ARG);
  CHECK(pkv_varlen_attention_splitk(NULL, NULL, NULL, NULL, NULL, NULL, 1, 1, 1, 1, 1, 0.125f, 4,
                                    2, 64, 16, NULL, 0, NULL, 0, NULL) == PKV_ERR_INVALID_ARG);
  CHECK(pkv_varlen_attention_splitk_vllm_layout(NULL, NULL, NULL, NULL, NULL, NULL, 1, 1, 1, 1, 1,
                                                0.125f, 4, 2, 64, 16, NULL, 0, NULL, 0,
                                                NULL) == PKV_ERR_INVALID_ARG);
  CHECK(pkv_append_vllm_layout(NULL, NULL, NULL, 1, NULL, NULL, 8, 16, 2, 64, NULL) ==
        PKV_ERR_INVALID_ARG);
  CHECK(pkv_decode_vllm_layout(NULL, NULL, NULL, NULL, NULL, 1, 1, 1, 0.125f, 4, 2, 64, 16, NULL,
                               0, NULL, 0, NULL) == PKV_ERR_INVALID_ARG);
  CHECK(pkv_decode_splitk_noalloc(NULL, NULL, NULL, NULL, NULL, 1, 1, 1, 0.125f, 4, 2, 64, 16,
                                  NULL, 0, NULL) == PKV_ERR_INVALID_ARG);
  CHECK(pkv_qkv_norm_rope_append(NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL,
                                 1, 1, 1, 8, 4, 2, 64, 16, 100, 1e-6f, NULL) ==
        PKV_ERR_INVALID_ARG);
  CHECK(pkv_qkv_norm_rope_append_decode(NULL, NULL, NULL, NULL, NULL, 100, 1e-6f, NULL, NULL, NULL,
                                        NULL, 1, 1, 8, 0.125f, 4, 2, 64, 16, NULL, 0, NULL, 0,
                                        NULL) == PKV_ERR_INVALID_ARG);
  CHECK(pkv_read_device_status(NULL, NULL) == PKV_ERR_INVALID_ARG);
  printf("all ok\n");
  return 0;
}
