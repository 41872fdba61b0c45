/* A C99 program written against include/vt_paged_attn.h alone: it includes
 * the header, links the library and runs the calls that need no GPU (the
 * version, status strings and every check that rejects arguments on the host
 * before CUDA is touched).  Exit status 0 and "c abi: ok" when all hold. */
#include <stdio.h>
#include <string.h>

#include "vt_paged_attn.h"

static int failures = 0;

#define CHECK(cond)                                                  \
  do {                                                               \
    if (!(cond)) {                                                   \
      printf("FAIL %s:%d: %s\n", __FILE__, __LINE__, #cond);         \
      ++failures;                                                    \
    }                                                                \
  } while (0)

int main(void) {
  /* stand-in device addresses: never dereferenced, every call below returns
   * from its host-side checks */
  void* out = (void*)0x1000;
  const void* q = (const void*)0x2000;
  const void* kc = (const void*)0x3000;
  const void* vc = (const void*)0x4000;
  const int32_t* bt = (const int32_t*)0x5000;
  const int32_t* cl = (const int32_t*)0x6000;
  const float* ks = (const float*)0x7000;
  const float* vs = (const float*)0x7100;
  vt_plan plan;

  CHECK(vt_paged_attn_version() == 10100);
  CHECK(strcmp(vt_status_string(VT_OK), "ok") == 0);
  CHECK(vt_status_string(VT_ERR_UNSUPPORTED) != NULL);

  /* empty batch: a no-op */
  CHECK(vt_paged_attn_decode(NULL, NULL, kc, vc, bt, cl, 0, 16, 8, 128, 32, 0.088f, 0, NULL, 4, 16, VT_BF16) ==
        VT_OK);
  /* misaligned q, bad group, unsupported head_dim and block size */
  CHECK(vt_paged_attn_decode(out, (const void*)0x2008, kc, vc, bt, cl, 2, 16, 8, 128, 32, 0.088f, 0, NULL, 4, 16,
                             VT_BF16) == VT_ERR_INVALID_ARG);
  CHECK(vt_paged_attn_decode(out, q, kc, vc, bt, cl, 2, 12, 8, 128, 32, 0.088f, 0, NULL, 4, 16, VT_BF16) ==
        VT_ERR_INVALID_ARG);
  CHECK(vt_paged_attn_decode(out, q, kc, vc, bt, cl, 2, 16, 8, 96, 32, 0.088f, 0, NULL, 4, 16, VT_BF16) ==
        VT_ERR_UNSUPPORTED);
  CHECK(vt_paged_attn_decode(out, q, kc, vc, bt, cl, 2, 16, 8, 128, 16, 0.088f, 0, NULL, 4, 16, VT_BF16) ==
        VT_ERR_UNSUPPORTED);
  CHECK(vt_paged_attn_decode_noalloc(out, q, kc, vc, bt, NULL, 2, 16, 8, 128, 32, 0.088f, 0, NULL, 4, 16,
                                     VT_BF16) == VT_ERR_INVALID_ARG);
  /* FP8: scales are required; head_dim 512 is not taken */
  CHECK(vt_paged_attn_decode_fp8(out, q, kc, vc, NULL, vs, bt, cl, 2, 16, 8, 128, 32, 0.088f, 0, NULL, 4, 16) ==
        VT_ERR_INVALID_ARG);
  CHECK(vt_paged_attn_decode_fp8(out, q, kc, vc, ks, vs, bt, cl, 2, 16, 8, 512, 32, 0.088f, 0, NULL, 4, 16) ==
        VT_ERR_UNSUPPORTED);
  /* several new tokens: q_len >= 1, and an FP8 cache only through its entry */
  CHECK(vt_paged_attn_decode_multi(out, q, kc, vc, bt, cl, 2, 0, 16, 8, 128, 32, 0.088f, 0, NULL, 4, 16,
                                   VT_BF16) == VT_ERR_INVALID_ARG);
  CHECK(vt_paged_attn_decode_multi(out, q, kc, vc, bt, cl, 2, 3, 16, 8, 128, 32, 0.088f, 0, NULL, 4, 16,
                                   VT_E4M3) == VT_ERR_INVALID_ARG);
  CHECK(vt_paged_attn_decode_multi_fp8(out, q, kc, vc, ks, vs, bt, cl, 2, 0, 16, 8, 128, 32, 0.088f, 0, NULL, 4,
                                       16) == VT_ERR_INVALID_ARG);
  /* settings */
  CHECK(vt_paged_attn_set_override(-1, 0) == VT_ERR_INVALID_ARG);
  CHECK(vt_paged_attn_set_override(0, 0) == VT_OK);
  CHECK(vt_paged_attn_set_overlap(2) == VT_ERR_INVALID_ARG);
  CHECK(vt_paged_attn_set_segment_cost(65) == VT_ERR_INVALID_ARG);
  CHECK(vt_paged_attn_set_segment_cost(-1) == VT_OK);
  CHECK(vt_paged_attn_set_test_wait(1000, -1, 3) == VT_ERR_INVALID_ARG);
  CHECK(vt_paged_attn_set_workspace((void*)0x1010, 1u << 20, NULL) == VT_ERR_INVALID_ARG);
  /* nothing has been launched on this thread */
  CHECK(vt_paged_attn_last_plan(&plan) == VT_ERR_INVALID_ARG);
  CHECK(vt_paged_attn_last_plan(NULL) == VT_ERR_INVALID_ARG);
  CHECK(vt_paged_attn_workspace_bytes(4, 12, 8, 128, VT_BF16) == 0);

  printf("%s\n", failures ? "c abi: FAIL" : "c abi: ok");
  return failures ? 1 : 0;
}
