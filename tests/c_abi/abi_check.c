/* abi_check.c -- a plain C11 program that includes the public header and
 * links libspecverify.so, to show the boundary is usable from C alone.  It
 * only makes calls that the library answers on the host (sizes, argument
 * errors, empty batches), so it runs without a GPU.  Exit status 0 = every
 * check passed; otherwise the number of the first failed check. */
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "spec_verify.h"

#define CHECK(n, cond)                                  \
  do {                                                  \
    if (!(cond)) {                                      \
      fprintf(stderr, "abi_check: check %d failed\n", n); \
      return n;                                         \
    }                                                   \
  } while (0)

int main(void) {
  void* fake = (void*)(uintptr_t)(1u << 20); /* never dereferenced */
  float* ffake = (float*)fake;
  int32_t* ifake = (int32_t*)fake;
  double* dfake = (double*)fake;

  /* workspace sizes: multiples of 256, growing with the batch; 0 when invalid */
  size_t w1 = spec_verify_workspace_size(64, 5, 128256, SPEC_DTYPE_BF16, SPEC_MODE_SAMPLE);
  size_t w2 = spec_verify_workspace_size(128, 5, 128256, SPEC_DTYPE_BF16, SPEC_MODE_SAMPLE);
  CHECK(1, w1 > 0 && w1 % 256 == 0 && w2 >= w1);
  CHECK(2, spec_verify_workspace_size(-1, 5, 1000, SPEC_DTYPE_F32, SPEC_MODE_SAMPLE) == 0);
  CHECK(3, spec_verify_workspace_size(4, SPEC_MAX_K + 1, 1000, SPEC_DTYPE_F32, SPEC_MODE_SAMPLE) == 0);
  CHECK(4, spec_verify_workspace_size(4, 4, 1000, 7, SPEC_MODE_SAMPLE) == 0);

  /* argument errors return before any launch */
  CHECK(5, spec_verify(fake, fake, ifake, ffake, 4, 4, 1000, SPEC_DTYPE_F32, 0.0f,
                       SPEC_MODE_SAMPLE, ifake, ifake, fake, w1, NULL) == SPEC_ERR_INVALID_ARG);
  CHECK(6, spec_verify(fake, fake, ifake, ffake, 4, 4, 1000, SPEC_DTYPE_F32, 1.0f, 9, ifake, ifake,
                       fake, w1, NULL) == SPEC_ERR_INVALID_ARG);
  CHECK(7, spec_verify(fake, fake, ifake, ffake, 0, 4, 1000, SPEC_DTYPE_F32, 1.0f,
                       SPEC_MODE_SAMPLE, ifake, ifake, fake, w1, NULL) == SPEC_OK);
  CHECK(8, spec_draft_sample(fake, ffake, -1, 1000, SPEC_DTYPE_F32, 1.0f, ifake, NULL, fake, w1,
                             NULL, NULL) == SPEC_ERR_INVALID_ARG);
  CHECK(9, spec_verify_scd(fake, fake, ifake, ffake, 4, 4, 1024, SPEC_DTYPE_F32, 1.0f, 1.5,
                           ifake, ifake, fake, w1, NULL, NULL, NULL, NULL,
                           NULL) == SPEC_ERR_INVALID_ARG);
  CHECK(10, spec_verify_scd(fake, fake, ifake, ffake, 0, 4, 1024, SPEC_DTYPE_F32, 1.0f, 0.1,
                            ifake, ifake, fake, w1, NULL, NULL, NULL, NULL, NULL) == SPEC_OK);
  CHECK(11, spec_rejection_cut(ffake, 4, 0, 0.5, dfake, ifake, ifake, NULL, NULL) ==
                SPEC_ERR_INVALID_ARG);
  CHECK(12, spec_rejection_cut(ffake, 0, 1000, 0.5, dfake, ifake, ifake, NULL, NULL) == SPEC_OK);
  CHECK(13, spec_rejection_cut(ffake, 4, 1000, -0.5, dfake, ifake, ifake, NULL, NULL) ==
                SPEC_ERR_INVALID_ARG);

  /* every return code has a description */
  CHECK(14, strcmp(spec_status_string(SPEC_OK), "ok") == 0);
  for (int c = SPEC_OK; c <= SPEC_ERR_SCRATCH_LIMIT; ++c)
    CHECK(15, spec_status_string(c) != NULL && spec_status_string(c)[0] != '\0');
  /* the wait bound: set, and back to the default */
  CHECK(16, spec_set_wait_limit(5000u) == SPEC_OK);
  CHECK(17, spec_set_wait_limit(0u) == SPEC_OK);
  printf("abi_check: all checks passed\n");
  return 0;
}
