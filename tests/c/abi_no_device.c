/*
 * Plain C99 client of libswiglu: compiles against include/swiglu.h alone (no
 * CUDA or C++ headers) and calls the entry points that need no GPU. Exits 0
 * when every check holds; prints the failing check otherwise.
 */
#include <stdio.h>
#include <string.h>

#include "swiglu.h"

static int failures = 0;
#define CHECK(cond)                                          \
  do {                                                       \
    if (!(cond)) {                                           \
      fprintf(stderr, "check failed: %s (line %d)\n", #cond, __LINE__); \
      ++failures;                                            \
    }                                                        \
  } while (0)

int main(void) {
  /* packed sizes: 2 matrices x Np x Kp x 2 bytes, Np to 128, Kp to 64 */
  CHECK(swiglu_packed_weight_bytes(64, 128) == (size_t)2 * 128 * 64 * 2);
  CHECK(swiglu_packed_weight_bytes(72, 136) == (size_t)2 * 256 * 128 * 2);
  CHECK(swiglu_packed_weight_bytes(0, 128) == 0);
  CHECK(swiglu_packed_weight_bytes(64, -8) == 0);
  CHECK(swiglu_packed_weight_bytes_fp8(128, 128) == (size_t)2 * 128 * 128);
  CHECK(swiglu_down_packed_bytes(64, 256) == (size_t)256 * 64 * 2);
  /* status strings exist for every code */
  for (int c = SWIGLU_OK; c <= SWIGLU_ERR_NO_DEVICE; ++c) {
    const char* s = swiglu_status_string((swiglu_status_t)c);
    CHECK(s != NULL && strlen(s) > 0);
  }
  /* argument errors come before any device access */
  char buf[64];
  CHECK(swiglu_plan_string(16, 64, 64, 0, NULL, 0) == SWIGLU_ERR_INVALID_ARG);
  CHECK(swiglu_forward(NULL, NULL, NULL, 4, 64, 64, NULL) == SWIGLU_ERR_INVALID_ARG);
  CHECK(swiglu_forward((void*)0x10000, (void*)0x20000, (void*)0x30000, 4, 60, 64, NULL) ==
        SWIGLU_ERR_UNSUPPORTED); /* K % 8 */
  CHECK(swiglu_forward((void*)0x10000, (void*)0x20000, (void*)0x30000, 0, 64, 64, NULL) ==
        SWIGLU_OK); /* M = 0: nothing to do */
  (void)buf;
  if (failures == 0) printf("c abi ok\n");
  return failures == 0 ? 0 : 1;
}
