/*
 * A plain C client of the library's C ABI: no C++, no torch, only the header
 * and the shared library.  It checks the version, the error strings, the
 * host-side argument checks and the empty-problem fast path; with
 * --no-device (a machine without a usable GPU) it also checks that a valid
 * call returns an error code instead of computing anywhere else, since the
 * library has no CPU path.  Prints OK and exits 0 when every check passes.
 */
#include <stdalign.h>
#include <stdio.h>
#include <string.h>

#include "attn.h"

static int fails = 0;
#define CHECK(c)                                                     \
  do {                                                               \
    if (!(c)) {                                                      \
      printf("FAIL %s:%d %s\n", __FILE__, __LINE__, #c);             \
      ++fails;                                                       \
    }                                                                \
  } while (0)

int main(int argc, char **argv) {
  const int no_device = argc > 1 && strcmp(argv[1], "--no-device") == 0;
  static alignas(16) unsigned char buf[4096];
  void *p = buf;
  float *lp = (float *)buf;
  attn_plan plan;

  CHECK(attn_version() == 100);
  CHECK(strlen(attn_strerror(ATTN_ERR_ARG)) > 0);
  CHECK(strstr(attn_strerror(-99), "unknown") != NULL);

  /* sizes, flags, scale, pointers and alignment are checked on the host */
  CHECK(attn_fwd(p, p, p, p, lp, 1, 2, 1, 8, 8, 65, 0.125f, 0, NULL) == ATTN_ERR_ARG);
  CHECK(attn_fwd(p, p, p, p, lp, 1, 2, 1, 8, 8, 1088, 0.125f, 0, NULL) == ATTN_ERR_ARG);
  CHECK(attn_fwd(p, p, p, p, lp, 1, 3, 2, 8, 8, 64, 0.125f, 0, NULL) == ATTN_ERR_ARG);
  CHECK(attn_fwd(p, p, p, p, lp, 1, 2, 1, 8, 8, 64, 0.125f, 2, NULL) == ATTN_ERR_ARG);
  CHECK(attn_fwd(NULL, p, p, p, lp, 1, 2, 1, 8, 8, 64, 0.125f, 0, NULL) == ATTN_ERR_ARG);
  CHECK(attn_fwd(buf + 2, p, p, p, lp, 1, 2, 1, 8, 8, 64, 0.125f, 0, NULL) == ATTN_ERR_ALIGN);
  CHECK(attn_fwd_splitkv(p, p, p, p, lp, 1, 2, 1, 8, 8, 64, 0.125f, 0, 65, NULL) == ATTN_ERR_ARG);
  CHECK(attn_fwd_splitkv_noalloc(p, p, p, p, lp, 1, 2, 1, 8, 8, 64, 0.125f, 0, 0, NULL) == ATTN_ERR_ARG);
  CHECK(attn_fwd_plan(1, 2, 1, 8, 8, 65, 0, &plan) == ATTN_ERR_ARG);
  CHECK(attn_set_debug(8, 0) == ATTN_ERR_ARG);

  /* an empty problem succeeds without touching a device */
  CHECK(attn_fwd(NULL, NULL, NULL, NULL, NULL, 0, 2, 1, 8, 8, 64, 0.125f, 0, NULL) == ATTN_OK);
  CHECK(attn_fwd(NULL, NULL, NULL, NULL, NULL, 1, 2, 1, 0, 8, 64, 0.125f, 0, NULL) == ATTN_OK);

  if (no_device) {
    const int rc = attn_fwd(p, p, p, p, lp, 1, 2, 1, 8, 8, 64, 0.125f, 0, NULL);
    CHECK(rc == ATTN_ERR_LAUNCH || rc == ATTN_ERR_ARCH);
    CHECK(rc != ATTN_ERR_LAUNCH || strlen(attn_last_cuda_error()) > 0);
    CHECK(attn_fwd_plan(1, 2, 1, 8, 8, 64, 0, &plan) < 0);
  }
  printf("%s (%d failures)\n", fails ? "FAILED" : "OK", fails);
  return fails ? 1 : 0;
}
