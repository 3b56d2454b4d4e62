/*
 * A plain C99 consumer of include/mla.h: it compiles with -std=c99 -pedantic, links against
 * the library, and exercises the host-side argument checks (no call reaches a kernel, so
 * it runs without a GPU).  Exit status 0 when every check behaves as the header states.
 */
#include <stdio.h>
#include <string.h>

#include "mla.h"

static int expect(mla_status got, mla_status want, const char* what) {
  if (got != want) {
    fprintf(stderr, "%s: status %d, expected %d (%s)\n", what, (int)got, (int)want, mla_last_error());
    return 1;
  }
  return 0;
}

int main(void) {
  /* any 16-byte aligned, non-null address: the checks below never dereference it */
  static float dummy[64] __attribute__((aligned(16)));
  void* d = dummy;
  float* f = dummy;
  int bad = 0;

  bad += expect(mla_prefill(NULL, d, d, d, d, NULL, NULL, d, f, 1, 1, 1, 128, 64, 128, 0.1f, 1,
                            MLA_BF16, MLA_BF16, NULL),
                MLA_ERR_INVALID_ARG, "prefill: null q_nope");
  bad += expect(mla_prefill(d, d, d, d, d, NULL, NULL, d, f, 1, 1, 1, 64, 64, 128, 0.1f, 1,
                            MLA_BF16, MLA_BF16, NULL),
                MLA_ERR_UNSUPPORTED, "prefill: d_nope 64");
  bad += expect(mla_prefill(d, d, d, d, d, NULL, NULL, d, f, 1, 1, 1, 128, 64, 128, 0.1f, 1,
                            MLA_FP8_E4M3, MLA_FP32, NULL),
                MLA_ERR_INVALID_ARG, "prefill: fp8 without scales");
  bad += expect(mla_decode(d, d, d, NULL, (const int*)d, (const int*)d, d, f, 1, 16, 1, 512, 64,
                           32, 1, 1, 0.1f, 1, MLA_BF16, NULL, 0, NULL),
                MLA_ERR_UNSUPPORTED, "decode: page size 32");
  bad += expect(mla_decode(d, d, d, f, (const int*)d, (const int*)d, d, f, 1, 16, 1, 512, 64,
                           64, 1, 1, 0.1f, 1, MLA_BF16, NULL, 0, NULL),
                MLA_ERR_INVALID_ARG, "decode: bf16 cache with scales");
  bad += expect(mla_absorb(d, d, d, 4, 2, 96, 128, NULL), MLA_ERR_UNSUPPORTED, "absorb: K = 96");
  if (mla_version() <= 0) {
    fprintf(stderr, "mla_version: %d\n", mla_version());
    ++bad;
  }
  if (strlen(mla_last_error()) == 0) {
    fprintf(stderr, "mla_last_error: empty after a rejected call\n");
    ++bad;
  }
  return bad ? 1 : 0;
}
