/*
 * Calls the C ABI of include/spec_verify.h on every path that a host without
 * a usable GPU can reach -- status strings, launch counts, argument
 * validation of every entry point, a NULL handle, sizes outside the limits,
 * and a device call that fails -- so that the host side of the library can be
 * built and run under AddressSanitizer and UndefinedBehaviorSanitizer
 * (tests/test_abi_sanitized.py).  Every call checks its status code.
 */
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "spec_verify.h"

static int failures = 0;
#define EXPECT(call, want)                                                             \
  do {                                                                                 \
    const sv_status got_ = (call);                                                     \
    if (got_ != (want)) {                                                              \
      fprintf(stderr, "%s:%d: %s returned %d, expected %d\n", __FILE__, __LINE__, #call, \
              (int)got_, (int)(want));                                                 \
      ++failures;                                                                      \
    }                                                                                  \
  } while (0)

int main(void) {
  /* plain queries */
  for (int s = -2; s < 12; ++s) {
    const char* t = spec_verify_status_string((sv_status)s);
    if (t == NULL || t[0] == '\0') {
      fprintf(stderr, "status %d has no text\n", s);
      ++failures;
    }
  }
  if (strcmp(spec_verify_status_string(SV_OK), "ok") != 0) ++failures;
  if (spec_verify_launches_per_run() < 1 || spec_verify_launches_per_filtered_run() < 1) ++failures;

  /* init: bad arguments are rejected before any device call, the handle stays NULL */
  spec_verify_t h = (spec_verify_t)0;
  EXPECT(spec_verify_init(NULL, 4, 4, 100, 0), SV_EINVAL);
  EXPECT(spec_verify_init(&h, 0, 4, 100, 0), SV_EINVAL);
  EXPECT(spec_verify_init(&h, 4, 0, 100, 0), SV_EINVAL);
  EXPECT(spec_verify_init(&h, 4, 4, 0, 0), SV_EINVAL);
  EXPECT(spec_verify_init(&h, -3, 4, 100, 0), SV_EINVAL);
  EXPECT(spec_verify_init(&h, 4, SV_MAX_K + 1, 100, 0), SV_EUNSUPPORTED);
  EXPECT(spec_verify_init(&h, 4, 4, SV_MAX_V + 1, 0), SV_EUNSUPPORTED);
  if (h != NULL) ++failures;
  /* valid sizes but a device index that cannot exist: a CUDA failure, no handle */
  EXPECT(spec_verify_init(&h, 4, 4, 100, 1 << 20), SV_ECUDA);
  if (h != NULL) ++failures;
  /* device 0: a CUDA failure on a host without a GPU; a handle where there is one */
  {
    const sv_status s = spec_verify_init(&h, 2, 3, 1000, 0);
    if (s == SV_OK) {
      EXPECT(spec_verify_set_gate_policy(h, NULL, 0, 0.0f), SV_OK);
      EXPECT(spec_verify_free(h), SV_OK);
    } else if (s != SV_ECUDA) {
      fprintf(stderr, "init on device 0 returned %d\n", (int)s);
      ++failures;
    }
    h = (spec_verify_t)0;
  }

  /* every entry point with a NULL handle */
  float x[16] = {0};
  int32_t d[4] = {0}, len[4], tok[8];
  float ap[4], ms[4], pq[4], aq[4], stats[64];
  int8_t fl[4];
  uint64_t cnt[SV_NUM_COUNTERS];
  EXPECT(spec_verify_run(NULL, x, SV_F32, x, SV_F32, d, 1, 1.0f, SV_PLAIN, 0.5f, NULL, NULL, 1u, len, tok,
                         ap, fl, cnt, NULL),
         SV_EINVAL);
  EXPECT(spec_verify_run_ex(NULL, x, SV_F32, x, SV_BF16, d, 1, 1.0f, SV_GATED_MU, 0.5f, NULL, NULL, 1u, 0u,
                            NULL, NULL, len, tok, ap, fl, cnt, stats, NULL),
         SV_EINVAL);
  EXPECT(spec_verify_run_host(NULL, x, SV_F32, x, SV_F32, d, 1, 1.0f, SV_PLAIN, 0.5f, NULL, NULL, 1u, len,
                              tok, ap, fl, cnt, NULL),
         SV_EINVAL);
  EXPECT(spec_verify_diagnostics(NULL, x, SV_F32, x, SV_F32, d, 1, 1.0f, SV_PLAIN, 0.5f, NULL, NULL, ms, pq,
                                 aq, NULL),
         SV_EINVAL);
  const float sched[2] = {0.3f, 0.5f};
  EXPECT(spec_verify_set_gate_policy(NULL, sched, 2, 0.1f), SV_EINVAL);
  EXPECT(spec_verify_set_filters(NULL, 5, 0.9f, 0.0f, 0, 1.0f, 0.0f), SV_EINVAL);
  EXPECT(spec_verify_mark_next(NULL, NULL, NULL), SV_EINVAL);
  EXPECT(spec_verify_free(NULL), SV_OK);

  /* the allocation-free entry point checks sizes before touching the device */
  EXPECT(spec_verify_run_noalloc(x, SV_F32, x, SV_F32, d, -1, 3, 100, 1.0f, SV_PLAIN, 0.5f, NULL, NULL, 1u,
                                 len, tok, ap, fl, cnt, NULL),
         SV_EINVAL);
  EXPECT(spec_verify_run_noalloc(x, SV_F32, x, SV_F32, d, 4, 0, 100, 1.0f, SV_PLAIN, 0.5f, NULL, NULL, 1u,
                                 len, tok, ap, fl, cnt, NULL),
         SV_EINVAL);
  EXPECT(spec_verify_run_noalloc(x, SV_F32, x, SV_F32, d, 4, 3, 0, 1.0f, SV_PLAIN, 0.5f, NULL, NULL, 1u,
                                 len, tok, ap, fl, cnt, NULL),
         SV_EINVAL);
  EXPECT(spec_verify_run_noalloc(x, SV_F32, x, SV_F32, d, 4, SV_MAX_K + 1, 100, 1.0f, SV_PLAIN, 0.5f, NULL,
                                 NULL, 1u, len, tok, ap, fl, cnt, NULL),
         SV_EUNSUPPORTED);
  EXPECT(spec_verify_run_noalloc(x, SV_F32, x, SV_F32, d, 256, 8, 151936, 1.0f, SV_PLAIN, 0.5f, NULL, NULL,
                                 1u, len, tok, ap, fl, cnt, NULL),
         SV_EUNSUPPORTED);
  EXPECT(spec_verify_run_noalloc(x, SV_F32, x, SV_F32, d, 0x7fffffff, 32, SV_MAX_V, 1.0f, SV_PLAIN, 0.5f,
                                 NULL, NULL, 1u, len, tok, ap, fl, cnt, NULL),
         SV_EUNSUPPORTED);
  EXPECT(spec_verify_run_noalloc(x, SV_F32, x, SV_F32, d, 0, 5, 128256, 1.0f, SV_PLAIN, 0.5f, NULL, NULL, 1u,
                                 len, tok, ap, fl, cnt, NULL),
         SV_OK);

  printf("%d failed checks\n", failures);
  return failures == 0 ? 0 : 1;
}
