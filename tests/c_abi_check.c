/* A plain C99 consumer of include/lmce.h: it must compile as C with warnings as errors, link
 * against liblmce.so, and get LMCE_ERR_ARG back from every entry point given a null handle
 * (no device is touched on that path). */
#include <stdio.h>
#include <string.h>

#include "lmce.h"

static int failures = 0;

static void expect(const char* what, int got, int want) {
  if (got != want) {
    printf("%s: got %d, want %d\n", what, got, want);
    ++failures;
  }
}

int main(void) {
  lmce_config cfg;
  lmce_handle* h = NULL;
  double d = 0.0;
  int64_t n = 0;
  memset(&cfg, 0, sizeof cfg);
  expect("create(NULL cfg)", lmce_create(NULL, NULL, &h), LMCE_ERR_ARG);
  expect("create(C = 0)", lmce_create(&cfg, (float*)16, &h), LMCE_ERR_ARG);
  expect("microstep", lmce_microstep(NULL, NULL, NULL, NULL, 0, 1, NULL, NULL, NULL), LMCE_ERR_ARG);
  expect("microstep_compact",
         lmce_microstep_compact(NULL, NULL, NULL, NULL, 0, 0, 1, NULL, NULL, NULL), LMCE_ERR_ARG);
  expect("microstep_ln",
         lmce_microstep_ln(NULL, NULL, NULL, NULL, LMCE_LN_LAYERNORM, 1e-5f, NULL, NULL, 0, 1, NULL, NULL, NULL,
                           NULL, NULL),
         LMCE_ERR_ARG);
  expect("microstep_ln_compact",
         lmce_microstep_ln_compact(NULL, NULL, NULL, NULL, LMCE_LN_RMSNORM, 1e-5f, NULL, NULL, 0, 0, 1, NULL,
                                   NULL, NULL, NULL, NULL),
         LMCE_ERR_ARG);
  expect("finalize", lmce_finalize(NULL, &d, &n, &d, NULL), LMCE_ERR_ARG);
  expect("dw_sumsq", lmce_dw_sumsq(NULL, &d, NULL), LMCE_ERR_ARG);
  expect("adamw", lmce_adamw(NULL, NULL, NULL, NULL, NULL, 1, 1e-3f, 0.9f, 0.95f, 1e-8f, 0.1f, 1.0f, NULL),
         LMCE_ERR_ARG);
  expect("profile", lmce_profile(NULL, 1), LMCE_ERR_ARG);
  expect("test_stall_next_microstep", lmce_test_stall_next_microstep(NULL, 1000000), LMCE_ERR_ARG);
  expect("clip_coef(NULL)", lmce_clip_coef(1.0, 1.0, NULL), LMCE_ERR_ARG);
  expect("test_bounds_limit", lmce_test_bounds_limit(NULL, 0), LMCE_ERR_ARG);
  if (lmce_debug_bounds() != 0 && lmce_debug_bounds() != 1) {
    printf("debug_bounds\n");
    ++failures;
  }
  {
    float c = 0.f;
    expect("clip_coef(4, 1)", lmce_clip_coef(4.0, 1.0, &c), LMCE_OK);
    if (!(c > 0.4999f && c < 0.5f)) {
      printf("clip_coef(4, 1) = %g\n", (double)c);
      ++failures;
    }
  }
  expect("destroy(NULL)", lmce_destroy(NULL), LMCE_OK);
  if (lmce_status_string(LMCE_OK) == NULL || lmce_launch_count(NULL) != 0 || lmce_selected_path(NULL) != -1) {
    printf("status / count / path queries\n");
    ++failures;
  }
  printf(failures ? "FAILED\n" : "ok\n");
  return failures ? 1 : 0;
}
