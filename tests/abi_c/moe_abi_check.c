/*
 * A plain C11 client of include/moe.h: it compiles the header as C (and the
 * test also compiles it as C++), links libmoe.so and exercises the calls that
 * need no GPU -- layer creation and its validation, every option key with
 * valid and invalid values, workspace sizing, statistics before any forward,
 * the call-order and argument errors of the forward entry points, and the
 * per-thread error message.  Prints one line per failed check and exits with
 * the number of failures.
 */
#include <pthread.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "moe.h"

static int failures = 0;

#define CHECK(cond)                                                  \
  do {                                                               \
    if (!(cond)) {                                                   \
      printf("FAILED line %d: %s\n", __LINE__, #cond);               \
      ++failures;                                                    \
    }                                                                \
  } while (0)

static void* other_thread(void* arg) {
  (void)arg;
  /* a failure on this thread must not change the main thread's message */
  moe_layer_t* bad = moe_layer_create(100, 512, 8, 2, 0);
  CHECK(bad == NULL);
  CHECK(strlen(moe_last_error()) > 0);
  return NULL;
}

int main(void) {
  /* creation and its validation */
  moe_layer_t* h = moe_layer_create(4096, 14336, 8, 2, 0);
  CHECK(h != NULL);
  CHECK(strcmp(moe_last_error(), "") == 0);
  CHECK(moe_layer_create(4096, 14336, 8, 9, 0) == NULL);  /* k > E */
  CHECK(strlen(moe_last_error()) > 0);
  CHECK(moe_layer_create(4096, 14336, 257, 2, 0) == NULL); /* E > 256 */
  CHECK(moe_layer_create(4096, 14336, 64, 17, 0) == NULL); /* k > 16 */
  CHECK(moe_layer_create(4096, 100, 8, 2, 0) == NULL);     /* f % 128 */
  CHECK(moe_layer_create(4096, 14336, 8, 2, 2) == NULL);   /* S > 1 */
  if (!h) return failures;

  /* the per-thread error message */
  moe_layer_t* ok = moe_layer_create(256, 512, 8, 2, 1);
  CHECK(ok != NULL && strcmp(moe_last_error(), "") == 0);
  pthread_t th;
  CHECK(pthread_create(&th, NULL, other_thread, NULL) == 0);
  CHECK(pthread_join(th, NULL) == 0);
  CHECK(strcmp(moe_last_error(), "") == 0);
  moe_layer_destroy(ok);

  /* options: valid values are taken, invalid ones refused */
  struct { int key; long long good, bad; } opts[] = {
      {MOE_OPT_MODE, MOE_MODE_STATIC, 3},
      {MOE_OPT_TIMEOUT_NS, 50000000, 10},
      {MOE_OPT_MOVER_CTAS, 4, -1},
      {MOE_OPT_GRID_CTAS, 37, 5000},
      {MOE_OPT_SPLIT_K, 4, 3},
      {MOE_OPT_TOKENS_PER_TILE, 160, 8},
      {MOE_OPT_ROUTE_TOKENS, 64, 96},
      {MOE_OPT_CLAIM_AHEAD, 2, -2},
      {MOE_OPT_RELEASE, 0, 2},
      {MOE_OPT_ROUTE_SPLITS, 8, 9},
      {MOE_OPT_L2_PREFETCH, 1 << 20, -2},
  };
  for (size_t i = 0; i < sizeof(opts) / sizeof(opts[0]); ++i) {
    CHECK(moe_layer_set_option(h, opts[i].key, opts[i].good) == MOE_OK);
    CHECK(moe_layer_set_option(h, opts[i].key, opts[i].bad) == MOE_E_INVAL);
  }
  CHECK(moe_layer_set_option(h, MOE_OPT_PREFETCH, 0) == MOE_OK);
  CHECK(moe_layer_set_option(h, MOE_OPT_BANDS, 0) == MOE_OK);
  CHECK(moe_layer_set_option(h, MOE_OPT_FAULT_DROP_TASK, -1) == MOE_OK);
  CHECK(moe_layer_set_option(h, 999, 1) == MOE_E_INVAL);
  CHECK(moe_layer_set_option(NULL, MOE_OPT_MODE, 0) == MOE_E_INVAL);

  /* workspace sizing: at least the permuted tokens (T*k rows of d bf16)
   * for every T_max, -1 on bad input.  (It is not monotone in T_max: small
   * layers keep fp32 down-projection partials, large ones bf16 outputs.) */
  for (int T = 1; T <= 32768; T *= 2) {
    const long long b = moe_layer_workspace_bytes(h, T);
    CHECK(b >= (long long)T * 2 * 4096 * 2);
  }
  CHECK(moe_layer_workspace_bytes(NULL, 64) == -1);
  CHECK(moe_layer_workspace_bytes(h, -1) == -1);

  /* no forward yet: no statistics */
  CHECK(moe_layer_get_stat(h, MOE_STAT_MOVER_CTAS) == -1);
  CHECK(moe_layer_get_stat(h, MOE_STAT_SPLIT_K) == -1);
  CHECK(moe_layer_get_stat(NULL, MOE_STAT_TASKS) == -1);

  /* call order and arguments, refused before any CUDA call */
  static _Alignas(16) uint16_t buf[64];
  CHECK(moe_layer_forward(h, 1, buf, buf, buf, buf, buf, buf, NULL) == MOE_E_STATE);
  CHECK(moe_layer_forward(NULL, 1, buf, buf, buf, buf, buf, buf, NULL) == MOE_E_INVAL);
  CHECK(moe_layer_forward_host(h, 1, buf, buf, buf, buf, buf, buf, NULL) == MOE_E_STATE);
  CHECK(moe_layer_forward_noalloc(NULL, 1, buf, buf, buf, buf, buf, buf, NULL) == MOE_E_INVAL);
  CHECK(moe_layer_forward_residual_norm(h, 1, buf, buf, buf, buf, buf, NULL, buf, 1e-6f, buf,
                                        buf, NULL) == MOE_E_INVAL);
  CHECK(moe_layer_forward_residual_norm(h, 1, buf, buf, buf, buf, buf, buf, buf, -1.0f, buf,
                                        buf, NULL) == MOE_E_INVAL);
  float best = 0.0f;
  CHECK(moe_layer_calibrate(h, 1, buf, buf, buf, buf, buf, buf, 3, &best, NULL) == MOE_E_STATE);
  CHECK(moe_layer_calibrate(NULL, 1, buf, buf, buf, buf, buf, buf, 3, &best, NULL) ==
        MOE_E_INVAL);
  CHECK(moe_layer_get_routing(h, NULL, NULL, NULL, NULL, NULL, NULL, NULL) == MOE_E_STATE);
  CHECK(moe_layer_get_trace(NULL, NULL, 0, NULL) == -1);

  moe_layer_destroy(h);
  moe_layer_destroy(NULL);
  printf("%d failures\n", failures);
  return failures;
}
