/* dispatch_cost.c -- host cost of one granikv_dispatch call, timed from C (no binding layer).
 *
 * GraniKV (arXiv:2608.15584), "B.5 Per-Step Dispatch Overhead": the pages measure their
 * per-step dispatch at under 1 us of CPU time.  This times granikv_dispatch on a host-only
 * context (no device): one HOT prefix of 16384 tokens, the Llama-3.1-8B attention shape
 * (32/8/128, bf16), B requests with log-normal-like suffix lengths, dispatched again and again
 * into one plan (as a serving loop does); the lengths grow by one token every other call (and
 * start over every 64 calls).  Prints one line per B: median and minimum microseconds per call
 * over repeated batches of calls; a failed dispatch ends the program with status 5.
 *
 *   usage: dispatch_cost B1 [B2 ...]
 */
#include <stdio.h>
#include <stdlib.h>
#include <time.h>

#include "granikv.h"

static double now_us(void) {
  struct timespec ts;
  clock_gettime(CLOCK_MONOTONIC, &ts);
  return ts.tv_sec * 1e6 + ts.tv_nsec * 1e-3;
}

static int cmp_double(const void* a, const void* b) {
  const double x = *(const double*)a, y = *(const double*)b;
  return x < y ? -1 : x > y;
}

int main(int argc, char** argv) {
  for (int a = 1; a < argc; ++a) {
    const int B = atoi(argv[a]);
    if (B <= 0) return 2;
    granikv_config cfg = {0};
    cfg.n_layers = 1;
    cfg.n_q = 32;
    cfg.n_kv = 8;
    cfg.head_dim = 128;
    cfg.dtype = GRANIKV_DTYPE_BF16;
    cfg.n_slots = 400000;
    cfg.max_batch = B;
    cfg.host_only = 1;
    granikv_ctx* ctx = NULL;
    if (granikv_create(&cfg, &ctx) != GRANIKV_OK) return 3;
    int32_t sid = -1;
    int64_t off = 0;
    if (granikv_hot_alloc(ctx, 16384, &sid, &off) != GRANIKV_OK) return 4;
    int32_t* slab = malloc(sizeof(int32_t) * B);
    int32_t* len = malloc(sizeof(int32_t) * B);
    int32_t* base = malloc(sizeof(int32_t) * B);
    unsigned s = 12345u;
    for (int b = 0; b < B; ++b) {
      slab[b] = sid;
      s = s * 1664525u + 1013904223u;
      base[b] = len[b] = 32 + (int32_t)((s >> 8) % 600);  /* 32..631 tokens */
    }
    granikv_batch bt = {B, slab, len, NULL, 4096, NULL};
    granikv_plan* plan = NULL;
    granikv_plan_create(ctx, &plan);
    for (int i = 0; i < 64; ++i) {  /* warm the plan's working arrays */
      for (int b = 0; b < B; ++b) len[b] = base[b] + i;
      if (granikv_dispatch(ctx, &bt, plan) != GRANIKV_OK) return 5;
    }
    enum { kBatches = 31 };
    const int calls = B >= 1024 ? 200 : 2000;
    double per[kBatches];
    for (int r = 0; r < kBatches; ++r) {
      double t = 0.0;
      for (int i = 0; i < calls; ++i) {
        for (int b = 0; b < B; ++b) len[b] = base[b] + (i % 128) / 2;  /* lengths move */
        const double t0 = now_us();
        const granikv_status st = granikv_dispatch(ctx, &bt, plan);
        t += now_us() - t0;
        if (st != GRANIKV_OK) return 5;
      }
      per[r] = t / calls;
    }
    qsort(per, kBatches, sizeof(double), cmp_double);
    printf("B %d: %.3f us per dispatch (median), %.3f (min)\n", B, per[kBatches / 2], per[0]);
    granikv_plan_destroy(plan);
    granikv_destroy(ctx);
    free(slab);
    free(len);
    free(base);
  }
  return 0;
}
