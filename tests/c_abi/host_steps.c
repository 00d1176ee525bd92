/* A plain C client of libdms.so: it uses only include/dms.h, host memory and
 * the legacy default stream (no CUDA runtime calls of its own).
 *
 * It creates a cache, runs decode steps from host buffers (dms_step_host),
 * and checks two facts that hold for any inputs:
 *   - the first step sees one key, so every query head's output is that
 *     token's V row, exactly (softmax over one key is 1, and bf16 widens to
 *     fp32 exactly);
 *   - every later output lies within the range of the V values seen so far
 *     (it is a convex combination of retained V rows).
 * Exit status 0 on success, 1 on a failed check, 2 on a library error.
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "dms.h"

enum { B = 2, HKV = 2, G = 4, HQ = HKV * G, D = 128, CAP = 64, W = 16, STEPS = 40 };

static uint32_t rng = 12345u;
static float next_uniform(void) { /* xorshift32 in [-1, 1) */
  rng ^= rng << 13;
  rng ^= rng >> 17;
  rng ^= rng << 5;
  return (float)(rng >> 8) / 8388608.0f - 1.0f;
}

static uint16_t to_bf16(float x) { /* round to nearest even (inputs are finite) */
  uint32_t u;
  memcpy(&u, &x, 4);
  u += 0x7fffu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

static float from_bf16(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float x;
  memcpy(&x, &u, 4);
  return x;
}

static int check(int rc, const char* what) {
  if (rc != DMS_OK) {
    fprintf(stderr, "%s: %s (%d)\n", what, dms_error_string(rc), rc);
    exit(2);
  }
  return rc;
}

int main(void) {
  dms_cache_t* cache = dms_cache_create(B, HKV, CAP, D, W);
  if (!cache) {
    fprintf(stderr, "dms_cache_create: %s\n", dms_error_string(dms_last_error()));
    return 2;
  }
  uint16_t* k = malloc(sizeof(uint16_t) * B * HKV * D);
  uint16_t* v = malloc(sizeof(uint16_t) * B * HKV * D);
  uint16_t* q = malloc(sizeof(uint16_t) * B * HQ * D);
  float* logit = malloc(sizeof(float) * B * HKV);
  float* out = malloc(sizeof(float) * B * HQ * D);
  float vmin[B * HKV * D], vmax[B * HKV * D];
  const float scale = 1.0f / sqrtf((float)D);
  int bad = 0;
  for (int t = 0; t < STEPS; ++t) {
    for (int i = 0; i < B * HKV * D; ++i) {
      k[i] = to_bf16(next_uniform());
      v[i] = to_bf16(next_uniform());
      const float vi = from_bf16(v[i]);
      vmin[i] = t == 0 ? vi : fminf(vmin[i], vi);
      vmax[i] = t == 0 ? vi : fmaxf(vmax[i], vi);
    }
    for (int i = 0; i < B * HQ * D; ++i) q[i] = to_bf16(next_uniform());
    for (int i = 0; i < B * HKV; ++i) logit[i] = next_uniform();
    check(dms_step_host(cache, k, v, logit, q, out, scale, HQ, NULL), "dms_step_host");
    check(dms_step_host_join(cache, NULL), "dms_step_host_join");
    check(dms_cache_status(cache, NULL), "dms_cache_status"); /* synchronizes the stream */
    for (int b = 0; b < B; ++b)
      for (int g = 0; g < HQ; ++g)
        for (int d = 0; d < D; ++d) {
          const int h = g / G, kv = (b * HKV + h) * D + d;
          const float o = out[(b * HQ + g) * D + d];
          if (t == 0 && o != from_bf16(v[kv])) ++bad;
          /* evicted tokens leave the range only narrower; allow fp32 rounding */
          if (!(o >= vmin[kv] - 1e-5f && o <= vmax[kv] + 1e-5f)) ++bad;
        }
  }
  if (dms_cache_position(cache) != STEPS) ++bad;
  dms_cache_destroy(cache);
  free(k);
  free(v);
  free(q);
  free(logit);
  free(out);
  if (bad) {
    fprintf(stderr, "%d checks failed\n", bad);
    return 1;
  }
  printf("ok: %d host-buffer steps\n", STEPS);
  return 0;
}
