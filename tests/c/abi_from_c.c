/* A plain C99 caller of the library through include/attn_jvp.h.  It makes
 * only calls that return before any GPU work (argument validation, status
 * strings, the launch counter, the wait-bound setter), so it runs on a
 * machine without a GPU; it prints the number of failed checks and exits
 * nonzero if there is one. */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "attn_jvp.h"

static int fails = 0;

static void expect(const char* what, attn_status got, attn_status want) {
  if (got != want) {
    printf("%s: got %d (%s), want %d\n", what, (int)got, attn_status_string(got), (int)want);
    ++fails;
  }
}

static attn_shape shape(int32_t M, int32_t N, int32_t dqk, int32_t dv) {
  attn_shape s;
  memset(&s, 0, sizeof s);
  s.B = 1;
  s.H = 2;
  s.M = M;
  s.N = N;
  s.Dqk = dqk;
  s.Dv = dv;
  return s;
}

int main(void) {
  /* 16-byte aligned addresses that validation rejects before using them */
  void* p = (void*)(uintptr_t)0x10000;
  void* odd = (void*)(uintptr_t)0x10008;
  float* l = (float*)p;
  const float nan_scale = NAN;
  attn_shape s = shape(128, 128, 64, 64);

  expect("null shape", attn_fwd_jvp(NULL, p, p, p, p, p, p, NULL, NULL, 0, nan_scale, p, p, l, NULL),
         ATTN_ERR_INVALID_ARG);
  expect("null tangent", attn_fwd_jvp(&s, p, p, p, NULL, p, p, NULL, NULL, 0, nan_scale, p, p, l, NULL),
         ATTN_ERR_INVALID_ARG);
  expect("misaligned q", attn_fwd_jvp(&s, odd, p, p, p, p, p, NULL, NULL, 0, nan_scale, p, p, l, NULL),
         ATTN_ERR_MISALIGNED);
  expect("bad scale", attn_fwd_jvp(&s, p, p, p, p, p, p, NULL, NULL, 0, -1.0f, p, p, l, NULL),
         ATTN_ERR_INVALID_ARG);
  attn_shape cross = shape(128, 256, 64, 64);
  expect("causal cross attention", attn_fwd_jvp(&cross, p, p, p, p, p, p, NULL, NULL, 1, nan_scale, p, p, l, NULL),
         ATTN_ERR_INVALID_ARG);
  attn_shape d96 = shape(128, 128, 96, 64);
  expect("head dim 96", attn_fwd_jvp(&d96, p, p, p, p, p, p, NULL, NULL, 0, nan_scale, p, p, l, NULL),
         ATTN_ERR_UNSUPPORTED);
  attn_shape d512 = shape(128, 128, 512, 256);
  expect("head dim 512", attn_fwd_jvp(&d512, p, p, p, p, p, p, NULL, NULL, 0, nan_scale, p, p, l, NULL),
         ATTN_ERR_UNSUPPORTED);
  attn_shape empty = shape(0, 128, 64, 64);
  expect("empty problem", attn_fwd(&empty, NULL, p, p, NULL, NULL, 0, nan_scale, NULL, NULL, NULL), ATTN_OK);

  /* a bias with jagged inputs is not supported (dense only) */
  attn_bias b;
  memset(&b, 0, sizeof b);
  b.bias = (const float*)p;
  attn_shape jag = shape(0, 0, 64, 64);
  jag.T = 64;
  jag.max_seq_len = 64;
  expect("jagged backward with a bias",
         attn_bwd(&jag, p, p, p, p, p, l, (const int32_t*)p, &b, 0, nan_scale, p, p, p, l, NULL),
         ATTN_ERR_UNSUPPORTED);
  expect("backward stages outside the flags",
         attn_bwd_stages(&s, p, p, p, p, p, l, NULL, NULL, 0, nan_scale, p, p, p, l, 0, 8u, NULL),
         ATTN_ERR_INVALID_ARG);

  for (int st = 0; st <= 5; ++st) {
    const char* msg = attn_status_string((attn_status)st);
    if (msg == NULL || msg[0] == '\0') {
      printf("status %d has no description\n", st);
      ++fails;
    }
  }
  attn_set_wait_timeout_ns(2000000000ull);
  (void)attn_launch_count();
  printf("%d\n", fails);
  return fails != 0;
}
