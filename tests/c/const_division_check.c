/* Exhaustive check of the constant-divisor division the write kernels use for
 * their scales: q0 = RN(x * RN(1/d)), r = fma(-q0, d, x), q = fma(r, RN(1/d), q0)
 * (Markstein's correction step).  For each divisor it walks every fp32 input of
 * the range the kernels feed it and counts results that differ from the IEEE
 * quotient x / d.  Prints one line per divisor: d, first input, mismatches. */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

static float f_of(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }
static uint32_t u_of(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }

static long long mismatches(float d, float first) {
  const float rd = 1.0f / d;
  long long bad = 0;
  uint32_t u;
  for (u = u_of(first); u < 0x7F800000u; ++u) {   /* every finite x >= first */
    const float x = f_of(u);
    const float q0 = x * rd;
    const float r = fmaf(-q0, d, x);
    const float q = fmaf(r, rd, q0);
    if (u_of(q) != u_of(x / d)) ++bad;
  }
  return bad;
}

int main(void) {
  /* scales of max(amax, 1e-8): x >= 1e-8; KVarN's (max - min): any x >= 0 */
  const float ds[5] = {127.0f, 448.0f, 7.0f, 15.0f, 3.0f};
  const float first[5] = {1e-8f, 1e-8f, 1e-8f, 0.0f, 0.0f};
  int k;
  for (k = 0; k < 5; ++k) printf("%g %a %lld\n", ds[k], first[k], mismatches(ds[k], first[k]));
  return 0;
}
