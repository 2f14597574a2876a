/* The NVFP4 block-scale division s = fl(b / p), p = fl(6 gs), computed the way
 * the quantize kernels compute it: r = fl(1 / p) once per launch, q0 = fl(b r),
 * q = fl(q0 + fl(b - q0 p) r) (Markstein's correction, both steps fused
 * multiply-adds), with q0 itself when b < 2^-100 takes the exact division and
 * when q0 is outside [2^-64, 1024) -- where the block scale is only e4m3(q0),
 * 448 above and 0 below 2^-10.  This program compares that against the
 * correctly rounded quotient (a double division rounded once to float: exact
 * for float operands, 53 >= 2 * 24 + 2) for every positive finite bf16 amax
 * (gs = fl(amax / 2688)) and every bf16 block maximum b <= amax, and for every
 * bf16 b against pseudo-random normal divisors (a quarter with an all-ones
 * mantissa).  It prints the number of pairs whose e4m3 rounding could differ
 * (expected: 0) and exits 1 if there is one. */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

static float f_of(uint32_t u) { float x; memcpy(&x, &u, 4); return x; }
static uint32_t u_of(float x) { uint32_t v; memcpy(&v, &x, 4); return v; }
static float bf16(uint32_t h) { return f_of(h << 16); }
static float exact_div(float b, float p) { return (float)((double)b / (double)p); }

static float kernel_div(float b, float p, float r) {
  if (b < 0x1p-100f) return exact_div(b, p);
  const float q0 = b * r;
  if (!(q0 < 1024.0f) || q0 < 0x1p-64f) return q0;
  return fmaf(fmaf(-q0, p, b), r, q0);
}

/* 1 if the two quotients can give different e4m3 block scales */
static int differs(float x, float y) {
  if (x < 0x1p-11f) return !(y < 0x1p-10f);   /* both round to a zero scale */
  if (x >= 1024.0f) return !(y >= 464.0f);    /* both saturate at 448 */
  return u_of(x) != u_of(y);
}

int main(int argc, char** argv) {
  const int random_divisors = argc > 1 ? atoi(argv[1]) : 2000;
  long long pairs = 0, bad = 0;
  for (uint32_t a = 1; a < 0x7F80; ++a) {
    const float p = 6.0f * (bf16(a) / 2688.0f);
    if (!(p >= 0x1p-126f && p < 0x1p126f)) continue;  /* the kernels divide exactly there */
    const float r = 1.0f / p;
    for (uint32_t bb = 1; bb <= a; ++bb, ++pairs) bad += differs(exact_div(bf16(bb), p), kernel_div(bf16(bb), p, r));
  }
  uint64_t s = 88172645463325252ull;
  for (int it = 0; it < random_divisors; ++it) {
    s ^= s << 13; s ^= s >> 7; s ^= s << 17;
    uint32_t pb = (uint32_t)(s >> 20) & 0x7FFFFFFFu;
    if (it % 4 == 0) pb = (pb & 0x7F800000u) | 0x7FFFFFu;
    const float p = f_of(pb);
    if (!(p >= 0x1p-126f && p < 0x1p126f)) continue;
    const float r = 1.0f / p;
    for (uint32_t bb = 1; bb < 0x7F80; ++bb, ++pairs) bad += differs(exact_div(bf16(bb), p), kernel_div(bf16(bb), p, r));
  }
  printf("%lld pairs, %lld differ\n", pairs, bad);
  return bad != 0;
}
