/* Checks the division method the CUDA kernels use for q = a / b with one reciprocal per
 * block: r = RN(1/b), q0 = RN(a r), e = RN(a - q0 b) (one fma), q = RN(q0 + e r) (one fma)
 * -- Markstein's correction (P. Markstein, IBM J. Res. Dev. 34(1), 1990) -- against IEEE
 * binary32 division, and the negated form the kernels run (qn = -q, also for signed zeros).
 * Division is invariant under scaling by powers of two (away from under/overflow), so
 * operands are taken in [1, 2) with their full mantissa ranges:
 *   part 1: every divisor mantissa (2^23) against 24 dividends each;
 *   part 2: every dividend mantissa (2^23) against 600 divisors (near 1, near 2, near sqrt 2,
 *           near 4/3, and random).
 * Prints "checked N mismatches M" and exits non-zero on any mismatch. */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

static float f_of(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }
static uint32_t u_of(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }
static uint64_t st = 0x9E3779B97F4A7C15ull;
static uint64_t rnd(void) { st ^= st << 13; st ^= st >> 7; st ^= st << 17; return st; }

static long bad = 0, tot = 0;

static void check(float a, float b, float r) {
  const float q0 = a * r;
  const float e = fmaf(-q0, b, a);
  const float q = fmaf(e, r, q0);
  const float nr = -r;                 /* negated form */
  const float q0n = a * nr;
  const float en = fmaf(q0n, b, a);
  const float qn = fmaf(en, nr, q0n);
  const float ref = a / b;
  ++tot;
  /* the direct form turns -0 into +0 (e = +0, +0 + -0 = +0); the kernels use the negated
     form, which must match everywhere */
  const int direct_ok = (a == 0.0f) || u_of(q) == u_of(ref);
  if (!direct_ok || u_of(qn) != (u_of(ref) ^ 0x80000000u)) {
    if (bad < 5) printf("mismatch a=%a b=%a q=%a qn=%a ref=%a\n", a, b, q, qn, ref);
    ++bad;
  }
}

int main(void) {
  for (uint32_t mb = 0; mb < (1u << 23); ++mb) {
    const float b = f_of(0x3f800000u | mb);
    const float r = 1.0f / b;
    for (int k = 0; k < 24; ++k) {
      float a = f_of(0x3f800000u | (uint32_t)(rnd() & 0x7fffff));
      if (k >= 16) a = f_of(u_of((float)(k - 15) * 0.5f * b) + (uint32_t)((int)(rnd() % 9) - 4));
      check(a, b, r);
    }
  }
  uint32_t bs[600];
  int nb = 0;
  for (int k = 0; k < 64; ++k) {
    bs[nb++] = 0x3f800000u + k;
    bs[nb++] = 0x3fffffffu - k;
    bs[nb++] = 0x3fb504f3u + k - 32;
    bs[nb++] = 0x3faaaaaau + k - 32;
  }
  while (nb < 600) bs[nb++] = 0x3f800000u | (uint32_t)(rnd() & 0x7fffff);
  for (int i = 0; i < nb; ++i) {
    const float b = f_of(bs[i]);
    const float r = 1.0f / b;
    for (uint32_t ma = 0; ma < (1u << 23); ++ma) check(f_of(0x3f800000u | ma), b, r);
  }
  /* signed zeros: -0 / b must stay -0 in both forms */
  check(-0.0f, 3.0f, 1.0f / 3.0f);
  check(0.0f, 3.0f, 1.0f / 3.0f);
  printf("checked %ld mismatches %ld\n", tot, bad);
  return bad != 0;
}
