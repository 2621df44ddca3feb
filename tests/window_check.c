/* window_check.c -- checks the bracketing window the activation kernel
   quantises fp32 values with: with r = RN(1/scale), rl = RN(r (1 - 2^-20))
   and rh = RN(r (1 + 2^-20)), the products RN(x rl) and RN(x rh) lie below
   and above RN(x / scale), so where their E4M3 bytes agree, that byte is
   e4m3(RN(x / scale)) (rounding to E4M3 is monotone).  Where they differ the
   kernel divides; this program counts those cases too.

   Usage: window_check COUNT SEED [noshrink]
          window_check encode   (binary32 values on stdin, their bytes on stdout)
     COUNT random (x, scale) pairs: scale with a random binary32 significand
     and an exponent in [-40, 40].  Half the x are scale * t * 448 with t
     uniform in [-1, 1] and 0 to 20 low significand bits cleared; the other
     half sit on an E4M3 rounding midpoint M: x = RN(M scale) moved by -2 to
     2 units in the last place, so that RN(x / scale) falls on either side of
     M, or on it.
     "noshrink" uses rl = rh = r (a control: the bytes then agree where they
     should not, and the check must see mismatches).
   Prints "cases N agree A mismatches M" and exits 0.

   The E4M3 encoder here is written from the format (OCP E4M3: 4 exponent
   bits, bias 7, 3 mantissa bits, max 448, no infinity): round to nearest
   even on the grid of the binade, saturate finite overflow to 448. */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

static uint32_t f2u(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  return u;
}

static float u2f(uint32_t u) {
  float f;
  memcpy(&f, &u, 4);
  return f;
}

static uint8_t e4m3(float v) {
  const uint8_t s = (f2u(v) >> 31) ? 0x80 : 0x00;
  if (isnan(v)) return (uint8_t)(s | 0x7F);
  double a = fabs((double)v);
  if (a >= 464.0) return (uint8_t)(s | 0x7E); /* saturate: 448 = 1.75 * 2^8 */
  int e;
  frexp(a, &e);                               /* a = m 2^e, m in [0.5, 1) */
  int k = e - 1;                              /* a in [2^k, 2^(k+1)) */
  if (k < -6) k = -6;                         /* subnormal grid below 2^-6 */
  const double step = ldexp(1.0, k - 3);
  const double n = nearbyint(a / step);       /* round to nearest even */
  const double q = n * step;
  if (q == 0.0) return s;
  int qe;
  frexp(q, &qe);
  const int kk = qe - 1;
  if (kk < -6) return (uint8_t)(s | (uint8_t)(q / ldexp(1.0, -9)));   /* subnormal code */
  if (q > 448.0) return (uint8_t)(s | 0x7E);
  const int mant = (int)(q / ldexp(1.0, kk - 3)) - 8;
  return (uint8_t)(s | ((kk + 7) << 3) | mant);
}

static uint64_t rng_state;
static uint64_t next_u64(void) { /* splitmix64 */
  uint64_t z = (rng_state += 0x9E3779B97F4A7C15ull);
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

int main(int argc, char **argv) {
  if (argc > 1 && strcmp(argv[1], "encode") == 0) {   /* the encoder alone, for its own test */
    float v;
    while (fread(&v, sizeof v, 1, stdin) == 1) putchar(e4m3(v));
    return 0;
  }
  const long long count = argc > 1 ? atoll(argv[1]) : 1000000;
  rng_state = argc > 2 ? strtoull(argv[2], NULL, 10) : 1;
  const int noshrink = argc > 3 && strcmp(argv[3], "noshrink") == 0;
  long long agree = 0, bad = 0;
  for (long long i = 0; i < count; ++i) {
    const uint64_t w = next_u64(), w2 = next_u64();
    const int ex = (int)(w % 81) - 40;
    const float scale = ldexpf(u2f(0x3F800000u | (uint32_t)(w >> 41)), ex);
    float x;
    if (w2 & 1) {
      const double t = ((double)(w2 >> 11) / 9007199254740992.0) * 2.0 - 1.0;
      x = (float)(t * 448.0 * scale);
      const int clear = (int)((w >> 8) % 21);
      x = u2f(f2u(x) & ~((1u << clear) - 1u));
    } else {
      /* the midpoint between adjacent positive E4M3 values, codes c and c + 1
         (c in 1 .. 125; code c has exponent field c >> 3, mantissa c & 7) */
      const int code = (int)((w2 >> 8) % 125) + 1;
      const int e = code >> 3, m = code & 7;
      const double c0 = e == 0 ? ldexp(m, -9) : ldexp(8 + m, e - 10);
      const int e1 = (code + 1) >> 3, m1 = (code + 1) & 7;
      const double c1 = e1 == 0 ? ldexp(m1, -9) : ldexp(8 + m1, e1 - 10);
      const double mid = (c0 + c1) / 2;
      x = (float)(mid * (double)scale);
      x = u2f(f2u(x) + (uint32_t)((int)((w2 >> 40) % 5) - 2));
      if (w2 & 2) x = -x;
    }
    const float r = 1.0f / scale;
    const float rl = noshrink ? r : r * (1.0f - 0x1p-20f);
    const float rh = noshrink ? r : r * (1.0f + 0x1p-20f);
    const uint8_t lo = e4m3(x * rl), hi = e4m3(x * rh);
    if (lo != hi) continue;
    agree++;
    if (lo != e4m3(x / scale)) bad++;
  }
  printf("cases %lld agree %lld mismatches %lld\n", count, agree, bad);
  return 0;
}
